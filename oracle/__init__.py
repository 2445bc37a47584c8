"""fp64 CPU oracle for the fused LM-head GRPO/GSPO loss.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it.  The product path (``gspo_logprob_gb300`` and its CUDA library) never
imports, links or runs anything here, and this package imports nothing from
it: the two share no code, constants or helpers.  Inputs come from the
independent ``synth`` package.

Every function computes the plain definition of its quantity in float64
(full logits materialised per row chunk, log-softmax, autograd-free analytic
gradients, explicit loops for per-sequence and per-segment sums).

Parity pins (tests/test_oracle_*.py) tie each function to something other
than itself: closed forms, invariants, library routines, finite differences
and a hand-derived worked example.  Functions without such a pin are listed
as "parity unpinned" in the module docstring of ``grpo_head_oracle``.
"""
from .grpo_head_oracle import (  # noqa: F401
    OracleError,
    as_f64,
    dlogits,
    forward_backward,
    group_advantages,
    grpo_loss,
    gspo_loss,
    head_backward,
    head_logits,
    selected_logprob,
    streamed_lse,
)
