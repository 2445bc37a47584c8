"""GB300-native fused LM-head GRPO / GSPO loss.

The compute lives in ``libgrpohead.so`` (hand-written sm_103a CUDA: tcgen05
tensor-core tiles fed by TMA, online fp32 log-sum-exp over the vocabulary,
GRPO/GSPO epilogues).  This package is a thin ctypes binding with the same
entry-point names as the C ABI in ``include/grpo_head.h``:

    grpo_head_forward, gspo_segment_loss, grpo_head_backward, grpo_group_advantage

The binding is imported lazily so that ``import gspo_logprob_gb300`` works on a
machine without the built library; the first call then fails loudly if the
library is missing.
"""
__all__ = ["grpo_head_forward", "gspo_segment_loss", "grpo_head_backward", "grpo_group_advantage",
           "grpo_loss_from_sequence_totals", "grpo_head_logprob_shard", "grpo_logprob_merge",
           "vocab_shard_bounds", "gspo_segment_partials", "gspo_segment_loss_from_partials",
           "grpo_head_backward_shard", "grpo_dh_merge", "build", "ops"]


def build(verbose: bool = False) -> str:
    from .buildlib import build as _build
    return _build(verbose=verbose)


def __getattr__(name):
    if name in ("grpo_head_forward", "gspo_segment_loss", "grpo_head_backward", "grpo_group_advantage",
                "grpo_loss_from_sequence_totals", "grpo_head_logprob_shard", "grpo_logprob_merge",
                "vocab_shard_bounds", "gspo_segment_partials", "gspo_segment_loss_from_partials",
                "grpo_head_backward_shard", "grpo_dh_merge", "ops"):
        import importlib
        ops = importlib.import_module(".ops", __name__)
        return ops if name == "ops" else getattr(ops, name)
    raise AttributeError(name)
