"""The forward entry point for callers that cannot allocate device memory.

Such callers (device memory wholly owned by another allocator, or no
cudaMalloc allowed mid-step because it can synchronise the device) call
grpo_head_forward_noalloc, which keeps its scratch in a fixed device array
instead of a caller workspace.  This file checks, through the C ABI, that it
returns what grpo_head_forward returns with a caller workspace, on two calls
in a row (different problems, so stale scratch contents would show), and that
a problem too large for the array is refused before any GPU work.  It is
named to be collected last.
"""
import ctypes
import dataclasses
import math

import numpy as np
import pytest
import torch

from synth import CONFIGS, make_workload

from gpu_helpers import dev_head, dev_tensor, gpu_lib  # noqa: F401

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _problem(cfg, dtype, N=None):
    w = make_workload(cfg, dtype=dtype, N=N)
    H, W, y, m = dev_head(w)
    N, V = H.shape[0], W.shape[0]
    old = dev_tensor((-math.log(V) + w["u_old"]).astype(np.float32))
    ref = dev_tensor((-math.log(V) + w["u_ref"]).astype(np.float32))
    adv = dev_tensor(np.linspace(-1.0, 1.0, w["num_seqs"]).astype(np.float32))
    seq = dev_tensor(w["seq_id"])
    return w, (H, W, y, m), (old, ref, adv, seq)


def _call(lib, tensors, extra, num_seqs, noalloc):
    from gspo_logprob_gb300._abi import GhGrpo, GhHead
    H, W, y, m = tensors
    old, ref, adv, seq = extra
    N, D, V = H.shape[0], H.shape[1], W.shape[0]
    head = GhHead(N=N, D=D, V=V, dtype=0 if H.dtype == torch.bfloat16 else 1, row_tile=0, H=H.data_ptr(),
                  W=W.data_ptr(), targets=y.data_ptr(), mask=m.data_ptr())
    g = GhGrpo(old_logp=old.data_ptr(), ref_logp=ref.data_ptr(), adv=adv.data_ptr(), seq_id=seq.data_ptr(),
               num_seqs=num_seqs, reduction=0, eps_low=0.2, eps_high=0.28, beta=0.04, norm=0.0)
    out = {k: torch.full((N,), float("nan"), device="cuda") for k in ("logp", "lse", "coef")}
    out["loss3"] = torch.full((3,), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if noalloc:
        rc = lib.grpo_head_forward_noalloc(ctypes.byref(head), ctypes.byref(g), _ptr(out["logp"]), _ptr(out["lse"]),
                                           _ptr(out["coef"]), _ptr(out["loss3"]), _ptr(st), stream)
    else:
        nbytes = lib.grpo_head_forward_workspace_size(ctypes.byref(head))
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        rc = lib.grpo_head_forward(ctypes.byref(head), ctypes.byref(g), _ptr(out["logp"]), _ptr(out["lse"]),
                                   _ptr(out["coef"]), _ptr(out["loss3"]), _ptr(st), _ptr(ws), nbytes, stream)
    assert rc == 0, lib.gh_last_error()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out


def test_noalloc_forward_matches_workspace_forward(gpu_lib):
    lib = gpu_lib
    # calls in a row on different problems (bf16 tensor-core path, the fp32
    # path with a different scratch layout, and a bf16 forward with D > 2048,
    # whose tiles are handed out from a counter kept in the scratch); each must
    # equal the regular entry
    long_k = dataclasses.replace(CONFIGS[2], D=3072, V=3000)
    for cfg, dtype, n in ((CONFIGS[2], "bf16", None), (CONFIGS[0], "fp32", None), (long_k, "bf16", 512)):
        w, tensors, extra = _problem(cfg, dtype, n)
        want = _call(lib, tensors, extra, w["num_seqs"], noalloc=False)
        got = _call(lib, tensors, extra, w["num_seqs"], noalloc=True)
        for k in ("logp", "lse", "coef", "loss3"):
            # same kernels and same arithmetic: expected bitwise, checked with the
            # fp32 logp tolerance the parity tests use
            assert torch.isfinite(got[k]).all(), k
            assert torch.allclose(got[k], want[k], rtol=0, atol=1e-4), k
            assert torch.equal(got[k], want[k]), k


def test_noalloc_rejects_problems_larger_than_its_buffer(gpu_lib):
    lib = gpu_lib
    from gspo_logprob_gb300._abi import GhHead
    # 1M tokens x 151936 vocabulary needs ~1.25 GB of forward scratch: refused
    # on the host, before any pointer is touched or any kernel launched
    fake = 0x10000
    head = GhHead(N=1 << 20, D=4096, V=151936, dtype=0, row_tile=0, H=fake, W=fake, targets=fake, mask=fake)
    n0 = lib.gh_launch_count()
    rc = lib.grpo_head_forward_noalloc(ctypes.byref(head), None, fake, fake, None, None, fake, None)
    assert rc == 1  # GH_ERR_INVALID_ARG
    assert b"no-allocation buffer" in lib.gh_last_error()
    assert lib.gh_launch_count() == n0
