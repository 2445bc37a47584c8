"""Shared helpers of the GPU parity tests: device copies of synth inputs, the
oracle's view of the same inputs, and the comparison metrics the stated
tolerances are written in."""
import numpy as np
import pytest
import torch

import oracle
from synth import bf16_bits_to_f32

# tolerances stated for the method (fp32 and bf16 configurations)
FP32_LOSS_REL = 1e-5
FP32_LOGP_ABS = 1e-4
FP32_GRAD_ABS = 2e-4
BF16_LOGP_ABS = 3e-2
BF16_LOSS_REL = 2e-3
BF16_GRAD_COS = 0.999
BF16_GRAD_MAXREL = 5e-2


@pytest.fixture(scope="session")
def gpu_lib():
    """Build (if needed) and load the CUDA library; the GPU must be present."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from gspo_logprob_gb300 import build
    build()
    from gspo_logprob_gb300 import _abi
    return _abi.load()


def dev_tensor(x, dtype_name=None):
    """numpy -> CUDA tensor; uint16 arrays tagged bf16 become bfloat16 tensors (same bits)."""
    if dtype_name == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x))
    return t.cuda()


def f64(x, dtype_name):
    return oracle.as_f64(x, dtype_name)


def host_head(w):
    """float64 H, W (exact stored values) for the oracle."""
    return f64(w["H"], w["dtype"]), f64(w["W"], w["dtype"])


def dev_head(w):
    return (dev_tensor(w["H"], w["dtype"]), dev_tensor(w["W"], w["dtype"]),
            dev_tensor(w["targets"]), dev_tensor(w["mask"]))


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))


def assert_grad_bf16(got, want, name):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    cos = cosine(got, want)
    mx = float(np.max(np.abs(want)))
    err = float(np.max(np.abs(got - want)))
    assert cos >= BF16_GRAD_COS, f"{name}: cosine {cos}"
    assert err <= BF16_GRAD_MAXREL * mx, f"{name}: max abs err {err} vs max|grad| {mx}"
    return cos, err / max(mx, 1e-300)


def loss_scale(res):
    """Reference magnitude for relative loss checks: the loss can nearly cancel
    when advantages are group-normalised, so it is the larger of |loss| and the
    sum of the magnitudes of the summed terms (oracle ``abs_terms``)."""
    return max(abs(res["loss"]), res["abs_terms"])


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else \
        t.detach().cpu().numpy().astype(np.float64)


def bf16_np(t):
    """bf16 CUDA tensor -> exact float64 numpy."""
    return bf16_bits_to_f32(t.detach().cpu().view(torch.int16).numpy().view(np.uint16)).astype(np.float64)
