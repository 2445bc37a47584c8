"""Seeded random shapes against the fp64 oracle: forward (logp, LSE), GRPO loss
and coef, and backward (dH, dW), bf16 and fp32.  The shapes are ragged on
purpose: N of 1 and just past a row tile, V = 1 and vocabularies ending one
column into a tile or one column into a second and third backward block, D of
8 (bf16) and D not a multiple of 4 (fp32).  Masks, sequence layouts (with
empty sequences), groups, targets (including column V-1) and the reduction are
drawn per case."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from synth import f32_to_bf16_bits

from gpu_helpers import (BF16_LOGP_ABS, BF16_LOSS_REL, FP32_GRAD_ABS, FP32_LOGP_ABS, FP32_LOSS_REL,  # noqa: F401
                         assert_grad_bf16, bf16_np, dev_head, dev_tensor, gpu_lib, host_head, loss_scale)

pytestmark = pytest.mark.gpu

CASES = [  # dtype, N, D, V
    ("bf16", 1, 8, 1), ("bf16", 7, 16, 3), ("bf16", 255, 24, 257), ("bf16", 257, 136, 1023),
    ("bf16", 513, 64, 5000), ("bf16", 1000, 520, 4097), ("bf16", 2049, 128, 16385), ("bf16", 300, 256, 32769),
    ("bf16", 64, 8, 256), ("bf16", 129, 72, 511),
    ("fp32", 1, 3, 1), ("fp32", 33, 17, 100), ("fp32", 300, 64, 300), ("fp32", 130, 130, 1030),
    ("fp32", 517, 5, 2000), ("fp32", 64, 256, 17000),
]


def _inputs(dtype, N, D, V, seed):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, D)).astype(np.float32)
    W = (rng.standard_normal((V, D)) * (1.5 / math.sqrt(D))).astype(np.float32)
    G = int(rng.choice([1, 2, 4]))
    S = G * int(rng.integers(1, 4))
    cuts = np.sort(rng.integers(0, N + 1, S - 1))
    seq = np.searchsorted(cuts, np.arange(N), side="right").astype(np.int32)   # nondecreasing, may skip ids
    mask = (rng.random(N) < 0.85).astype(np.uint8)
    mask[0] = 1
    y = rng.integers(0, V, N).astype(np.int32)
    y[-1] = V - 1
    w = dict(H=f32_to_bf16_bits(H) if dtype == "bf16" else H, W=f32_to_bf16_bits(W) if dtype == "bf16" else W,
             targets=y, mask=mask, seq_id=seq, dtype=dtype)
    rewards = (rng.random(S) < 0.5).astype(np.float32)
    reduction = str(rng.choice(["token_mean", "seq_mean", "fixed"]))
    norm = float(rng.integers(1, 2 * N + 1)) if reduction == "fixed" else 0.0
    return w, rng, G, S, rewards, reduction, norm


@pytest.mark.parametrize("dtype,N,D,V", CASES, ids=lambda x: str(x))
def test_random_shapes_match_oracle(gpu_lib, dtype, N, D, V):
    import gspo_logprob_gb300 as g
    seed = zlib.crc32(f"{dtype}-{N}-{D}-{V}".encode())
    w, rng, G, S, rewards, reduction, norm = _inputs(dtype, N, D, V, seed)
    Hh, Wh = host_head(w)
    lp, lse, _ = oracle.selected_logprob(Hh, Wh, w["targets"], w["mask"])
    old = (lp + rng.uniform(-0.05, 0.05, N)).astype(np.float32)
    ref = (lp + rng.uniform(-0.2, 0.2, N)).astype(np.float32)
    adv = oracle.group_advantages(rewards.astype(np.float64), G).astype(np.float32)
    eps_low, eps_high, beta = 0.2, 0.28, 0.04
    o = oracle.forward_backward(Hh, Wh, w["targets"], w["mask"], w["seq_id"], adv.astype(np.float64), S,
                                old.astype(np.float64), ref.astype(np.float64), eps_low, eps_high, beta, reduction,
                                norm)
    Hd, Wd, y, m = dev_head(w)
    fw = g.grpo_head_forward(Hd, Wd, y, m, old_logp=dev_tensor(old), ref_logp=dev_tensor(ref), adv=dev_tensor(adv),
                             seq_id=dev_tensor(w["seq_id"]), num_seqs=S, eps_low=eps_low, eps_high=eps_high,
                             beta=beta, reduction=reduction, norm=norm)
    bw = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"])
    torch.cuda.synchronize()
    assert int(fw["status"].item()) == 0 and int(bw["status"].item()) == 0
    tol_lp = FP32_LOGP_ABS if dtype == "fp32" else BF16_LOGP_ABS
    assert np.max(np.abs(fw["logp"].cpu().numpy() - o["logp"])) <= tol_lp
    assert np.max(np.abs(fw["lse"].cpu().numpy() - o["lse"])) <= tol_lp
    loss = fw["loss3"].cpu().numpy().astype(np.float64)
    rel = FP32_LOSS_REL if dtype == "fp32" else BF16_LOSS_REL
    assert abs(loss[0] - o["loss"]) <= rel * max(loss_scale(o), 1e-30), (loss, o["loss"])
    coef = fw["coef"].cpu().numpy()
    assert np.max(np.abs(coef - o["coef"])) <= (1e-5 if dtype == "fp32" else 2e-3) * max(1e-30, np.abs(o["coef"]).max())
    if dtype == "fp32":
        dH, dW = bw["dH"].cpu().numpy(), bw["dW"].cpu().numpy()
        assert np.max(np.abs(dH - o["dH"])) <= FP32_GRAD_ABS and np.max(np.abs(dW - o["dW"])) <= FP32_GRAD_ABS
    else:
        for got, want, name in ((bf16_np(bw["dH"]), o["dH"], "dH"), (bw["dW"].cpu().numpy(), o["dW"], "dW")):
            if np.abs(want).max() == 0.0:      # V = 1: every softmax row is one-hot at the target
                assert np.abs(got).max() == 0.0, name
            else:
                assert_grad_bf16(got, want, name)
    assert np.all(bf16_np(bw["dH"])[w["mask"] == 0] == 0.0) if dtype == "bf16" else \
        np.all(bw["dH"].cpu().numpy()[w["mask"] == 0] == 0.0)
