"""Edge and limit cases on the GPU: the largest sequence / segment counts the
single-CTA loss kernels accept, one-token sequences, a vocabulary of one
column, and argument errors that must be refused on the host."""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import f32_to_bf16_bits

from gpu_helpers import dev_head, dev_tensor, gpu_lib, host_head, loss_scale  # noqa: F401

pytestmark = pytest.mark.gpu

MAX_SEQS = 16384


def test_grpo_at_the_sequence_limit(gpu_lib):
    # 16384 sequences of 2 tokens (N = 32768) with a tiny head: the per-sequence
    # shared-memory tables are at their maximum
    import gspo_logprob_gb300 as g
    rng = np.random.default_rng(1)
    S, T, D, V = MAX_SEQS, 2, 8, 16
    N = S * T
    Hf = rng.standard_normal((N, D)).astype(np.float32)
    Wf = rng.standard_normal((V, D)).astype(np.float32)
    y = rng.integers(0, V, N).astype(np.int32)
    mask = np.ones(N, np.uint8)
    mask[1::7] = 0
    seq = np.repeat(np.arange(S, dtype=np.int32), T)
    w = dict(H=f32_to_bf16_bits(Hf), W=f32_to_bf16_bits(Wf), targets=y, mask=mask, dtype="bf16")
    H, W = host_head(w)
    lp, _, _ = oracle.selected_logprob(H, W, y, mask)
    old = (lp + rng.uniform(-0.3, 0.3, N)).astype(np.float32)
    ref = (lp + rng.uniform(-0.2, 0.2, N)).astype(np.float32)
    adv = rng.standard_normal(S).astype(np.float32)
    Hd, Wd, yd, md = dev_head(w)
    for red in ("token_mean", "seq_mean"):
        fw = g.grpo_head_forward(Hd, Wd, yd, md, old_logp=dev_tensor(old), ref_logp=dev_tensor(ref),
                                 adv=dev_tensor(adv), seq_id=dev_tensor(seq), num_seqs=S, eps_low=0.2, eps_high=0.28,
                                 beta=0.04, reduction=red)
        o = oracle.grpo_loss(lp, old.astype(np.float64), ref.astype(np.float64), mask, seq, adv.astype(np.float64), S,
                             0.2, 0.28, 0.04, red)
        assert int(fw["status"].item()) == 0
        assert abs(float(fw["loss3"][0].item()) - o["loss"]) <= 2e-3 * loss_scale(o)
        r = o["ratio"]
        far = (np.abs(r - 0.8) > 1e-3) & (np.abs(r - 1.28) > 1e-3)
        np.testing.assert_allclose(fw["coef"].cpu().numpy()[far], o["coef"][far], rtol=2e-3,
                                   atol=1e-3 * np.abs(o["coef"]).max())


def test_gspo_at_the_segment_limit(gpu_lib):
    import gspo_logprob_gb300 as g
    rng = np.random.default_rng(2)
    S = MAX_SEQS
    N = 3 * S + 5
    seg = np.repeat(np.arange(S, dtype=np.int32), 3)
    seg = np.concatenate([seg, np.full(5, -1, np.int32)])
    mask = (seg >= 0).astype(np.uint8)
    logp = (-rng.uniform(0.1, 5, N)).astype(np.float32)
    old = (logp + rng.uniform(-0.2, 0.2, N)).astype(np.float32)
    A = rng.standard_normal(S).astype(np.float32)
    res = g.gspo_segment_loss(dev_tensor(logp), dev_tensor(old), dev_tensor(mask), dev_tensor(seg), S, dev_tensor(A),
                              eps_low=0.2, eps_high=0.28, divisor=float(S))
    o = oracle.gspo_loss(logp.astype(np.float64), old.astype(np.float64), mask, seg, S, A.astype(np.float64), 0.2, 0.28,
                         float(S))
    assert int(res["status"].item()) == 0
    assert abs(float(res["loss"].item()) - o["loss"]) <= 1e-5 * max(abs(o["loss"]), o["abs_terms"])
    np.testing.assert_allclose(res["seg_ratio"].cpu().numpy(), o["seg_ratio"], rtol=1e-5)


def test_single_column_vocabulary_and_single_token(gpu_lib):
    # V = 1: every LSE equals the only logit and every valid logp is exactly 0
    import gspo_logprob_gb300 as g
    for dtype in ("bf16", "fp32"):
        rng = np.random.default_rng(3)
        N, D = 1, 16
        Hf = rng.standard_normal((N, D)).astype(np.float32)
        Wf = rng.standard_normal((1, D)).astype(np.float32)
        w = dict(H=f32_to_bf16_bits(Hf) if dtype == "bf16" else Hf, W=f32_to_bf16_bits(Wf) if dtype == "bf16" else Wf,
                 targets=np.zeros(N, np.int32), mask=np.ones(N, np.uint8), dtype=dtype)
        Hd, Wd, yd, md = dev_head(w)
        out = g.grpo_head_forward(Hd, Wd, yd, md)
        H, W = host_head(w)
        assert out["logp"].cpu().numpy()[0] == 0.0
        assert abs(float(out["lse"].item()) - float((H @ W.T)[0, 0])) < 1e-5


def test_host_side_refusals(gpu_lib):
    import gspo_logprob_gb300 as g
    from gspo_logprob_gb300 import _abi
    H = torch.zeros(4, 12, dtype=torch.bfloat16, device="cuda")     # D = 12: not a multiple of 8
    W = torch.zeros(10, 12, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(4, dtype=torch.int32, device="cuda")
    m = torch.ones(4, dtype=torch.uint8, device="cuda")
    with pytest.raises(_abi.GhError, match="D % 8"):
        g.grpo_head_forward(H, W, y, m)
    H = torch.zeros(4, 16, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(10, 16, dtype=torch.bfloat16, device="cuda")
    seq = torch.zeros(4, dtype=torch.int32, device="cuda")
    z = torch.zeros(4, device="cuda")
    with pytest.raises(_abi.GhError, match="num_seqs"):
        g.grpo_head_forward(H, W, y, m, old_logp=z, ref_logp=z, adv=torch.zeros(MAX_SEQS + 1, device="cuda"),
                            seq_id=seq, num_seqs=MAX_SEQS + 1)
    with pytest.raises(_abi.GhError, match="fixed reduction"):
        g.grpo_head_forward(H, W, y, m, old_logp=z, ref_logp=z, adv=torch.zeros(1, device="cuda"), seq_id=seq,
                            num_seqs=1, reduction="fixed")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_nonfinite_input_is_flagged_and_contained(gpu_lib, dtype):
    # a NaN in one row of H (a poisoned input made on the host) sets the
    # non-finite status bit and gives that row a non-finite LSE (fmax ignores
    # NaN, so its split maxima stay -inf); every other row's logp and LSE keep
    # the bits of the clean call
    import gspo_logprob_gb300 as g
    from synth import CONFIGS, make_workload
    w = make_workload(CONFIGS[1], dtype=dtype, N=300)
    Hd, Wd, y, m = dev_head(w)
    clean = g.grpo_head_forward(Hd, Wd, y, m)
    bad = Hd.clone()
    bad[37, 11] = float("nan")
    pois = g.grpo_head_forward(bad, Wd, y, m)
    torch.cuda.synchronize()
    assert int(clean["status"].item()) == 0
    assert int(pois["status"].item()) & 2          # GH_DEV_NONFINITE
    assert not math.isfinite(float(pois["lse"][37].item()))
    keep = torch.ones(300, dtype=torch.bool, device="cuda")
    keep[37] = False
    assert torch.equal(pois["lse"][keep].view(torch.int32), clean["lse"][keep].view(torch.int32))
    assert torch.equal(pois["logp"][keep].view(torch.int32), clean["logp"][keep].view(torch.int32))
