"""Parity at the full sizes of the two large workloads, in the launch
configuration the benchmark times: the oracle recomputes sampled rows one by
one (logp, LSE, dH rows); dW is checked through properties that hold at any
size (vanishing column sums, exact grad_output scaling, determinism)."""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_workload

from gpu_helpers import BF16_LOGP_ABS, assert_grad_bf16, bf16_np, dev_head, dev_tensor, gpu_lib  # noqa: F401

pytestmark = pytest.mark.gpu


def _sample_rows(N, k, seed):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(N, size=k, replace=False))
    rows[0] = 0
    rows[-1] = N - 1
    return rows


def test_large_vocab_micro_batch_sampled_rows(gpu_lib):
    import gspo_logprob_gb300 as g
    cfg = CONFIGS[4]   # one micro-batch: N=8192, D=4096, V=151936
    w = make_workload(cfg)
    N, V = cfg.N, cfg.V
    rows = _sample_rows(N, 12, 4)
    Ws = oracle.as_f64(w["W"], "bf16")
    Hs = oracle.as_f64(w["H"][rows], "bf16")
    lp_s, lse_s, _ = oracle.selected_logprob(Hs, Ws, w["targets"][rows], w["mask"][rows])
    # old/ref: oracle log-probs on the sampled rows, a fixed stand-in elsewhere
    old = (-math.log(V) + w["u_old"]).astype(np.float32)
    ref = (-math.log(V) + w["u_ref"]).astype(np.float32)
    old[rows] = (lp_s + w["u_old"][rows]).astype(np.float32)
    ref[rows] = (lp_s + w["u_ref"][rows]).astype(np.float32)
    adv = oracle.group_advantages(w["rewards"], w["group_size"]).astype(np.float32)
    norm = float(w["mask"].sum())
    Hd, Wd, y, m = dev_head(w)
    fw = g.grpo_head_forward(Hd, Wd, y, m, old_logp=dev_tensor(old), ref_logp=dev_tensor(ref), adv=dev_tensor(adv),
                             seq_id=dev_tensor(w["seq_id"]), num_seqs=w["num_seqs"], eps_low=cfg.eps_low,
                             eps_high=cfg.eps_high, beta=cfg.beta, norm=norm)
    bw = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"])
    torch.cuda.synchronize()
    assert int(fw["status"].item()) == 0 and int(bw["status"].item()) == 0
    lp = fw["logp"].cpu().numpy()[rows]
    lse = fw["lse"].cpu().numpy()[rows]
    print(f"sampled max |dlogp| {np.max(np.abs(lp - lp_s)):.2e} |dlse| {np.max(np.abs(lse - lse_s)):.2e}")
    assert np.max(np.abs(lp - lp_s)) <= BF16_LOGP_ABS and np.max(np.abs(lse - lse_s)) <= BF16_LOGP_ABS
    # dH rows: the oracle's coefficient for the sampled rows (fixed global normaliser)
    seq = w["seq_id"][rows]
    o = oracle.grpo_loss(lp_s, old[rows].astype(np.float64), ref[rows].astype(np.float64), w["mask"][rows], seq,
                         adv.astype(np.float64), w["num_seqs"], cfg.eps_low, cfg.eps_high, cfg.beta, "token_mean",
                         norm)
    np.testing.assert_allclose(fw["coef"].cpu().numpy()[rows], o["coef"], rtol=1e-3,
                               atol=1e-3 * np.abs(o["coef"]).max())
    dH_s, _ = oracle.head_backward(Hs, Ws, w["targets"][rows], lse_s, o["coef"])
    act = w["mask"][rows] > 0
    assert act.sum() >= 3
    assert_grad_bf16(bf16_np(bw["dH"])[rows][act], dH_s[act], "dH sampled rows")
    # dW: columns of dW sum to ~0 (softmax rows sum to one; bf16 dlogits rounding aside)
    dW = bw["dW"]
    colsum = dW.double().sum(0).abs().max().item()
    colabs = dW.double().abs().sum(0).max().item()
    assert colsum <= 1e-2 * colabs, (colsum, colabs)
    # exact scaling with grad_output and bitwise determinism
    go = torch.tensor([2.0], device="cuda")
    bw2 = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"], grad_out=go)
    assert torch.equal(bw2["dW"], 2.0 * dW)
    bw3 = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"])
    assert torch.equal(bw3["dW"].view(torch.int32), dW.view(torch.int32))
    assert torch.equal(bw3["dH"].view(torch.int16), bw["dH"].view(torch.int16))


def test_gspo_full_size_sampled_rows(gpu_lib):
    import gspo_logprob_gb300 as g
    cfg = CONFIGS[3]   # N=16384, D=2048, V=32000
    w = make_workload(cfg)
    rows = _sample_rows(cfg.N, 24, 3)
    Ws = oracle.as_f64(w["W"], "bf16")
    Hs = oracle.as_f64(w["H"][rows], "bf16")
    lp_s, lse_s, _ = oracle.selected_logprob(Hs, Ws, w["targets"][rows], w["mask"][rows])
    Hd, Wd, y, m = dev_head(w)
    fw = g.grpo_head_forward(Hd, Wd, y, m)
    assert int(fw["status"].item()) == 0
    assert np.max(np.abs(fw["logp"].cpu().numpy()[rows] - lp_s)) <= BF16_LOGP_ABS
    assert np.max(np.abs(fw["lse"].cpu().numpy()[rows] - lse_s)) <= BF16_LOGP_ABS


def test_gspo_full_size_end_to_end(gpu_lib):
    # the whole packed-GSPO workload (N=16384, D=2048, V=32000), forward, loss
    # and backward, element by element against the fp64 oracle
    import gspo_logprob_gb300 as g
    from gpu_helpers import BF16_LOSS_REL, host_head
    cfg = CONFIGS[3]
    w = make_workload(cfg, masked_frac=0.1)
    H, W = host_head(w)
    lp_o, lse_o, _ = oracle.selected_logprob(H, W, w["targets"], w["mask"])
    old = (lp_o + w["u_old"]).astype(np.float32)
    A = oracle.group_advantages(w["rewards"], w["group_size"]).astype(np.float32)
    S = cfg.num_docs
    o = oracle.gspo_loss(lp_o, old.astype(np.float64), w["mask"], w["seq_id"], S, A.astype(np.float64),
                         cfg.eps_low, cfg.eps_high, float(S))
    dH_o, dW_o = oracle.head_backward(H, W, w["targets"], lse_o, o["coef"])
    Hd, Wd, y, m = dev_head(w)
    fw = g.grpo_head_forward(Hd, Wd, y, m)
    gs = g.gspo_segment_loss(fw["logp"], dev_tensor(old), m, dev_tensor(w["seq_id"]), S, dev_tensor(A),
                             eps_low=cfg.eps_low, eps_high=cfg.eps_high, divisor=float(S))
    bw = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], gs["coef"])
    torch.cuda.synchronize()
    assert int(fw["status"].item()) == 0 and int(gs["status"].item()) == 0 and int(bw["status"].item()) == 0
    assert np.max(np.abs(fw["logp"].cpu().numpy() - lp_o)) <= BF16_LOGP_ABS
    assert np.max(np.abs(fw["lse"].cpu().numpy() - lse_o)) <= BF16_LOGP_ABS
    sc = max(abs(o["loss"]), o["abs_terms"])
    assert abs(float(gs["loss"].item()) - o["loss"]) <= BF16_LOSS_REL * sc
    rho = o["seg_ratio"]
    near = (np.abs(rho - (1 - cfg.eps_low)) < 2e-5) | (np.abs(rho - (1 + cfg.eps_high)) < 2e-5)
    if not near.any():
        assert_grad_bf16(bf16_np(bw["dH"]), dH_o, "dH")
        assert_grad_bf16(bw["dW"].cpu().numpy(), dW_o, "dW")
    else:
        # a segment at a clip edge switches its gradient on or off: compare the
        # rows of documents away from the edges
        keep = np.array([s < 0 or not near[s] for s in w["seq_id"]])
        assert_grad_bf16(bf16_np(bw["dH"])[keep], dH_o[keep], "dH (rows away from clip edges)")
