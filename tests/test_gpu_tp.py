"""Vocabulary-parallel log-prob on one GPU: the vocabulary is cut into shards
on the global 256-column split grid, each shard runs as a separate call (as
a tensor-parallel rank would), the shard outputs are gathered in shard order
and merged.  The result must equal the whole-vocabulary forward bit for bit,
for every shard count; and match the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, f32_to_bf16_bits, make_workload

from gpu_helpers import dev_head, gpu_lib, host_head  # noqa: F401

pytestmark = pytest.mark.gpu


def _tp_forward(H, W, y, m, V, P):
    import gspo_logprob_gb300 as g
    bounds = g.vocab_shard_bounds(V, P)
    outs = []
    for start, ln in bounds:
        outs.append(g.grpo_head_logprob_shard(H, W[start:start + ln], y, m, vocab_start=start, V_total=V))
    part_m = torch.cat([o["part_m"] for o in outs])          # all-gather along splits, shard order
    part_s = torch.cat([o["part_s"] for o in outs])
    zy = torch.stack([o["zy"] for o in outs])
    starts = [b[0] for b in bounds] + [V]
    merged = g.grpo_logprob_merge(part_m, part_s, zy, starts, y, m, V_total=V)
    st = sum(int(o["status"].item()) for o in outs) | int(merged["status"].item())
    return merged, st


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("P", [2, 3, 5])
def test_tp_equals_single_shard_bitwise(gpu_lib, dtype, P):
    import gspo_logprob_gb300 as g
    w = make_workload(CONFIGS[1], dtype=dtype)   # N=4096, D=256, V=5000: 20 splits
    H, W, y, m = dev_head(w)
    base = g.grpo_head_forward(H, W, y, m)
    merged, st = _tp_forward(H, W, y, m, CONFIGS[1].V, P)
    assert st == 0
    assert torch.equal(merged["lse"].view(torch.int32), base["lse"].view(torch.int32))
    assert torch.equal(merged["logp"].view(torch.int32), base["logp"].view(torch.int32))


@pytest.mark.parametrize("P", [1, 4, 7])
def test_tp_large_vocabulary_matches_oracle(gpu_lib, P):
    # V = 20000 (79 splits, ragged last tile), N ragged, targets everywhere
    import gspo_logprob_gb300 as g
    rng = np.random.default_rng(P)
    N, D, V = 1000, 128, 20000
    Hf = rng.standard_normal((N, D), dtype=np.float32)
    Wf = (rng.standard_normal((V, D)) / math.sqrt(D)).astype(np.float32)
    y = rng.integers(0, V, N).astype(np.int32)
    y[:7] = [0, 255, 256, 1023, 1024, V - 1, 19967]
    w = dict(H=f32_to_bf16_bits(Hf), W=f32_to_bf16_bits(Wf), targets=y, mask=np.ones(N, np.uint8), dtype="bf16")
    Hd, Wd, yd, md = dev_head(w)
    merged, st = _tp_forward(Hd, Wd, yd, md, V, P)
    assert st == 0
    base = g.grpo_head_forward(Hd, Wd, yd, md)
    assert torch.equal(merged["lse"].view(torch.int32), base["lse"].view(torch.int32))
    assert torch.equal(merged["logp"].view(torch.int32), base["logp"].view(torch.int32))
    lp_o, lse_o, _ = oracle.selected_logprob(*host_head(w), y)
    assert np.max(np.abs(merged["logp"].cpu().numpy() - lp_o)) < 1e-3
    assert np.max(np.abs(merged["lse"].cpu().numpy() - lse_o)) < 1e-3


@pytest.mark.parametrize("P", [2, 3])
def test_tp_long_k_shards_equal_whole_bitwise(gpu_lib, P):
    # D = 2560 (40 K blocks): the whole-vocabulary forward takes its tiles on
    # demand from a counter in its workspace, the shards (no workspace) deal
    # theirs round-robin; every tile is the same computation either way
    import gspo_logprob_gb300 as g
    rng = np.random.default_rng(40 + P)
    N, D, V = 1100, 2560, 9000
    Hf = rng.standard_normal((N, D), dtype=np.float32)
    Wf = (rng.standard_normal((V, D)) / math.sqrt(D)).astype(np.float32)
    y = rng.integers(0, V, N).astype(np.int32)
    w = dict(H=f32_to_bf16_bits(Hf), W=f32_to_bf16_bits(Wf), targets=y, mask=np.ones(N, np.uint8), dtype="bf16")
    Hd, Wd, yd, md = dev_head(w)
    base = g.grpo_head_forward(Hd, Wd, yd, md)
    merged, st = _tp_forward(Hd, Wd, yd, md, V, P)
    assert st == 0 and int(base["status"].item()) == 0
    assert torch.equal(merged["lse"].view(torch.int32), base["lse"].view(torch.int32))
    assert torch.equal(merged["logp"].view(torch.int32), base["logp"].view(torch.int32))
    lp_o, lse_o, _ = oracle.selected_logprob(*host_head(w), y)
    assert np.max(np.abs(base["lse"].cpu().numpy() - lse_o)) < 3e-2


def test_tp_out_of_range_targets(gpu_lib):
    w = make_workload(CONFIGS[1], dtype="bf16")
    y = w["targets"].copy()
    m = w["mask"].copy()
    y[7], y[8] = 5000, -3
    m[8] = 0
    w.update(targets=y, mask=m)
    H, W, yd, md = dev_head(w)
    merged, st = _tp_forward(H, W, yd, md, 5000, 3)
    assert st & 1                           # GH_DEV_TARGET_OOR
    lp = merged["logp"].cpu().numpy()
    assert math.isnan(lp[7]) and lp[8] == 0.0


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("P", [2, 4])
def test_tp_backward(gpu_lib, P, dtype):
    # vocabulary-parallel backward: each shard's dlogits use the full-vocabulary
    # LSE and coef; dW rows come out bitwise equal to the single-shard backward
    # (the same row chunks, and fp32 K slices that do not depend on the shard's
    # width), dH is the shard-ordered sum of fp32 partials (fp32 rounding of that
    # sum differs from one accumulation), checked against the oracle
    import gspo_logprob_gb300 as g
    from gpu_helpers import FP32_GRAD_ABS, assert_grad_bf16, bf16_np, dev_tensor
    cfg = CONFIGS[2]
    w = make_workload(cfg, dtype=dtype)
    H, W = host_head(w)
    lp, lse, _ = oracle.selected_logprob(H, W, w["targets"], w["mask"])
    old = (lp + w["u_old"]).astype(np.float32)
    ref = (lp + w["u_ref"]).astype(np.float32)
    adv = oracle.group_advantages(w["rewards"], w["group_size"]).astype(np.float32)
    Hd, Wd, y, m = dev_head(w)
    V = cfg.V
    fw = g.grpo_head_forward(Hd, Wd, y, m, old_logp=dev_tensor(old), ref_logp=dev_tensor(ref), adv=dev_tensor(adv),
                             seq_id=dev_tensor(w["seq_id"]), num_seqs=w["num_seqs"], eps_low=cfg.eps_low,
                             eps_high=cfg.eps_high, beta=cfg.beta)
    whole = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"])
    bounds = g.vocab_shard_bounds(V, P)
    parts = [g.grpo_head_backward_shard(Hd, Wd[s:s + n], y, m, fw["lse"], fw["coef"], vocab_start=s, V_total=V)
             for s, n in bounds]
    dW = torch.cat([p["dW"] for p in parts])
    dH = g.grpo_dh_merge(torch.stack([p["dH_partial"] for p in parts]), dtype=Hd.dtype)
    torch.cuda.synchronize()
    assert all(int(p["status"].item()) == 0 for p in parts)
    assert torch.equal(dW.view(torch.int32), whole["dW"].view(torch.int32))
    o = oracle.forward_backward(H, W, w["targets"], w["mask"], w["seq_id"], adv.astype(np.float64), w["num_seqs"],
                                old.astype(np.float64), ref.astype(np.float64), cfg.eps_low, cfg.eps_high, cfg.beta)
    if dtype == "bf16":
        assert_grad_bf16(bf16_np(dH), o["dH"], "dH (tensor parallel)")
        assert_grad_bf16(bf16_np(whole["dH"]), bf16_np(dH), "dH tp vs single")
    else:
        assert np.max(np.abs(dH.cpu().numpy() - o["dH"])) <= FP32_GRAD_ABS
        assert np.max(np.abs(dW.cpu().numpy() - o["dW"])) <= FP32_GRAD_ABS
