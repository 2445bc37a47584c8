"""The O(N) loss kernels: the GRPO loss and the GSPO seam run one CTA per
sequence (segment) with a last-CTA fold, or one CTA over all of them when no
scratch slots are available.  Checked here: both launch shapes give the same
bits for every output; the clipped-token and clipped-segment counts equal the
oracle's (Fast-LLM PR #554, What: the seam's metric outputs); more sequences
than scratch slots still match the oracle."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_workload

from gpu_helpers import dev_head, dev_tensor, gpu_lib, host_head  # noqa: F401

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _child(env):
    full = dict(os.environ)
    full.update(env)
    r = subprocess.run([sys.executable, os.path.join(HERE, "loss_child.py")], env=full, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_one_cta_and_grid_give_the_same_bits(gpu_lib):
    grid = _child({"GH_LOSS_ONE_CTA": "0"})
    one = _child({"GH_LOSS_ONE_CTA": "1"})
    assert len(grid) >= 20
    diff = [k for k in grid if grid[k] != one[k]]
    assert not diff, diff


# the sequence level averages the log-ratio noise over a sequence, so it gets a
# narrow band for some sequences to clip
@pytest.mark.parametrize("reduction,ratio_level,delta,eps", [("token_mean", "token", 0.0, None),
                                                             ("seq_mean", "sequence", 0.0, 0.01),
                                                             ("fixed", "token", 1.1, None)])
def test_grpo_clipped_tokens_match_oracle(gpu_lib, reduction, ratio_level, delta, eps):
    import gspo_logprob_gb300 as g
    cfg = CONFIGS[2]
    w = make_workload(cfg, old_noise=0.5)
    H, W = host_head(w)
    lp, _, _ = oracle.selected_logprob(H, W, w["targets"], w["mask"])
    old = (lp + w["u_old"]).astype(np.float32)
    ref = (lp + w["u_ref"]).astype(np.float32)
    adv = oracle.group_advantages(w["rewards"], w["group_size"]).astype(np.float32)
    norm = 1024.0 if reduction == "fixed" else 0.0
    el, eh = (cfg.eps_low, cfg.eps_high) if eps is None else (eps, eps)
    o = oracle.grpo_loss(lp, old.astype(np.float64), ref.astype(np.float64), w["mask"], w["seq_id"],
                         adv.astype(np.float64), w["num_seqs"], el, eh, cfg.beta, reduction, norm,
                         delta=delta, ratio_level=ratio_level)
    m = w["mask"] > 0
    want = int(np.sum(m & (o["act"] == 0)))
    # tokens whose ratio sits within 1e-4 of an edge may fall either way
    r = o["ratio"]
    edges = [1 - el, 1 + eh] + ([delta] if delta > 0 else [])
    near = m & np.any([np.abs(r - e) < 1e-4 for e in edges], axis=0)
    Hd, Wd, y, md = dev_head(w)
    fw = g.grpo_head_forward(Hd, Wd, y, md, old_logp=dev_tensor(old), ref_logp=dev_tensor(ref), adv=dev_tensor(adv),
                             seq_id=dev_tensor(w["seq_id"]), num_seqs=w["num_seqs"], eps_low=el, eps_high=eh,
                             beta=cfg.beta, reduction=reduction, norm=norm, delta=delta, ratio_level=ratio_level,
                             clip_count=True)
    got = int(fw["num_clipped"].item())
    print(f"{reduction}/{ratio_level}/{delta}: clipped {got} of {int(m.sum())} active (oracle {want})")
    assert 0 < want < int(m.sum())
    assert abs(got - want) <= int(near.sum())


@pytest.mark.parametrize("band", ["config", "wide"])
def test_gspo_clipped_segments_match_oracle(gpu_lib, band):
    import gspo_logprob_gb300 as g
    cfg = CONFIGS[3]
    w = make_workload(cfg, masked_frac=0.1, with_weight=False)
    rng = np.random.default_rng(5)
    N, S = cfg.N, cfg.num_docs
    logp = (-rng.uniform(0.05, 6.0, N)).astype(np.float32)
    old = (logp.astype(np.float64) + w["u_old"]).astype(np.float32)
    A = oracle.group_advantages(w["rewards"], w["group_size"]).astype(np.float32)
    el, eh = (cfg.eps_low, cfg.eps_high) if band == "config" else (0.2, 0.2)
    o = oracle.gspo_loss(logp.astype(np.float64), old.astype(np.float64), w["mask"], w["seq_id"], S,
                         A.astype(np.float64), el, eh, float(S))
    live = o["counts"] > 0
    want = int(np.sum(live & ~o["seg_act"]))
    rho = o["seg_ratio"]
    near = live & ((np.abs(rho - (1 - el)) < 2e-5) | (np.abs(rho - (1 + eh)) < 2e-5))
    assert not near.any()
    r = g.gspo_segment_loss(dev_tensor(logp), dev_tensor(old), dev_tensor(w["mask"]), dev_tensor(w["seq_id"]), S,
                            dev_tensor(A), eps_low=el, eps_high=eh, divisor=float(S))
    got = int(r["num_clipped"].item())
    print(f"{band}: {got} of {int(live.sum())} live segments clipped (oracle {want})")
    assert got == want
    if band == "wide":
        assert want == 0
    else:
        assert 0 < want < live.sum()


def test_more_sequences_than_scratch_slots(gpu_lib):
    # 96 tokens in 80 sequences (many empty, ids skipping values): more
    # sequences than the max(64, N / 8) scratch slots, so the loss runs on one
    # CTA; it must still match the oracle
    import gspo_logprob_gb300 as g
    rng = np.random.default_rng(12)
    N, D, V, S = 96, 64, 700, 80
    H = rng.standard_normal((N, D)).astype(np.float32)
    W = (rng.standard_normal((V, D)) / 8).astype(np.float32)
    y = rng.integers(0, V, N).astype(np.int32)
    mask = (rng.random(N) < 0.8).astype(np.uint8)
    seq = np.sort(rng.integers(0, S, N)).astype(np.int32)
    lp, _, _ = oracle.selected_logprob(H.astype(np.float64), W.astype(np.float64), y, mask)
    old = (lp + rng.uniform(-0.4, 0.4, N)).astype(np.float32)
    ref = (lp + rng.uniform(-0.2, 0.2, N)).astype(np.float32)
    adv = rng.standard_normal(S).astype(np.float32)
    for red in ("token_mean", "seq_mean"):
        o = oracle.grpo_loss(lp, old.astype(np.float64), ref.astype(np.float64), mask, seq, adv.astype(np.float64),
                             S, 0.2, 0.28, 0.04, red)
        fw = g.grpo_head_forward(dev_tensor(H), dev_tensor(W), dev_tensor(y), dev_tensor(mask),
                                 old_logp=dev_tensor(old), ref_logp=dev_tensor(ref), adv=dev_tensor(adv),
                                 seq_id=dev_tensor(seq), num_seqs=S, eps_low=0.2, eps_high=0.28, beta=0.04,
                                 reduction=red, clip_count=True)
        torch.cuda.synchronize()
        assert int(fw["status"].item()) == 0
        sc = max(abs(o["loss"]), o["abs_terms"])
        assert abs(float(fw["loss3"][0].item()) - o["loss"]) <= 1e-5 * sc
        np.testing.assert_allclose(fw["coef"].cpu().numpy(), o["coef"], rtol=1e-4, atol=1e-7)
        r = o["ratio"]
        near = (mask > 0) & ((np.abs(r - 0.8) < 1e-5) | (np.abs(r - 1.28) < 1e-5))
        assert abs(int(fw["num_clipped"].item()) - int(np.sum((mask > 0) & (o["act"] == 0)))) <= int(near.sum())
