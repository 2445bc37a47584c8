"""Pins for the oracle's GSPO segment loss (CPU)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from synth import CONFIGS, make_workload

GOLD = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _ev(expr):
    return float(eval(expr, {"__builtins__": {}}, {"log": math.log, "exp": math.exp}))


def test_worked_example():
    g = json.load(open(GOLD))["gspo"]
    toks = g["tokens"]
    logp = np.array([_ev(t["logp"]) for t in toks])
    old = logp - np.array([_ev(t["log_ratio"]) for t in toks])
    mask = np.array([t["mask"] for t in toks], dtype=np.uint8)
    seg = np.array([t["seg"] for t in toks])
    e = g["expected"]
    res = oracle.gspo_loss(logp, old, mask, seg, g["num_segments"], np.array(g["adv"]),
                           g["eps_low"], g["eps_high"], g["divisor"])
    np.testing.assert_allclose(res["seg_ratio"], [_ev(x) for x in e["seg_ratio"]], atol=1e-12)
    np.testing.assert_allclose(res["seg_loss"], [_ev(x) for x in e["seg_loss"]], atol=1e-12)
    assert abs(res["loss"] - _ev(e["loss"])) < 1e-12
    np.testing.assert_allclose(res["coef"], [_ev(x) for x in e["coef"]], atol=1e-12)
    assert abs(res["mean_logp"] - _ev(e["mean_logp"])) < 1e-12
    tw = oracle.gspo_loss(logp, old, mask, seg, g["num_segments"], np.array(g["adv"]),
                          g["eps_low"], g["eps_high"], g["divisor"], token_weighted=True)
    assert abs(tw["loss"] - _ev(e["loss_token_weighted"])) < 1e-12


def test_length_one_segments_reduce_to_token_ppo():
    # every token its own segment: the sequence-level ratio is the token
    # ratio, so GSPO with divisor C equals token PPO-clip (beta = 0) with
    # the fixed normaliser C, loss and per-token gradients alike.
    rng = np.random.default_rng(1)
    N = 40
    logp = -rng.uniform(0.1, 4, N)
    old = logp + rng.uniform(-0.5, 0.5, N)
    adv = rng.standard_normal(N)
    mask = np.ones(N, dtype=np.uint8)
    seg = np.arange(N)
    g = oracle.gspo_loss(logp, old, mask, seg, N, adv, 0.2, 0.28, 17.0)
    t = oracle.grpo_loss(logp, old, None, mask, seg, adv, N, 0.2, 0.28, 0.0, "fixed", 17.0)
    assert abs(g["loss"] - t["loss"]) < 1e-13
    np.testing.assert_allclose(g["coef"], t["coef"], atol=1e-14)


def test_single_segment_ratio_is_exp_mean():
    rng = np.random.default_rng(2)
    N = 33
    logp = -rng.uniform(0.1, 4, N)
    old = logp + rng.uniform(-0.3, 0.3, N)
    mask = (rng.random(N) < 0.8).astype(np.uint8)
    seg = np.zeros(N, dtype=np.int64)
    res = oracle.gspo_loss(logp, old, mask, seg, 1, np.array([0.7]), 0.2, 0.2, 1.0)
    want = math.exp(np.mean((logp - old)[mask > 0]))
    assert abs(res["seg_ratio"][0] - want) < 1e-13


def test_counts_match_bincount_on_packed_layout():
    w = make_workload(CONFIGS[3], N=4096, with_weight=False, masked_frac=0.1)
    mask, seg = w["mask"], w["seq_id"]
    S = CONFIGS[3].num_docs
    rng = np.random.default_rng(3)
    logp = -rng.uniform(0.1, 4, 4096)
    res = oracle.gspo_loss(logp, logp, mask, seg, S, np.ones(S), 3e-4, 4e-4, float(S))
    valid = (seg >= 0) & (mask > 0)
    np.testing.assert_array_equal(res["counts"], np.bincount(seg[valid], minlength=S))
    # ratio 1 everywhere -> every live segment loss is -A
    live = res["counts"] > 0
    np.testing.assert_allclose(res["seg_loss"][live], -1.0, atol=0)


def test_coef_is_derivative_of_loss():
    rng = np.random.default_rng(4)
    N, S = 60, 7
    seg = np.sort(rng.integers(0, S, N))
    seg[-4:] = -1
    mask = (rng.random(N) < 0.85).astype(np.uint8)
    mask[-4:] = 0
    logp = -rng.uniform(0.1, 3, N)
    old = logp + rng.uniform(-0.6, 0.6, N)
    adv = rng.standard_normal(S)
    for tw in (False, True):
        args = (old, mask, seg, S, adv, 0.1, 0.15, 5.0, tw)
        res = oracle.gspo_loss(logp, *args)
        rho = res["seg_ratio"]
        h = 1e-6
        for i in range(N):
            s = seg[i]
            if s >= 0 and (abs(rho[s] - 0.9) < 1e-4 or abs(rho[s] - 1.15) < 1e-4):
                continue
            lp = logp.copy()
            lp[i] += h
            up = oracle.gspo_loss(lp, *args)["loss"]
            lp[i] -= 2 * h
            dn = oracle.gspo_loss(lp, *args)["loss"]
            assert abs((up - dn) / (2 * h) - res["coef"][i]) < 1e-7


def test_gspo_layout_structure():
    # packed documents: contiguous, nondecreasing ids, -1 only as a tail
    w = make_workload(CONFIGS[3], with_weight=False)
    seg = w["seq_id"]
    valid = seg[seg >= 0]
    assert np.all(np.diff(valid) >= 0)
    if (seg < 0).any():
        first = np.argmax(seg < 0)
        assert np.all(seg[first:] == -1)
    assert seg.shape == (16384,)


def test_divisor_must_be_positive():
    with pytest.raises(oracle.OracleError):
        oracle.gspo_loss(np.zeros(2), np.zeros(2), np.ones(2, np.uint8), np.zeros(2, int), 1,
                         np.ones(1), 0.2, 0.2, 0.0)


def test_kl_term_length_one_segments_equal_token_grpo():
    # every token its own segment: the segment-mean KL is the token KL, so GSPO
    # with beta and divisor C equals token-level GRPO with the fixed normaliser C
    rng = np.random.default_rng(31)
    N = 36
    logp = -rng.uniform(0.1, 4, N)
    old = logp + rng.uniform(-0.4, 0.4, N)
    ref = logp + rng.uniform(-0.3, 0.3, N)
    adv = rng.standard_normal(N)
    mask = np.ones(N, dtype=np.uint8)
    seg = np.arange(N)
    g = oracle.gspo_loss(logp, old, mask, seg, N, adv, 0.2, 0.28, 11.0, ref=ref, beta=0.07)
    t = oracle.grpo_loss(logp, old, ref, mask, seg, adv, N, 0.2, 0.28, 0.07, "fixed", 11.0)
    assert abs(g["loss"] - t["loss"]) < 1e-14
    np.testing.assert_allclose(g["coef"], t["coef"], atol=1e-15)


def test_kl_term_zero_at_reference_and_nonnegative():
    w = make_workload(CONFIGS[3], N=2048, with_weight=False, masked_frac=0.1)
    rng = np.random.default_rng(32)
    logp = -rng.uniform(0.1, 4, 2048)
    old = logp + rng.uniform(-0.01, 0.01, 2048)
    S = CONFIGS[3].num_docs
    adv = rng.standard_normal(S)
    base = oracle.gspo_loss(logp, old, w["mask"], w["seq_id"], S, adv, 0.2, 0.2, 48.0)
    same = oracle.gspo_loss(logp, old, w["mask"], w["seq_id"], S, adv, 0.2, 0.2, 48.0, ref=logp, beta=0.5)
    assert abs(same["loss"] - base["loss"]) < 1e-14
    np.testing.assert_allclose(same["coef"], base["coef"], atol=1e-16)
    ref = logp + rng.uniform(-0.3, 0.3, 2048)
    kl = oracle.gspo_loss(logp, old, w["mask"], w["seq_id"], S, adv, 0.2, 0.2, 48.0, ref=ref, beta=0.5)
    assert np.all(kl["seg_kl"] >= 0.0) and kl["loss"] >= base["loss"]


def test_kl_term_coef_is_derivative():
    rng = np.random.default_rng(33)
    N, S = 50, 6
    seg = np.sort(rng.integers(0, S, N))
    seg[-3:] = -1
    mask = (rng.random(N) < 0.85).astype(np.uint8)
    mask[-3:] = 0
    logp = -rng.uniform(0.1, 3, N)
    old = logp + rng.uniform(-0.5, 0.5, N)
    ref = logp + rng.uniform(-0.3, 0.3, N)
    adv = rng.standard_normal(S)
    for tw in (False, True):
        args = (old, mask, seg, S, adv, 0.1, 0.15, 4.0, tw, ref, 0.3)
        res = oracle.gspo_loss(logp, *args)
        rho = res["seg_ratio"]
        h = 1e-6
        for i in range(N):
            s = seg[i]
            if s >= 0 and (abs(rho[s] - 0.9) < 1e-4 or abs(rho[s] - 1.15) < 1e-4):
                continue
            lp = logp.copy()
            lp[i] += h
            up = oracle.gspo_loss(lp, *args)["loss"]
            lp[i] -= 2 * h
            dn = oracle.gspo_loss(lp, *args)["loss"]
            assert abs((up - dn) / (2 * h) - res["coef"][i]) < 1e-7


def test_segment_act_by_clip_region():
    # act_s (the segment's policy term moves with rho) in each region of the
    # clip, for one-token segments with log-ratio log(rho): inside the band
    # always; above 1 + eps_high only for A < 0; below 1 - eps_low only for A > 0
    rho = np.array([1.0, 1.5, 1.5, 0.5, 0.5, 1.1])
    adv = np.array([0.7, 0.7, -0.7, 0.7, -0.7, -0.3])
    want = np.array([True, False, True, True, False, True])
    logp = np.full(6, -1.0)
    old = logp - np.log(rho)
    res = oracle.gspo_loss(logp, old, np.ones(6, np.uint8), np.arange(6), 6, adv, 0.2, 0.28, 6.0)
    assert np.array_equal(res["seg_act"], want)
    assert np.array_equal(res["coef"] != 0, want)            # the cut-off segments carry no gradient


def test_segment_act_matches_token_act_for_one_token_segments():
    # one-token segments: the segment's act is the token-level GRPO act,
    # computed by the oracle's separate token code
    rng = np.random.default_rng(9)
    N = 200
    logp = -rng.uniform(0.1, 4, N)
    old = logp + rng.uniform(-0.6, 0.6, N)
    adv = rng.standard_normal(N)
    mask = np.ones(N, dtype=np.uint8)
    seg = np.arange(N)
    g = oracle.gspo_loss(logp, old, mask, seg, N, adv, 0.2, 0.28, 5.0)
    t = oracle.grpo_loss(logp, old, None, mask, seg, adv, N, 0.2, 0.28, 0.0, "fixed", 5.0)
    assert 0 < int((~g["seg_act"]).sum()) < N
    assert np.array_equal(g["seg_act"], t["act"] > 0)
