"""Pins for the oracle's GRPO loss and group-normalised advantages (CPU)."""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _ev(expr):
    return float(eval(expr, {"__builtins__": {}}, {"log": math.log, "exp": math.exp}))


def _grpo_case(seed, nseq=6, T=10, eps=(0.2, 0.28), spread=0.1):
    rng = np.random.default_rng(seed)
    N = nseq * T
    logp = -rng.uniform(0.1, 5.0, N)
    old = logp + rng.uniform(-spread, spread, N)
    ref = logp + rng.uniform(-0.2, 0.2, N)
    lengths = rng.integers(2, T + 1, nseq)
    mask = (np.arange(T)[None, :] < lengths[:, None]).astype(np.uint8).reshape(-1)
    seq = np.repeat(np.arange(nseq), T)
    adv = rng.standard_normal(nseq)
    return logp, old, ref, mask, seq, adv, nseq


def test_worked_example():
    g = json.load(open(GOLD))["grpo"]
    toks = g["tokens"]
    logp = np.full(len(toks), g["logp"])
    r = np.array([_ev(t["r"]) for t in toks])
    d = np.array([_ev(t["d"]) for t in toks])
    old = logp - np.log(r)
    ref = logp + d
    mask = np.array([t["mask"] for t in toks], dtype=np.uint8)
    seq = np.array([t["seq"] for t in toks])
    for red, norm, key in (("token_mean", 0.0, "token_mean"), ("seq_mean", 0.0, "seq_mean"),
                           ("fixed", 8.0, "fixed_8")):
        res = oracle.grpo_loss(logp, old, ref, mask, seq, np.array(g["adv"]), 2, g["eps_low"],
                               g["eps_high"], g["beta"], red, norm)
        exp = g["expected"][key]
        assert abs(res["policy"] - _ev(exp["policy"])) < 1e-12, red
        assert abs(res["kl"] - _ev(exp["kl"])) < 1e-12, red
        assert abs(res["loss"] - _ev(exp["loss"])) < 1e-12, red
        if "coef_scale" in exp:
            want = np.array([_ev(t["coef_num"]) for t in toks]) * _ev(exp["coef_scale"])
            np.testing.assert_allclose(res["coef"], want, rtol=0, atol=1e-12)


def test_ratio_one_beta_zero_closed_form():
    # old = logp, beta = 0: every ratio is 1 and the loss is -sum(m A)/sum(m).
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(1)
    res = oracle.grpo_loss(logp, logp, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.0)
    want = -np.sum(mask * adv[seq]) / np.sum(mask)
    assert abs(res["loss"] - want) < 1e-13


def test_clip_inactive_inside_band():
    # all ratios within [1-eps_low, 1+eps_high]: the clipped loss equals the
    # unclipped one (eps huge), and so do the gradients.
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(2, spread=0.15)
    a = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.05)
    b = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 50.0, 50.0, 0.05)
    assert abs(a["loss"] - b["loss"]) < 1e-14
    np.testing.assert_allclose(a["coef"], b["coef"], atol=1e-15)


def test_clip_active_outside_band():
    # with wide ratios some tokens clip: the loss differs from the unclipped
    # one, and clipped tokens carry no policy gradient.
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(3, spread=1.0)
    a = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.0)
    b = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 50.0, 50.0, 0.0)
    assert a["loss"] > b["loss"]  # the pessimistic bound can only raise the loss
    clipped = (a["act"] == 0) & (mask > 0)
    assert clipped.any()
    assert np.all(a["coef"][clipped] == 0.0)


def test_k3_nonnegative_and_zero_at_equality():
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(4)
    a = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 1.0)
    assert a["kl"] >= 0.0
    assert np.all(a["per_seq_kl"] >= 0.0)
    b = oracle.grpo_loss(logp, old, logp, mask, seq, adv, nseq, 0.2, 0.28, 1.0)
    assert b["kl"] == 0.0
    assert abs(b["loss"] - b["policy"]) == 0.0


def test_zero_advantage_zero_policy():
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(5, spread=0.8)
    res = oracle.grpo_loss(logp, old, ref, mask, seq, np.zeros(nseq), nseq, 0.2, 0.28, 0.0)
    assert res["policy"] == 0.0 and res["loss"] == 0.0
    assert np.all(res["coef"] == 0.0)


def test_reductions_coincide_on_equal_lengths():
    rng = np.random.default_rng(6)
    nseq, T = 5, 8
    N = nseq * T
    logp = -rng.uniform(0.1, 4, N)
    old = logp + rng.uniform(-0.3, 0.3, N)
    ref = logp + rng.uniform(-0.2, 0.2, N)
    mask = np.ones(N, dtype=np.uint8)
    seq = np.repeat(np.arange(nseq), T)
    adv = rng.standard_normal(nseq)
    a = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.2, 0.1, "token_mean")
    b = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.2, 0.1, "seq_mean")
    c = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.2, 0.1, "fixed", float(N))
    assert abs(a["loss"] - b["loss"]) < 1e-14 and abs(a["loss"] - c["loss"]) < 1e-14
    np.testing.assert_allclose(a["coef"], b["coef"], atol=1e-15)
    np.testing.assert_allclose(a["coef"], c["coef"], atol=1e-15)


def test_reductions_differ_on_unequal_lengths():
    # the normalisers differ by more than a scale factor once lengths vary
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(7)
    a = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.0, "token_mean")
    b = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.0, "seq_mean")
    assert abs(a["loss"] - b["loss"]) > 1e-6


@pytest.mark.parametrize("reduction", ["token_mean", "seq_mean", "fixed"])
def test_coef_is_derivative_of_loss(reduction):
    # central finite differences of the loss in each logp
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(8, spread=0.6)
    args = (old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.07, reduction, 37.0 if reduction == "fixed" else 0.0)
    res = oracle.grpo_loss(logp, *args)
    # skip tokens whose ratio sits within 1e-4 of a clip edge
    r = res["ratio"]
    far = (np.abs(r - 0.8) > 1e-4) & (np.abs(r - 1.28) > 1e-4)
    h = 1e-6
    for i in range(len(logp)):
        if not far[i]:
            continue
        lp = logp.copy()
        lp[i] += h
        up = oracle.grpo_loss(lp, *args)["loss"]
        lp[i] -= 2 * h
        dn = oracle.grpo_loss(lp, *args)["loss"]
        fd = (up - dn) / (2 * h)
        assert abs(fd - res["coef"][i]) < 1e-7, (i, fd, res["coef"][i])


def test_no_active_tokens():
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(9)
    z = np.zeros_like(mask)
    with pytest.raises(oracle.OracleError):
        oracle.grpo_loss(logp, old, ref, z, seq, adv, nseq, 0.2, 0.2, 0.1, "token_mean")
    with pytest.raises(oracle.OracleError):
        oracle.grpo_loss(logp, old, ref, z, seq, adv, nseq, 0.2, 0.2, 0.1, "seq_mean")
    res = oracle.grpo_loss(logp, old, ref, z, seq, adv, nseq, 0.2, 0.2, 0.1, "fixed", 16.0)
    assert res["loss"] == 0.0 and np.all(res["coef"] == 0.0)


def test_global_normaliser_splits_exactly():
    # token_mean with an external normaliser: two halves computed separately
    # with norm = total active tokens sum to the whole-batch loss.
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(10, nseq=6, T=10)
    whole = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.04)
    T = float(mask.sum())
    h = 30
    a = oracle.grpo_loss(logp[:h], old[:h], ref[:h], mask[:h], seq[:h], adv, nseq, 0.2, 0.28, 0.04,
                         "token_mean", T)
    b = oracle.grpo_loss(logp[h:], old[h:], ref[h:], mask[h:], seq[h:], adv, nseq, 0.2, 0.28, 0.04,
                         "token_mean", T)
    assert abs(a["loss"] + b["loss"] - whole["loss"]) < 1e-14
    np.testing.assert_allclose(np.concatenate([a["coef"], b["coef"]]), whole["coef"], atol=1e-16)


def test_group_advantages_match_numpy_std():
    rng = np.random.default_rng(11)
    r = rng.random(24)
    A = oracle.group_advantages(r, 8)
    for g in range(3):
        grp = r[8 * g:8 * g + 8]
        want = (grp - grp.mean()) / (np.std(grp, ddof=1) + 1e-4)
        np.testing.assert_allclose(A[8 * g:8 * g + 8], want, rtol=0, atol=1e-12)
        assert abs(A[8 * g:8 * g + 8].sum()) < 1e-9


def test_group_advantages_bernoulli_and_constant_groups():
    r = np.array([1, 1, 1, 1, 0, 1, 0, 1], dtype=np.float32)
    A = oracle.group_advantages(r, 4)
    assert np.all(A[:4] == 0.0)                    # identical rewards -> 0
    # mean 0.5, unbiased std sqrt(1/3): A = +-0.5/(sqrt(1/3)+1e-4)
    want = 0.5 / (math.sqrt(1.0 / 3.0) + 1e-4)
    np.testing.assert_allclose(A[4:], [-want, want, -want, want], atol=1e-12)
