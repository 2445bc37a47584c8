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


# ---------------------------------------------------------------- two-sided cap, sequence-level ratio
def test_two_sided_cap_worked_example():
    # A = -1, r = 3, delta = 2: the capped unclipped term -2 is the min, so
    # pg = 2 and the ratio gets no gradient (the cap binds); without the cap
    # pg = 3 with gradient -A r = 3.  A = -1, r = 1.5 is below the cap:
    # unchanged.  A = +1, r = 3 is clipped by eps either way (pg = -1.2).
    r = np.array([3.0, 1.5, 3.0])
    adv = np.array([-1.0, -1.0, 1.0])
    logp = np.full(3, -2.0)
    old = logp - np.log(r)
    mask = np.ones(3, dtype=np.uint8)
    seq = np.arange(3)
    capped = oracle.grpo_loss(logp, old, None, mask, seq, adv, 3, 0.2, 0.2, 0.0, "fixed", 1.0, delta=2.0)
    free = oracle.grpo_loss(logp, old, None, mask, seq, adv, 3, 0.2, 0.2, 0.0, "fixed", 1.0)
    np.testing.assert_allclose(capped["per_seq_policy"], [2.0, 1.5, -1.2], atol=1e-12)
    np.testing.assert_allclose(free["per_seq_policy"], [3.0, 1.5, -1.2], atol=1e-12)
    np.testing.assert_allclose(capped["coef"], [0.0, 1.5, 0.0], atol=1e-12)
    np.testing.assert_allclose(free["coef"], [3.0, 1.5, 0.0], atol=1e-12)


def test_cap_above_every_ratio_changes_nothing():
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(21, spread=0.8)
    rmax = float(np.exp(np.max((logp - old)[mask > 0])))
    a = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.05)
    b = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.05, delta=rmax * 1.01)
    assert a["loss"] == b["loss"]
    np.testing.assert_array_equal(a["coef"], b["coef"])


def test_sequence_ratio_with_one_token_sequences_is_token_ratio():
    rng = np.random.default_rng(22)
    N = 30
    logp = -rng.uniform(0.1, 4, N)
    old = logp + rng.uniform(-0.6, 0.6, N)
    ref = logp + rng.uniform(-0.2, 0.2, N)
    adv = rng.standard_normal(N)
    mask = np.ones(N, dtype=np.uint8)
    seq = np.arange(N)
    for red, norm in (("token_mean", 0.0), ("seq_mean", 0.0), ("fixed", 7.0)):
        a = oracle.grpo_loss(logp, old, ref, mask, seq, adv, N, 0.2, 0.28, 0.1, red, norm, delta=1.6)
        b = oracle.grpo_loss(logp, old, ref, mask, seq, adv, N, 0.2, 0.28, 0.1, red, norm, delta=1.6,
                             ratio_level="sequence")
        assert abs(a["loss"] - b["loss"]) < 1e-14
        np.testing.assert_allclose(a["coef"], b["coef"], atol=1e-15)


def test_sequence_ratio_with_constant_log_ratio_is_token_ratio():
    # old = logp - c_s on every token of sequence s: every token ratio equals
    # the sequence ratio, so both levels give the same loss and gradient
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(23, nseq=5, T=8)
    c = np.random.default_rng(3).uniform(-0.5, 0.5, nseq)
    old = logp - c[seq]
    for red in ("token_mean", "seq_mean"):
        a = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.1, red)
        b = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.1, red, ratio_level="sequence")
        assert abs(a["loss"] - b["loss"]) < 1e-14
        np.testing.assert_allclose(a["coef"], b["coef"], atol=1e-14)


def test_sequence_ratio_matches_token_weighted_gspo():
    # beta = 0, fixed constant C: sum_s n_s pg_s / C, the GSPO loss with
    # omega_s = n_s and divisor C (two independent oracle functions)
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(24, nseq=6, T=9, spread=0.4)
    a = oracle.grpo_loss(logp, old, None, mask, seq, adv, nseq, 0.2, 0.28, 0.0, "fixed", 13.0,
                         ratio_level="sequence")
    g = oracle.gspo_loss(logp, old, mask, seq, nseq, adv, 0.2, 0.28, 13.0, token_weighted=True)
    assert abs(a["loss"] - g["loss"]) < 1e-14
    np.testing.assert_allclose(a["coef"], g["coef"], atol=1e-15)


@pytest.mark.parametrize("ratio_level,delta", [("token", 1.15), ("sequence", 0.0), ("sequence", 1.1)])
@pytest.mark.parametrize("reduction", ["token_mean", "seq_mean", "fixed"])
def test_coef_is_derivative_with_cap_and_sequence_ratio(reduction, ratio_level, delta):
    logp, old, ref, mask, seq, adv, nseq = _grpo_case(25, spread=0.5)
    args = (old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.07, reduction, 37.0 if reduction == "fixed" else 0.0,
            delta, ratio_level)
    res = oracle.grpo_loss(logp, *args)
    r = res["ratio"]
    edges = [0.8, 1.28] + ([delta] if delta > 0 else [])
    far = np.all([np.abs(r - e) > 1e-4 for e in edges], axis=0)
    if ratio_level == "sequence":
        far = np.array([far[seq == seq[i]].all() for i in range(len(logp))])
    h = 1e-6
    checked = 0
    for i in range(len(logp)):
        if not far[i]:
            continue
        lp = logp.copy()
        lp[i] += h
        up = oracle.grpo_loss(lp, *args)["loss"]
        lp[i] -= 2 * h
        dn = oracle.grpo_loss(lp, *args)["loss"]
        assert abs((up - dn) / (2 * h) - res["coef"][i]) < 1e-7, (i, res["coef"][i])
        checked += 1
    assert checked > 20
