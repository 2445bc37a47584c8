"""Pins for the oracle's selected log-prob and streamed LSE (CPU only).

Each test ties the oracle to something other than itself: a closed form,
a library routine (scipy.special.logsumexp) or an invariant that a dropped
term, a wrong index or a padding mistake would break."""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from synth import CONFIGS, bf16_bits_to_f32, f32_to_bf16_bits, make_workload


def _rand(n, d, v, seed=0, wstd=None):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((n, d))
    W = rng.standard_normal((v, d)) * (wstd if wstd else 1.0 / math.sqrt(d))
    y = rng.integers(0, v, size=n)
    return H, W, y


def test_zero_weight_gives_log_V():
    # W = 0: every logit is 0, so LSE = log V over the REAL vocabulary
    # (log 500, not log 512: padding must not count) and logp = -log V.
    V, D, N = 500, 64, 17
    H = np.random.default_rng(1).standard_normal((N, D))
    W = np.zeros((V, D))
    y = np.arange(N) * 29 % V
    logp, lse, bad = oracle.selected_logprob(H, W, y)
    assert bad == 0
    np.testing.assert_allclose(lse, math.log(500.0), rtol=0, atol=1e-13)
    np.testing.assert_allclose(logp, -math.log(500.0), rtol=0, atol=1e-13)
    assert abs(math.log(512.0) - lse[0]) > 0.02


def test_one_hot_gather_closed_form():
    # D = V = 13, W = I, H_i = 30 e_{k_i}: z_i = 30 e_{k_i}.  logp of the hot
    # column is -log(1 + (V-1) e^-30); any other target gets 30 less.  A
    # transposed or shifted gather lands on the wrong branch.
    V = 13
    rng = np.random.default_rng(2)
    k = rng.integers(0, V, size=40)
    H = np.zeros((40, V))
    H[np.arange(40), k] = 30.0
    W = np.eye(V)
    y = np.where(np.arange(40) % 2 == 0, k, (k + 1 + np.arange(40) % 5) % V)
    logp, lse, _ = oracle.selected_logprob(H, W, y)
    base = -math.log1p((V - 1) * math.exp(-30.0))
    for i in range(40):
        want = base if y[i] == k[i] else base - 30.0
        assert abs(logp[i] - want) < 1e-12, (i, logp[i], want)
        assert abs(lse[i] - (30.0 - base)) < 1e-12


def test_lse_matches_library_logsumexp():
    H, W, y = _rand(33, 24, 301, seed=3, wstd=0.7)
    logp, lse, _ = oracle.selected_logprob(H, W, y, chunk_rows=8)
    Z = H @ W.T
    np.testing.assert_allclose(lse, logsumexp(Z, axis=1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(logp, Z[np.arange(33), y] - logsumexp(Z, axis=1), atol=1e-12)


def test_softmax_rows_sum_to_one():
    H, W, y = _rand(20, 16, 97, seed=4, wstd=1.5)
    _, lse, _ = oracle.selected_logprob(H, W, y)
    P = np.exp(H @ W.T - lse[:, None])
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-13)


def test_shift_invariance():
    # Append a constant feature: z_ij -> z_ij + c for every j.  logp must not
    # move and LSE must move by exactly c.
    H, W, y = _rand(12, 10, 50, seed=5)
    c = 3.25
    H2 = np.concatenate([H, np.ones((12, 1))], axis=1)
    W2 = np.concatenate([W, np.full((50, 1), c)], axis=1)
    lp1, lse1, _ = oracle.selected_logprob(H, W, y)
    lp2, lse2, _ = oracle.selected_logprob(H2, W2, y)
    np.testing.assert_allclose(lp2, lp1, atol=1e-12)
    np.testing.assert_allclose(lse2, lse1 + c, atol=1e-12)


def test_logp_nonpositive():
    H, W, y = _rand(64, 8, 40, seed=6, wstd=2.0)
    logp, _, _ = oracle.selected_logprob(H, W, y)
    assert np.all(logp <= 0.0)


@pytest.mark.parametrize("chunk", [1, 7, 64, 256, 500])
def test_streamed_lse_equals_plain(chunk):
    H, W, y = _rand(9, 12, 500, seed=7, wstd=1.2)
    Z = H @ W.T
    np.testing.assert_allclose(oracle.streamed_lse(Z, chunk), logsumexp(Z, axis=1),
                               rtol=0, atol=1e-12)


def test_streamed_lse_padding_identity():
    # 500 real columns padded to 1024 with -inf: two whole 256-wide chunks are
    # all padding and must contribute the identity (-inf, 0), not NaN.
    H, W, y = _rand(5, 12, 500, seed=8)
    Z = H @ W.T
    got = oracle.streamed_lse(Z, 256, padded_width=1024)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, logsumexp(Z, axis=1), atol=1e-12)


def test_bad_targets():
    H, W, y = _rand(6, 4, 10, seed=9)
    y = y.copy()
    y[1] = 10
    y[2] = -1
    y[3] = 12
    mask = np.array([1, 1, 0, 1, 1, 1], dtype=np.uint8)
    logp, lse, bad = oracle.selected_logprob(H, W, y, mask)
    assert bad == 2
    assert math.isnan(logp[1]) and math.isnan(logp[3])
    assert logp[2] == 0.0
    assert np.all(np.isfinite(lse))


def test_bf16_roundtrip_exact():
    # the synth bf16 bits and the oracle's upcast agree, and rounding is to
    # nearest even (1 + 2^-8 is a tie and rounds to 1; 1 + 3*2^-8 rounds up).
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 3.0e-3], dtype=np.float32)
    b = f32_to_bf16_bits(x)
    f = bf16_bits_to_f32(b)
    assert f[0] == 1.0 and f[1] == 1.0 and f[2] == np.float32(1.0 + 2**-6)
    assert f[3] == -2.5
    np.testing.assert_array_equal(oracle.as_f64(b, "bf16"), f.astype(np.float64))


def test_synth_is_deterministic():
    cfg = CONFIGS[0]
    a = make_workload(cfg)
    b = make_workload(cfg)
    for k in ("H", "W", "targets", "mask", "seq_id", "rewards", "u_old", "u_ref"):
        np.testing.assert_array_equal(a[k], b[k])
    assert a["H"].shape == (256, 64) and a["W"].shape == (500, 64)
