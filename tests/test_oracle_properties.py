"""Property checks of the oracle over random small shapes (hypothesis; CPU).

Each property is fixed by the mathematics rather than by the oracle's own
code: softmax rows sum to one; a streamed LSE over any chunking equals the
full LSE; logp <= 0; ratio 1 with beta = 0 gives loss = -sum(m A) / sum(m);
dlogits rows and dW columns sum to zero; one-token GSPO segments reduce to
token-level PPO-clip with the same fixed normaliser."""
import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402


def _problem(seed, N, D, V, scale):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * scale
    y = rng.integers(0, V, N)
    return rng, H, W, y


@settings(max_examples=40, deadline=None)
@given(seed=st.integers(0, 2**31 - 1), N=st.integers(1, 12), D=st.integers(1, 9), V=st.integers(1, 40),
       scale=st.sampled_from([0.0, 0.1, 1.0, 4.0]), chunk=st.integers(1, 45))
def test_lse_invariants(seed, N, D, V, scale, chunk):
    _, H, W, y = _problem(seed, N, D, V, scale)
    m = np.ones(N, dtype=np.uint8)
    lp, lse, _ = oracle.selected_logprob(H, W, y, m)
    Z = oracle.head_logits(H, W)
    P = np.exp(Z - lse[:, None])
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(lp <= 1e-12)
    np.testing.assert_allclose(oracle.streamed_lse(Z, chunk), lse, atol=1e-11)
    if scale == 0.0:   # W = 0: every logit is 0, LSE = log V exactly
        np.testing.assert_allclose(lse, np.log(V), atol=1e-12)


@settings(max_examples=30, deadline=None)
@given(seed=st.integers(0, 2**31 - 1), nseq=st.integers(1, 5), T=st.integers(1, 7),
       red=st.sampled_from(["token_mean", "seq_mean", "fixed"]))
def test_ratio_one_closed_form(seed, nseq, T, red):
    # old = logp and beta = 0: every ratio is 1, so each token's term is -A_s and
    # the loss is -sum_i w_i A_s(i)
    rng = np.random.default_rng(seed)
    N = nseq * T
    logp = -rng.uniform(0.1, 5.0, N)
    mask = (rng.random(N) < 0.7).astype(np.uint8)
    mask[0] = 1
    seq = np.repeat(np.arange(nseq), T)
    A = rng.standard_normal(nseq)
    norm = 3.7 if red == "fixed" else 0.0
    o = oracle.grpo_loss(logp, logp, None, mask, seq, A, nseq, 0.2, 0.28, 0.0, red, norm)
    n = np.bincount(seq[mask > 0], minlength=nseq)
    if red == "token_mean":
        want = -np.sum(mask * A[seq]) / mask.sum()
    elif red == "seq_mean":
        live = n > 0
        want = -np.sum(A[live]) / live.sum()
    else:
        want = -np.sum(mask * A[seq]) / norm
    assert abs(o["loss"] - want) <= 1e-12 * max(1.0, abs(want))


@settings(max_examples=25, deadline=None)
@given(seed=st.integers(0, 2**31 - 1), N=st.integers(1, 10), D=st.integers(1, 6), V=st.integers(2, 30))
def test_gradient_sums_vanish(seed, N, D, V):
    rng, H, W, y = _problem(seed, N, D, V, 0.7)
    m = np.ones(N, dtype=np.uint8)
    lp, lse, _ = oracle.selected_logprob(H, W, y, m)
    coef = rng.standard_normal(N)
    G = oracle.dlogits(H, W, y, lse, coef)
    np.testing.assert_allclose(G.sum(axis=1), 0.0, atol=1e-12)
    _, dW = oracle.head_backward(H, W, y, lse, coef)
    scale = np.abs(dW).sum(axis=0).max() + 1e-300
    assert np.max(np.abs(dW.sum(axis=0))) <= 1e-12 * max(1.0, scale)


@settings(max_examples=30, deadline=None)
@given(seed=st.integers(0, 2**31 - 1), N=st.integers(1, 20), div=st.floats(0.5, 50.0))
def test_one_token_segments_are_token_ppo(seed, N, div):
    rng = np.random.default_rng(seed)
    logp = -rng.uniform(0.1, 4.0, N)
    old = logp + rng.uniform(-0.6, 0.6, N)
    A = rng.standard_normal(N)
    mask = np.ones(N, dtype=np.uint8)
    seg = np.arange(N)
    g = oracle.gspo_loss(logp, old, mask, seg, N, A, 0.2, 0.28, div)
    t = oracle.grpo_loss(logp, old, None, mask, seg, A, N, 0.2, 0.28, 0.0, "fixed", div)
    assert abs(g["loss"] - t["loss"]) <= 1e-12 * max(1.0, abs(t["loss"]))
    np.testing.assert_allclose(g["coef"], t["coef"], atol=1e-13)
