"""Pins for the oracle's analytic head gradients (CPU): central finite
differences of the whole loss in H and W, and the vanishing row/column sums
that follow from softmax rows summing to one."""
import numpy as np
import pytest

import oracle


def _tiny(seed, N=12, D=6, V=13):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * 0.8
    y = rng.integers(0, V, N)
    nseq, T = 3, N // 3
    seq = np.repeat(np.arange(nseq), T)
    mask = np.ones(N, dtype=np.uint8)
    mask[T - 1] = 0
    mask[2 * T - 2:2 * T] = 0
    adv = np.array([0.9, -1.3, 0.4])
    logp0, _, _ = oracle.selected_logprob(H, W, y)
    old = logp0 + rng.uniform(-0.5, 0.5, N)
    ref = logp0 + rng.uniform(-0.3, 0.3, N)
    return H, W, y, mask, seq, adv, nseq, old, ref


def _loss(H, W, y, mask, seq, adv, nseq, old, ref, red, norm, beta=0.1):
    logp, _, _ = oracle.selected_logprob(H, W, y, mask)
    return oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, beta, red, norm)


@pytest.mark.parametrize("red,norm", [("token_mean", 0.0), ("seq_mean", 0.0), ("fixed", 20.0)])
def test_grpo_head_gradients_finite_differences(red, norm):
    H, W, y, mask, seq, adv, nseq, old, ref = _tiny(1)
    res = oracle.forward_backward(H, W, y, mask, seq, adv, nseq, old, ref, 0.2, 0.28, 0.1, red, norm,
                                  g0=1.0)
    r = res["ratio"]
    assert np.all((np.abs(r - 0.8) > 1e-3) & (np.abs(r - 1.28) > 1e-3))
    h = 1e-6
    for X, G in ((H, res["dH"]), (W, res["dW"])):
        for idx in np.ndindex(*X.shape):
            x0 = X[idx]
            X[idx] = x0 + h
            up = _loss(H, W, y, mask, seq, adv, nseq, old, ref, red, norm)["loss"]
            X[idx] = x0 - h
            dn = _loss(H, W, y, mask, seq, adv, nseq, old, ref, red, norm)["loss"]
            X[idx] = x0
            fd = (up - dn) / (2 * h)
            assert abs(fd - G[idx]) < 1e-7, (idx, fd, G[idx])


def test_grad_output_scales_linearly():
    H, W, y, mask, seq, adv, nseq, old, ref = _tiny(2)
    a = oracle.forward_backward(H, W, y, mask, seq, adv, nseq, old, ref, 0.2, 0.28, 0.1, g0=1.0)
    b = oracle.forward_backward(H, W, y, mask, seq, adv, nseq, old, ref, 0.2, 0.28, 0.1, g0=-2.5)
    np.testing.assert_allclose(b["dH"], -2.5 * a["dH"], atol=1e-14)
    np.testing.assert_allclose(b["dW"], -2.5 * a["dW"], atol=1e-14)


def test_gspo_head_gradients_finite_differences():
    rng = np.random.default_rng(3)
    N, D, V, S = 10, 5, 11, 3
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D))
    y = rng.integers(0, V, N)
    seg = np.array([0, 0, 0, 1, 1, 2, 2, 2, 2, -1])
    mask = np.array([1, 1, 1, 1, 1, 1, 0, 1, 1, 0], dtype=np.uint8)
    adv = np.array([1.1, -0.7, 0.5])
    logp0, lse0, _ = oracle.selected_logprob(H, W, y)
    old = logp0 + rng.uniform(-0.2, 0.2, N)

    def f(H, W):
        lp, _, _ = oracle.selected_logprob(H, W, y, mask)
        return oracle.gspo_loss(lp, old, mask, seg, S, adv, 0.3, 0.3, 3.0)

    res = f(H, W)
    dH, dW = oracle.head_backward(H, W, y, lse0, res["coef"])
    h = 1e-6
    for X, G in ((H, dH), (W, dW)):
        for idx in np.ndindex(*X.shape):
            x0 = X[idx]
            X[idx] = x0 + h
            up = f(H, W)["loss"]
            X[idx] = x0 - h
            dn = f(H, W)["loss"]
            X[idx] = x0
            assert abs((up - dn) / (2 * h) - G[idx]) < 1e-7


def test_dlogits_rows_and_dW_columns_sum_to_zero():
    H, W, y, mask, seq, adv, nseq, old, ref = _tiny(4, N=24, D=7, V=29)
    res = oracle.forward_backward(H, W, y, mask, seq, adv, nseq, old, ref, 0.2, 0.28, 0.1)
    G = oracle.dlogits(H, W, y, res["lse"], res["coef"])
    np.testing.assert_allclose(G.sum(axis=1), 0.0, atol=1e-15)
    np.testing.assert_allclose(res["dW"].sum(axis=0), 0.0, atol=1e-13)
    # inactive rows get no gradient at all
    assert np.all(res["dH"][mask == 0] == 0.0)


def test_chunked_backward_matches_unchunked():
    H, W, y, mask, seq, adv, nseq, old, ref = _tiny(5, N=30, D=4, V=9)
    res = oracle.forward_backward(H, W, y, mask, seq, adv, nseq, old, ref, 0.2, 0.28, 0.1)
    a = oracle.head_backward(H, W, y, res["lse"], res["coef"], chunk_rows=7)
    np.testing.assert_allclose(a[0], res["dH"], atol=1e-15)
    np.testing.assert_allclose(a[1], res["dW"], atol=1e-14)
