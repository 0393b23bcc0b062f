"""Pins of the cross-entropy oracle (oracle/ce.py) against things other than itself:
a pure-Python brute force written from the definition, the chunking invariance the page
states ("identical mean loss, identical grads"), the softmax's invariance to a shift of
all logits of a token, the W = 0 closed form, central finite differences, and the zero
sum of each gradient row over the vocabulary."""
import math
import random

import numpy as np
import pytest

from oracle import ce


def draw(n, v, d, seed):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((n, d))
    W = 0.5 * rng.standard_normal((v, d))
    y = rng.integers(0, v, size=n)
    return h, W, y


def brute_loss(h, W, y):
    """Triple loops, math.exp / math.log: no numpy arithmetic."""
    n, d = len(h), len(h[0])
    total = 0.0
    for i in range(n):
        logits = [sum(h[i][k] * W[j][k] for k in range(d)) for j in range(len(W))]
        m = max(logits)
        lse = m + math.log(sum(math.exp(x - m) for x in logits))
        total += lse - logits[y[i]]
    return total / n


def test_matches_a_pure_python_brute_force():
    h, W, y = draw(4, 7, 5, 1)
    loss, _ = ce.ce_fwd(h, W, y)
    assert loss == pytest.approx(brute_loss(h.tolist(), W.tolist(), y.tolist()), rel=1e-13, abs=1e-13)


@pytest.mark.parametrize("chunk", [1, 2, 7, 64])
def test_chunking_changes_nothing(chunk):
    h, W, y = draw(23, 31, 9, 2)
    loss, lse = ce.ce_fwd(h, W, y)
    loss_c, lse_c = ce.ce_fwd_chunked(h, W, y, chunk)
    assert loss_c == pytest.approx(loss, rel=1e-13)
    np.testing.assert_allclose(lse_c, lse, rtol=1e-13)
    dh, dW = ce.ce_bwd(h, W, y, dloss=0.7)
    dh_c, dW_c = ce.ce_bwd_chunked(h, W, y, chunk, dloss=0.7)
    np.testing.assert_allclose(dh_c, dh, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dW_c, dW, rtol=1e-12, atol=1e-15)


def test_shift_of_every_vocabulary_row_leaves_the_loss():
    """Adding u to every row of W adds h_i . u to every logit of token i."""
    h, W, y = draw(6, 11, 4, 3)
    u = np.random.default_rng(9).standard_normal(4)
    assert ce.ce_fwd(h, W + u, y)[0] == pytest.approx(ce.ce_fwd(h, W, y)[0], rel=1e-12)


def test_zero_head_closed_form():
    """W = 0: every logit is 0, so loss = log V, lse = log V, G = (1/V - onehot) / N,
    dh = G W = 0 and dW = G^T h."""
    n, v, d = 5, 13, 3
    h, _, y = draw(n, v, d, 4)
    W = np.zeros((v, d))
    loss, lse = ce.ce_fwd(h, W, y)
    assert loss == pytest.approx(math.log(v), rel=1e-14)
    np.testing.assert_allclose(lse, math.log(v), rtol=1e-14)
    dh, dW = ce.ce_bwd(h, W, y)
    assert np.abs(dh).max() == 0.0
    G = np.full((n, v), 1.0 / v)
    G[np.arange(n), y] -= 1.0
    np.testing.assert_allclose(dW, (G / n).T @ h, rtol=1e-13, atol=1e-16)


def test_gradients_match_finite_differences():
    h, W, y = draw(3, 5, 4, 5)
    dh, dW = ce.ce_bwd(h, W, y)
    step = 1e-6
    rnd = random.Random(0)
    for _ in range(6):
        i, k = rnd.randrange(3), rnd.randrange(4)
        hp, hm = h.copy(), h.copy()
        hp[i, k] += step
        hm[i, k] -= step
        fd = (ce.ce_fwd(hp, W, y)[0] - ce.ce_fwd(hm, W, y)[0]) / (2 * step)
        assert fd == pytest.approx(dh[i, k], rel=1e-6, abs=1e-9)
        j = rnd.randrange(5)
        Wp, Wm = W.copy(), W.copy()
        Wp[j, k] += step
        Wm[j, k] -= step
        fd = (ce.ce_fwd(h, Wp, y)[0] - ce.ce_fwd(h, Wm, y)[0]) / (2 * step)
        assert fd == pytest.approx(dW[j, k], rel=1e-6, abs=1e-9)


def test_vocabulary_sum_of_dW_is_zero():
    """Each gradient row (softmax minus one-hot) sums to zero over the vocabulary, so the
    rows of dW = G^T h sum to zero."""
    h, W, y = draw(17, 29, 6, 6)
    _, dW = ce.ce_bwd(h, W, y)
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-15)


def test_empty_batch():
    h, W, y = draw(0, 5, 3, 7)
    assert ce.ce_fwd(h, W, y)[0] == 0.0
    dh, dW = ce.ce_bwd(h, W, y)
    assert dh.shape == (0, 3) and not dW.any()
