"""fp64 CPU oracle for the chunked cross-entropy over a tied vocabulary head.

TEST INFRASTRUCTURE ONLY, under the same rule as the rest of ``oracle/``: only
``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` use it; it
shares no code with the CUDA path.

Source: "Fractus-1B training optimization -- 2026-08-22", section 1, "Bottleneck #3"
(the tied 50257-token head: logits = h W^T over the whole vocabulary, about half the
active FLOPs) and section 2, "Opt 3" (``chunked_cross_entropy(h, W, targets,
ce_chunk)``: the same mean loss and the same gradients, computed ce_chunk tokens at a
time so that only one chunk's logits exist at once, recomputed in the backward).  The
page prints no formula; the reading is the standard one:

    logits[i][j] = h_i . W_j                          (h: [N, d], W: [V, d])
    lse_i        = log sum_j exp(logits[i][j])
    loss         = (1/N) sum_i (lse_i - logits[i][y_i])
    G[i][j]      = (exp(logits[i][j] - lse_i) - [j == y_i]) * dloss / N
    dh = G W,  dW = G^T h                             (dloss: gradient of the loss)

Functions (numpy float64; ``h`` [N, d], ``W`` [V, d], ``y`` [N] integer):

* ``ce_fwd(h, W, y)``                 -> (loss, lse[N])   the definition, whole batch
* ``ce_fwd_chunked(h, W, y, chunk)``  -> (loss, lse[N])   the page's chunking
* ``ce_bwd(h, W, y, dloss=1.0)``      -> (dh, dW)
* ``ce_bwd_chunked(h, W, y, chunk, dloss=1.0)`` -> (dh, dW)

A library matmul serves as the logits and gradient contractions.  Parity status:
pinned by ``tests/test_oracle_ce.py`` (a pure-Python brute force, chunking invariance,
the shift invariance of the softmax, the W = 0 closed form, finite differences and the
zero column sums of G).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _lse_rows(logits):
    m = logits.max(axis=1, keepdims=True)
    return (m + np.log(np.exp(logits - m).sum(axis=1, keepdims=True)))[:, 0]


def ce_fwd(h, W, y):
    """Mean cross-entropy of the logits h W^T against targets y, and each row's
    log-sum-exp."""
    h, W = _f64(h), _f64(W)
    y = np.asarray(y, dtype=np.int64)
    logits = h @ W.T
    lse = _lse_rows(logits)
    n = h.shape[0]
    loss = float((lse - logits[np.arange(n), y]).sum() / n) if n else 0.0
    return loss, lse


def ce_fwd_chunked(h, W, y, chunk):
    """The same loss, ``chunk`` tokens at a time (only one chunk's logits at once)."""
    h, W = _f64(h), _f64(W)
    y = np.asarray(y, dtype=np.int64)
    n = h.shape[0]
    lse = np.empty(n)
    total = 0.0
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        logits = h[c0:c1] @ W.T
        lse[c0:c1] = _lse_rows(logits)
        total += float((lse[c0:c1] - logits[np.arange(c1 - c0), y[c0:c1]]).sum())
    return (total / n if n else 0.0), lse


def _grad_rows(logits, lse, y, scale):
    g = np.exp(logits - lse[:, None])
    g[np.arange(g.shape[0]), y] -= 1.0
    return g * scale


def ce_bwd(h, W, y, dloss=1.0):
    """Gradients of ``dloss * loss`` with respect to h and W."""
    h, W = _f64(h), _f64(W)
    y = np.asarray(y, dtype=np.int64)
    n = h.shape[0]
    if n == 0:
        return np.zeros_like(h), np.zeros_like(W)
    logits = h @ W.T
    G = _grad_rows(logits, _lse_rows(logits), y, dloss / n)
    return G @ W, G.T @ h


def ce_bwd_chunked(h, W, y, chunk, dloss=1.0):
    """The same gradients, recomputing each chunk's logits (dW summed over chunks)."""
    h, W = _f64(h), _f64(W)
    y = np.asarray(y, dtype=np.int64)
    n = h.shape[0]
    dh = np.zeros_like(h)
    dW = np.zeros_like(W)
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        logits = h[c0:c1] @ W.T
        G = _grad_rows(logits, _lse_rows(logits), y[c0:c1], dloss / n)
        dh[c0:c1] = G @ W
        dW += G.T @ h[c0:c1]
    return dh, dW
