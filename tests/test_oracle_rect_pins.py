"""Pins for the oracle on N_q != N_k (bottom-right causal alignment).

The pages only show N_q == N_k.  The readings for N_q != N_k (key j visible
to query i iff j <= i + N_k - N_q; a query with no visible key has O = 0,
L = +inf and zero gradients) are pinned here by facts that do not go through
the oracle's own rectangular code path:

* central finite differences of the loss sum(O * G), over every element of
  Q, K and V, for N_q < N_k and N_q > N_k, causal and not;
* embedding in a square problem: with N_k > N_q, the bottom-right causal
  problem is the last N_q query rows of the top-left causal square problem
  whose first N_k - N_q query rows carry dO = 0; with N_q > N_k, its
  non-empty rows are the square problem on the last N_k queries;
* closed forms for rows that see no key, and scipy's softmax / logsumexp for
  every row of a non-causal rectangular forward;
* the loop oracle equals the BLAS oracle on rectangular shapes.

A planted top-left alignment (j <= i regardless of N_k - N_q) passes the
finite-difference pin (its gradients are consistent with its own forward)
but the embedding pin rejects it.
"""

import numpy as np
import pytest
import scipy.special

from oracle import attention_backward, attention_backward_loops, attention_forward, attention_loss

SCALE = 0.35


def _inputs(nq, nk, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((nq, d))
    k = rng.standard_normal((nk, d))
    v = rng.standard_normal((nk, d))
    g = rng.standard_normal((nq, d))
    return q, k, v, g


def _fd(q, k, v, g, causal, eps=1e-6):
    base = {"Q": q, "K": k, "V": v}
    out = {}
    for name, X in base.items():
        grad = np.empty_like(X)
        for r in range(X.shape[0]):
            for c in range(X.shape[1]):
                ap, am = dict(base), dict(base)
                ap[name] = X.copy()
                am[name] = X.copy()
                ap[name][r, c] += eps
                am[name][r, c] -= eps
                fp = attention_loss(ap["Q"], ap["K"], ap["V"], g, SCALE, causal)
                fm = attention_loss(am["Q"], am["K"], am["V"], g, SCALE, causal)
                grad[r, c] = (fp - fm) / (2 * eps)
        out[name] = grad
    return out


@pytest.mark.parametrize("nq,nk", [(9, 14), (14, 9), (1, 6), (6, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_rectangular_gradients_match_finite_differences(nq, nk, causal):
    q, k, v, g = _inputs(nq, nk, 5, seed=nq * 31 + nk)
    fd = _fd(q, k, v, g, causal)
    r = attention_backward(q, k, v, g, SCALE, causal, rows=4)
    assert r.dQ.shape == (1, 1, nq, 5) and r.dK.shape == (1, 1, nk, 5) and r.dV.shape == (1, 1, nk, 5)
    err = max(np.abs(fd["Q"] - r.dQ[0, 0]).max(), np.abs(fd["K"] - r.dK[0, 0]).max(),
              np.abs(fd["V"] - r.dV[0, 0]).max())
    assert err <= 1e-8, err


def _embedded_more_keys(q, k, v, g):
    """N_k > N_q: the square causal problem with N_k - N_q leading query rows
    (their content is irrelevant; dO = 0 there)."""
    nq, nk = q.shape[0], k.shape[0]
    rng = np.random.default_rng(5)
    pad = nk - nq
    qs = np.concatenate([rng.standard_normal((pad, q.shape[1])), q])
    gs = np.concatenate([np.zeros((pad, g.shape[1])), g])
    return attention_backward(qs, k, v, gs, SCALE, True, rows=7), pad


def test_bottom_right_causal_is_the_tail_of_the_square_problem():
    q, k, v, g = _inputs(13, 40, 6, seed=1)
    r = attention_backward(q, k, v, g, SCALE, True, rows=5)
    sq, pad = _embedded_more_keys(q, k, v, g)
    np.testing.assert_allclose(r.O[0, 0], sq.O[0, 0, pad:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r.L[0, 0], sq.L[0, 0, pad:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r.dQ[0, 0], sq.dQ[0, 0, pad:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r.dK[0, 0], sq.dK[0, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r.dV[0, 0], sq.dV[0, 0], rtol=1e-12, atol=1e-13)


def test_more_queries_than_keys_empty_rows_and_square_tail():
    nq, nk, d = 30, 11, 6
    q, k, v, g = _inputs(nq, nk, d, seed=2)
    r = attention_backward(q, k, v, g, SCALE, True, rows=8)
    empty = nq - nk  # rows i < nq - nk see no key
    assert np.all(r.O[0, 0, :empty] == 0.0)
    assert np.all(np.isposinf(r.L[0, 0, :empty]))
    assert np.all(r.dQ[0, 0, :empty] == 0.0)
    assert np.all(r.D[0, 0, :empty] == 0.0)
    sq = attention_backward(q[empty:], k, v, g[empty:], SCALE, True, rows=8)
    for name in ("O", "L", "dQ"):
        np.testing.assert_allclose(getattr(r, name)[0, 0, empty:], getattr(sq, name)[0, 0], rtol=1e-12, atol=1e-13)
    for name in ("dK", "dV"):
        np.testing.assert_allclose(getattr(r, name)[0, 0], getattr(sq, name)[0, 0], rtol=1e-12, atol=1e-13)


def test_non_causal_rectangular_rows_match_scipy():
    q, k, v, _ = _inputs(17, 29, 4, seed=3)
    O, L = attention_forward(q, k, v, SCALE, False, rows=6)
    s = SCALE * q @ k.T
    np.testing.assert_allclose(L[0, 0], scipy.special.logsumexp(s, axis=1), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(O[0, 0], scipy.special.softmax(s, axis=1) @ v, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("nq,nk", [(7, 12), (12, 7)])
@pytest.mark.parametrize("causal", [False, True])
def test_rectangular_blas_equals_loops(nq, nk, causal):
    q, k, v, g = _inputs(nq, nk, 4, seed=4 + nq)
    a = attention_backward(q, k, v, g, SCALE, causal, rows=3)
    b = attention_backward_loops(q, k, v, g, SCALE, causal)
    for name in ("O", "L", "D", "dQ", "dK", "dV"):
        x, y = getattr(a, name), getattr(b, name)
        fin = np.isfinite(y)
        assert np.array_equal(np.isfinite(x), fin), name
        assert np.abs(x[fin] - y[fin]).max() <= 1e-13 * max(1.0, np.abs(y[fin]).max()), name


def test_planted_top_left_alignment_is_rejected():
    """Top-left masking on a rectangular problem: self-consistent, so finite
    differences cannot see it, but it is not the tail of the square problem."""
    q, k, v, g = _inputs(13, 40, 6, seed=1)
    s = SCALE * q @ k.T
    s = np.where(np.arange(40)[None, :] > np.arange(13)[:, None], -np.inf, s)
    P = np.exp(s - scipy.special.logsumexp(s, axis=1, keepdims=True))
    O_wrong = P @ v
    sq, pad = _embedded_more_keys(q, k, v, g)
    assert np.abs(O_wrong - sq.O[0, 0, pad:]).max() > 1e-3
