"""Pins for the float64 oracle: facts fixed by the pages and by mathematics,
not by the oracle's own formulas.

* the four-number block example of the 1point3acres FlashAttention write-up
  (printed value 0.9999546; tests/golden/four_number.json);
* library special cases: each row of the forward equals scipy's softmax and
  logsumexp applied to that row's scores;
* closed forms: Q = 0 gives uniform attention; N = 1 gives O = V, dV = dO,
  dQ = dK = 0; causal row 0 attends only to key 0;
* central finite differences of the loss sum(O * G) on the tiny workload
  (CS349E lecture 11 demo 1: N = 48, d = 16, eps = 1e-6), over every input
  element, causal and not;
* the identity D_i = dO_i . O_i (CUDA 算子工程 ch.16 §16.1) and four gradient
  invariants that follow from rows of P summing to 1 and rows of dS summing to 0;
* the causal executed-block count T(T+1)/2 (CS349E lecture 11 demo 4).

A final group plants plausible mistakes (a dropped scale, a dropped D, a
transposed product, a flipped sign) in copies of the backward and checks that
the finite-difference pin rejects each of them.
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.special

from fa_inputs import make_inputs, to_f64, workload
from oracle import (
    attention_backward,
    attention_backward_loops,
    attention_forward,
    attention_loss,
    causal_executed_tile_pairs,
)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tiny():
    w = workload("tiny")
    q, k, v, g = (to_f64(t)[0, 0] for t in make_inputs(w))
    return w, q, k, v, g


# ---------------------------------------------------------------- forward pins

def test_four_number_example():
    with open(os.path.join(GOLDEN, "four_number.json")) as f:
        gold = json.load(f)
    scores = np.array(gold["scores"])
    values = np.array(gold["values"])
    # realise the scores as S = scale * q k^T with d = 1, q = 1, scale = 1
    Q = np.ones((1, 1))
    K = scores.reshape(-1, 1)
    V = values.reshape(-1, 1)
    # a single query row: put it among 4 rows of the same query so N_q == N_k
    Qn = np.repeat(Q, 4, axis=0)
    O, L = attention_forward(Qn, K, V, scale=1.0)
    o = O[0, 0, 0, 0]
    tol = 0.5 * 10.0 ** (-gold["full_attention_printed_decimals"])
    assert abs(o - gold["full_attention_printed"]) <= tol
    assert o == pytest.approx(2 * math.exp(10) / (2 + 2 * math.exp(10)), rel=1e-15)
    # the naive per-block average the write-up warns about gives 0.5, the oracle does not
    assert abs(o - gold["naive_block_average_printed"]) > 0.4
    assert L[0, 0, 0] == pytest.approx(10.0 + math.log(2.0 + 2.0 * math.exp(-10.0)), rel=1e-15)


def test_four_number_example_across_a_tile_boundary():
    """Same weights spread over 64 + 64 keys: the later block holds the new max."""
    N = 128
    K = np.concatenate([np.zeros(64), np.full(64, 10.0)]).reshape(N, 1)
    V = np.concatenate([np.zeros(64), np.ones(64)]).reshape(N, 1)
    Q = np.ones((N, 1))
    O, _ = attention_forward(Q, K, V, scale=1.0)
    assert abs(O[0, 0, 5, 0] - 0.9999546) <= 5e-8


@pytest.mark.parametrize("causal", [False, True])
def test_forward_rows_match_scipy_softmax(causal):
    rng = np.random.default_rng(11)
    N, d = 37, 8
    Q, K, V = (rng.standard_normal((N, d)) for _ in range(3))
    scale = 0.7
    O, L = attention_forward(Q, K, V, scale, causal=causal, rows=5)
    for i in range(N):
        keys = slice(0, i + 1) if causal else slice(0, N)
        s = scale * (K[keys] @ Q[i])
        p = scipy.special.softmax(s)
        np.testing.assert_allclose(O[0, 0, i], p @ V[keys], rtol=1e-13, atol=1e-13)
        assert L[0, 0, i] == pytest.approx(scipy.special.logsumexp(s), rel=1e-14, abs=1e-14)


def test_L_bounds():
    """max_j S_ij <= L_i <= max_j S_ij + log N."""
    rng = np.random.default_rng(5)
    N, d = 64, 16
    Q, K, V = (rng.standard_normal((N, d)) for _ in range(3))
    Q *= 4.0
    for causal in (False, True):
        _, L = attention_forward(Q, K, V, 0.25, causal)
        S = 0.25 * Q @ K.T
        if causal:
            S = np.where(np.arange(N)[None, :] > np.arange(N)[:, None], -np.inf, S)
        m = S.max(axis=1)
        assert np.all(L[0, 0] >= m - 1e-12)
        assert np.all(L[0, 0] <= m + math.log(N) + 1e-12)


# -------------------------------------------------------------- closed forms

def test_zero_queries_give_uniform_attention():
    rng = np.random.default_rng(3)
    N, d = 29, 8
    K, V, G = (rng.standard_normal((N, d)) for _ in range(3))
    Q = np.zeros((N, d))
    r = attention_backward(Q, K, V, G, scale=0.5)
    np.testing.assert_allclose(r.O[0, 0], np.broadcast_to(V.mean(axis=0), (N, d)), atol=1e-14)
    np.testing.assert_allclose(r.L[0, 0], np.full(N, math.log(N)), atol=1e-14)
    np.testing.assert_allclose(r.dV[0, 0], np.broadcast_to(G.sum(axis=0) / N, (N, d)), atol=1e-13)


def test_single_key_closed_form():
    rng = np.random.default_rng(4)
    d = 16
    Q, K, V, G = (rng.standard_normal((1, d)) for _ in range(4))
    for causal in (False, True):
        r = attention_backward(Q, K, V, G, scale=0.25, causal=causal)
        np.testing.assert_array_equal(r.O[0, 0], V)
        np.testing.assert_array_equal(r.dV[0, 0], G)
        np.testing.assert_array_equal(r.dQ[0, 0], np.zeros((1, d)))
        np.testing.assert_array_equal(r.dK[0, 0], np.zeros((1, d)))
        assert r.L[0, 0, 0] == pytest.approx(0.25 * float(Q[0] @ K[0]), rel=1e-15)


def test_causal_first_row_and_last_key():
    w, q, k, v, g = _tiny()
    r = attention_backward(q, k, v, g, w.scale, causal=True)
    np.testing.assert_array_equal(r.O[0, 0, 0], v[0])
    np.testing.assert_array_equal(r.dQ[0, 0, 0], np.zeros(w.d))
    # the last key is seen only by the last query: dV_{N-1} = P_{N-1,N-1} dO_{N-1}
    N = w.N
    s = w.scale * (k @ q[N - 1])
    p_last = math.exp(s[N - 1] - scipy.special.logsumexp(s))
    np.testing.assert_allclose(r.dV[0, 0, N - 1], p_last * g[N - 1], rtol=1e-13)


# ------------------------------------------------------ finite differences

def _fd_grads(q, k, v, g, scale, causal, eps=1e-6):
    """Central differences of sum(O * G) for every element of Q, K and V."""
    out = {}
    for name in ("Q", "K", "V"):
        base = {"Q": q, "K": k, "V": v}
        X = base[name]
        grad = np.empty_like(X)
        for r in range(X.shape[0]):
            for c in range(X.shape[1]):
                xp, xm = X.copy(), X.copy()
                xp[r, c] += eps
                xm[r, c] -= eps
                ap, am = dict(base), dict(base)
                ap[name], am[name] = xp, xm
                fp = attention_loss(ap["Q"], ap["K"], ap["V"], g, scale, causal)
                fm = attention_loss(am["Q"], am["K"], am["V"], g, scale, causal)
                grad[r, c] = (fp - fm) / (2 * eps)
        out[name] = grad
    return out


@pytest.fixture(scope="module")
def tiny_fd():
    w, q, k, v, g = _tiny()
    return {c: _fd_grads(q, k, v, g, w.scale, c) for c in (False, True)}


def _fd_error(tiny_fd, causal, dQ, dK, dV):
    fd = tiny_fd[causal]
    return max(np.abs(fd["Q"] - dQ).max(), np.abs(fd["K"] - dK).max(), np.abs(fd["V"] - dV).max())


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_finite_differences(tiny_fd, causal):
    w, q, k, v, g = _tiny()
    r = attention_backward(q, k, v, g, w.scale, causal, rows=16)
    err = _fd_error(tiny_fd, causal, r.dQ[0, 0], r.dK[0, 0], r.dV[0, 0])
    assert err <= 1e-8, err


# Plausible mistakes, planted in copies of the backward on the CPU; the
# finite-difference pin must reject every one of them.
def _mutant_grads(q, k, v, g, scale, causal, mistake):
    N = q.shape[0]
    S = scale * q @ k.T
    if causal:
        S = np.where(np.arange(N)[None, :] > np.arange(N)[:, None], -np.inf, S)
    P = np.exp(S - scipy.special.logsumexp(S, axis=1, keepdims=True))
    dV = P.T @ g
    dP = g @ v.T
    D = np.sum(P * dP, axis=1, keepdims=True)
    dS = P * (dP - D)
    dQ = scale * dS @ k
    dK = scale * dS.T @ q
    if mistake == "dK_without_scale":
        dK = dS.T @ q
    elif mistake == "dropped_D":
        dS = P * dP
        dQ, dK = scale * dS @ k, scale * dS.T @ q
    elif mistake == "dV_transposed_P":
        dV = P @ g
    elif mistake == "D_sign":
        dS = P * (dP + D)
        dQ, dK = scale * dS @ k, scale * dS.T @ q
    elif mistake == "dK_uses_K":
        dK = scale * dS.T @ k
    elif mistake == "none":
        pass
    else:
        raise ValueError(mistake)
    return dQ, dK, dV


@pytest.mark.parametrize("mistake", ["dK_without_scale", "dropped_D", "dV_transposed_P", "D_sign", "dK_uses_K"])
def test_finite_differences_reject_planted_mistakes(tiny_fd, mistake):
    w, q, k, v, g = _tiny()
    for causal in (False, True):
        dQ, dK, dV = _mutant_grads(q, k, v, g, w.scale, causal, mistake)
        assert _fd_error(tiny_fd, causal, dQ, dK, dV) > 1e-4
    dQ, dK, dV = _mutant_grads(q, k, v, g, w.scale, False, "none")
    assert _fd_error(tiny_fd, False, dQ, dK, dV) <= 1e-8


# ------------------------------------------------------ identity, invariants

@pytest.mark.parametrize("causal", [False, True])
def test_D_identity(causal):
    rng = np.random.default_rng(8)
    B, H, N, d = 2, 2, 70, 16
    Q, K, V, G = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    r = attention_backward(Q, K, V, G, 0.3, causal, rows=32)
    assert np.abs(r.D - r.D_from_O).max() <= 1e-12 * max(1.0, np.abs(r.D).max())


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants(causal):
    rng = np.random.default_rng(9)
    N, d = 83, 16
    Q, K, V, G = (rng.standard_normal((N, d)) for _ in range(4))
    Q *= 2.0
    scale = 0.25
    r = attention_backward(Q, K, V, G, scale, causal, rows=20)
    dQ, dK, dV, D = r.dQ[0, 0], r.dK[0, 0], r.dV[0, 0], r.D[0, 0]
    # (i) rows of dS sum to zero -> sum_j dK_j = 0
    np.testing.assert_allclose(dK.sum(axis=0), 0.0, atol=1e-12)
    # (ii) rows of P sum to one -> sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dV.sum(axis=0), G.sum(axis=0), atol=1e-12)
    # (iii) S is bilinear in Q and K -> sum_i <Q_i, dQ_i> = sum_j <K_j, dK_j>
    assert np.sum(Q * dQ) == pytest.approx(np.sum(K * dK), rel=1e-11, abs=1e-11)
    # (iv) sum_j <V_j, dV_j> = sum_i D_i
    assert np.sum(V * dV) == pytest.approx(np.sum(D), rel=1e-11, abs=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_blas_oracle_equals_loop_oracle(causal):
    w, q, k, v, g = _tiny()
    a = attention_backward(q, k, v, g, w.scale, causal, rows=7)
    b = attention_backward_loops(q, k, v, g, w.scale, causal)
    for name in ("O", "L", "D", "dQ", "dK", "dV"):
        x, y = getattr(a, name), getattr(b, name)
        assert np.abs(x - y).max() <= 1e-13 * max(1.0, np.abs(y).max()), name


def test_row_block_size_does_not_change_results():
    rng = np.random.default_rng(12)
    N, d = 100, 8
    Q, K, V, G = (rng.standard_normal((N, d)) for _ in range(4))
    a = attention_backward(Q, K, V, G, 0.4, True, rows=100)
    b = attention_backward(Q, K, V, G, 0.4, True, rows=13)
    for name in ("dQ", "dK", "dV", "L"):
        np.testing.assert_allclose(getattr(a, name), getattr(b, name), rtol=1e-13, atol=1e-14)


# ------------------------------------------------------ causal block counts

@pytest.mark.parametrize("N,B", [(4096, 64), (4096, 128), (4096, 256), (8192, 128), (4000, 128), (33, 16)])
def test_causal_executed_pairs(N, B):
    T = -(-N // B)
    assert causal_executed_tile_pairs(N, B, B) == T * (T + 1) // 2
    if N % B == 0:
        frac = causal_executed_tile_pairs(N, B, B) / (T * T)
        assert frac == pytest.approx(0.5 + 0.5 / T)


def test_workload_shapes_match_page_sizes():
    with open(os.path.join(GOLDEN, "page_sizes.json")) as f:
        gold = json.load(f)
    w = workload("causal")
    assert (w.B, w.H, w.N, w.d) == (gold["B"], gold["H"], gold["N"], gold["d"])
    assert w.B * w.H * w.N * w.d * 2 == gold["Q_bytes"]
    assert w.B * w.H * w.N * w.N * 2 == gold["S_bf16_bytes"]
    assert w.B * w.H * w.N * 4 == gold["L_fp32_bytes"]


def _live_pairs_by_elements(N, Nk, Br, Bc, causal):
    """Brute force over every (query, key) entry: a block pair is live iff
    some entry in it is visible (j <= i + Nk - N under the causal mask)."""
    i = np.arange(N)[:, None]
    j = np.arange(Nk)[None, :]
    vis = (j <= i + (Nk - N)) if causal else np.ones((N, Nk), dtype=bool)
    count = 0
    for q0 in range(0, N, Br):
        for k0 in range(0, Nk, Bc):
            count += bool(vis[q0:q0 + Br, k0:k0 + Bc].any())
    return count


@pytest.mark.parametrize("N,Nk,Br,Bc", [(300, 300, 64, 64), (200, 330, 128, 128), (330, 200, 128, 128),
                                         (1000, 777, 128, 128), (257, 129, 64, 128), (50, 700, 32, 64),
                                         (700, 50, 64, 32), (128, 128, 128, 128)])
@pytest.mark.parametrize("causal", [True, False])
def test_executed_pairs_match_element_brute_force(N, Nk, Br, Bc, causal):
    """The block-level count (first key visible to the last query) equals a
    brute force over the mask's entries, for N_q != N_k, ragged tails and
    unequal block heights; without the mask every pair counts."""
    got = causal_executed_tile_pairs(N, Br, Bc, N_k=Nk, causal=causal)
    assert got == _live_pairs_by_elements(N, Nk, Br, Bc, causal)
    if not causal:
        assert got == (-(-N // Br)) * (-(-Nk // Bc))
