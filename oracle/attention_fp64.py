"""Plain float64 CPU oracle for scaled-dot-product attention and its backward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  It shares
no code with the CUDA library (no kernels, headers, helpers, tables or
constants) and never imports the product package.

What it computes is the dense definition of attention and of its gradient,
written out one step at a time with full rows of the N x N matrices S, P, dP and
dS materialised.  It is deliberately not tiled over keys and never uses an
online softmax, so a reader can check it against the pages by eye:

* forward  S = scale * Q K^T,  P = softmax(S) row-wise,  O = P V
  ("CUDA 算子工程" ch.16 "FA2 反向" §16.1; the scaled form with 1/sqrt(d) is
  the one in "FlashAttention 的反向传播设计" §一 and in the 1point3acres
  FlashAttention write-up, first formula);
* logsumexp  L_i = m_i + log(sum_j exp(S_ij - m_i))  (ch.16 §16.4; write-up,
  "logsumexp" paragraph), natural log, of the *scaled* scores;
* backward  dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,
  dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q
  (ch.16 §16.1 for the chain rule and the definition of D; the factor
  1/sqrt(d) on dQ and dK from "FlashAttention 的反向传播设计" §一 and from the
  write-up's remark that the gradients into Q and K carry the forward's
  1/sqrt(d); ch.16 §16.6 scales dK at write-out by softmax_scale).

Readings where the pages leave a step open:

* causal masking: the pages show only N_q == N_k, where key j is visible to
  query i iff j <= i (CS349E lecture 11 demo 4 masks the upper triangle;
  masked scores are -inf so their P is exactly 0).  For N_q != N_k the mask
  is aligned bottom-right, j <= i + (N_k - N_q): the last query sees every
  key, and at N_q == N_k this is the pages' mask;
* a query row that sees no key at all (causal, N_q > N_k) has an empty
  softmax: its O row is 0, its L is +inf (so that exp(S - L) = 0 in the
  backward) and its gradients are 0;
* D is computed by its definition (row sum of P * dP); the identity
  D_i = dO_i . O_i (ch.16 §16.1) is returned separately as ``D_from_O`` so
  tests can check the identity rather than assume it;
* all arithmetic is float64; inputs are upcast exactly from whatever dtype the
  caller used (for bf16 workloads: the bf16-rounded values).

A row-block size ``rows`` bounds memory: each block holds full rows of S, P,
dP, dS (rows x N).  Blocking over *query rows* changes nothing in the
arithmetic of a row, and dK/dV are plain sums over rows, so the result is the
dense definition.

Parity pins for every function here live in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = [
    "AttentionGrads",
    "attention_forward",
    "attention_backward",
    "attention_backward_loops",
    "attention_loss",
    "causal_executed_tile_pairs",
]


@dataclass
class AttentionGrads:
    """All float64 results for one (B, H, N_q, N_k, d) problem."""

    O: np.ndarray  # [B, H, N_q, d]
    L: np.ndarray  # [B, H, N_q]
    D: np.ndarray  # [B, H, N_q]   row sums of P * dP (definition)
    D_from_O: np.ndarray  # [B, H, N_q]  dO_i . O_i (identity of ch.16 §16.1)
    dQ: np.ndarray  # [B, H, N_q, d]
    dK: np.ndarray  # [B, H, N_k, d]
    dV: np.ndarray  # [B, H, N_k, d]


def _as4d(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    if x.ndim == 2:
        x = x[None, None]
    if x.ndim != 4:
        raise ValueError("expected [N, d] or [B, H, N, d]")
    return x


def _scores(q_rows: np.ndarray, k: np.ndarray, scale: float, row0: int, causal: bool, offset: int) -> np.ndarray:
    """S for a block of query rows starting at global row ``row0``: scale * Q K^T,
    with -inf where key j > query i + offset under the causal mask
    (offset = N_k - N_q)."""
    s = scale * (q_rows @ k.T)
    if causal:
        i = np.arange(row0, row0 + q_rows.shape[0])[:, None]
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j > i + offset, -np.inf, s)
    return s


def _softmax_rows(s: np.ndarray):
    """Row-wise max m, logsumexp L = m + log(sum exp(S - m)) and P = exp(S - L).

    Masked entries (-inf) give exactly 0.  The max is subtracted before the
    exponential as in the write-up's safe-softmax statistics (m, l).  A row
    with every entry masked gets L = +inf and P = 0."""
    m = np.max(s, axis=1)
    empty = m == -np.inf
    m_safe = np.where(empty, 0.0, m)
    ell = np.sum(np.exp(s - m_safe[:, None]), axis=1)
    with np.errstate(divide="ignore"):
        L = np.where(empty, np.inf, m_safe + np.log(np.where(empty, 1.0, ell)))
    P = np.where(empty[:, None], 0.0, np.exp(s - np.where(empty, 0.0, L)[:, None]))
    return L, P


def attention_forward(Q, K, V, scale: float, causal: bool = False, rows: int = 512):
    """Dense forward: returns (O, L), both float64.

    Q: [N_q, d] or [B, H, N_q, d]; K, V: [N_k, d] or [B, H, N_k, d].
    ``rows`` only bounds memory."""
    Q, K, V = _as4d(Q), _as4d(K), _as4d(V)
    B, H, N, d = Q.shape
    offset = K.shape[2] - N
    O = np.empty((B, H, N, V.shape[-1]))
    L = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, rows):
                r1 = min(N, r0 + rows)
                s = _scores(Q[b, h, r0:r1], K[b, h], scale, r0, causal, offset)
                Lr, P = _softmax_rows(s)
                L[b, h, r0:r1] = Lr
                O[b, h, r0:r1] = P @ V[b, h]
    return O, L


def attention_backward(Q, K, V, dO, scale: float, causal: bool = False, rows: int = 512) -> AttentionGrads:
    """Dense backward of O = softmax(scale Q K^T) V with upstream gradient dO.

    Step order follows ch.16 §16.1's list: recompute S and P, then dV = P^T dO,
    dP = dO V^T, D = rowsum(P * dP), dS = P * (dP - D), dQ = scale dS K,
    dK = scale dS^T Q.  Returns float64 O, L, D, D_from_O, dQ, dK, dV."""
    Q, K, V, dO = _as4d(Q), _as4d(K), _as4d(V), _as4d(dO)
    B, H, N, d = Q.shape
    Nk = K.shape[2]
    offset = Nk - N
    dv_dim = V.shape[-1]
    O = np.empty((B, H, N, dv_dim))
    L = np.empty((B, H, N))
    D = np.empty((B, H, N))
    D_from_O = np.empty((B, H, N))
    dQ = np.empty((B, H, N, d))
    dK = np.zeros((B, H, Nk, d))
    dV = np.zeros((B, H, Nk, dv_dim))
    for b in range(B):
        for h in range(H):
            q, k, v, g = Q[b, h], K[b, h], V[b, h], dO[b, h]
            for r0 in range(0, N, rows):
                r1 = min(N, r0 + rows)
                s = _scores(q[r0:r1], k, scale, r0, causal, offset)  # S (rows x N_k)
                Lr, P = _softmax_rows(s)                              # L, P
                o = P @ v                                             # O = P V
                dV[b, h] += P.T @ g[r0:r1]                            # dV = P^T dO
                dP = g[r0:r1] @ v.T                                   # dP = dO V^T
                Dr = np.sum(P * dP, axis=1)                           # D_i = sum_j P_ij dP_ij
                dS = P * (dP - Dr[:, None])                           # dS = P * (dP - D)
                dQ[b, h, r0:r1] = scale * (dS @ k)                    # dQ = scale dS K
                dK[b, h] += scale * (dS.T @ q[r0:r1])                 # dK = scale dS^T Q
                O[b, h, r0:r1] = o
                L[b, h, r0:r1] = Lr
                D[b, h, r0:r1] = Dr
                D_from_O[b, h, r0:r1] = np.sum(g[r0:r1] * o, axis=1)  # dO_i . O_i
    return AttentionGrads(O=O, L=L, D=D, D_from_O=D_from_O, dQ=dQ, dK=dK, dV=dV)


def attention_backward_loops(Q, K, V, dO, scale: float, causal: bool = False) -> AttentionGrads:
    """The same backward with explicit Python loops and no BLAS, for tiny
    [N_q, d] x [N_k, d] inputs only (seconds at N = 48, d = 16).  Every sum is
    written as a loop over its index, in the order of ch.16 §16.1."""
    q = np.asarray(Q, dtype=np.float64)
    k = np.asarray(K, dtype=np.float64)
    v = np.asarray(V, dtype=np.float64)
    g = np.asarray(dO, dtype=np.float64)
    nq, d = q.shape
    nk = k.shape[0]
    offset = nk - nq
    dv_dim = v.shape[1]
    S = [[0.0] * nk for _ in range(nq)]
    for i in range(nq):
        for j in range(nk):
            if causal and j > i + offset:
                S[i][j] = -math.inf
            else:
                acc = 0.0
                for c in range(d):
                    acc += q[i, c] * k[j, c]
                S[i][j] = scale * acc
    P = [[0.0] * nk for _ in range(nq)]
    L = [0.0] * nq
    for i in range(nq):
        m = max(S[i])
        if m == -math.inf:  # no visible key: empty softmax
            L[i] = math.inf
            continue
        ell = 0.0
        for j in range(nk):
            ell += math.exp(S[i][j] - m) if S[i][j] != -math.inf else 0.0
        L[i] = m + math.log(ell)
        for j in range(nk):
            P[i][j] = math.exp(S[i][j] - L[i]) if S[i][j] != -math.inf else 0.0
    O = np.zeros((nq, dv_dim))
    for i in range(nq):
        for c in range(dv_dim):
            acc = 0.0
            for j in range(nk):
                acc += P[i][j] * v[j, c]
            O[i, c] = acc
    dV = np.zeros((nk, dv_dim))
    for j in range(nk):
        for c in range(dv_dim):
            acc = 0.0
            for i in range(nq):
                acc += P[i][j] * g[i, c]
            dV[j, c] = acc
    dP = [[0.0] * nk for _ in range(nq)]
    for i in range(nq):
        for j in range(nk):
            acc = 0.0
            for c in range(dv_dim):
                acc += g[i, c] * v[j, c]
            dP[i][j] = acc
    D = [0.0] * nq
    for i in range(nq):
        acc = 0.0
        for j in range(nk):
            acc += P[i][j] * dP[i][j]
        D[i] = acc
    dS = [[P[i][j] * (dP[i][j] - D[i]) for j in range(nk)] for i in range(nq)]
    dQ = np.zeros((nq, d))
    dK = np.zeros((nk, d))
    for i in range(nq):
        for c in range(d):
            acc = 0.0
            for j in range(nk):
                acc += dS[i][j] * k[j, c]
            dQ[i, c] = scale * acc
    for j in range(nk):
        for c in range(d):
            acc = 0.0
            for i in range(nq):
                acc += dS[i][j] * q[i, c]
            dK[j, c] = scale * acc
    D_from_O = np.array([sum(g[i, c] * O[i, c] for c in range(dv_dim)) for i in range(nq)])
    return AttentionGrads(O=O[None, None], L=np.array(L)[None, None], D=np.array(D)[None, None],
                          D_from_O=D_from_O[None, None], dQ=dQ[None, None], dK=dK[None, None],
                          dV=dV[None, None])


def attention_loss(Q, K, V, G, scale: float, causal: bool = False) -> float:
    """The scalar loss sum(O * G) whose gradient with respect to O is G
    (CS349E lecture 11 demo 1 uses it for its gradient check)."""
    O, _ = attention_forward(Q, K, V, scale, causal)
    return float(np.sum(O * _as4d(G)))


def causal_executed_tile_pairs(N: int, Br: int, Bc: int, N_k: int | None = None, causal: bool = True) -> int:
    """Number of (key block, query block) pairs that hold at least one visible
    entry, counted by brute force over the blocks: query blocks of Br rows,
    key blocks of Bc rows.  Under the causal mask key j is visible to query i
    iff j <= i + (N_k - N) (N_k defaults to N, the pages' case); a pair is
    live iff its first key is visible to its last query.  Without the mask
    every pair is live.  CS349E lecture 11 demo 4 gives T(T+1)/2 for square
    blocks and N_k = N."""
    Nk = N if N_k is None else N_k
    offset = Nk - N
    tq = -(-N // Br)
    tk = -(-Nk // Bc)
    count = 0
    for kb in range(tk):
        j0 = kb * Bc
        for qb in range(tq):
            i1 = min(N, (qb + 1) * Br) - 1
            if not causal or j0 <= i1 + offset:
                count += 1
    return count
