"""Chunked (WY / UT) form of the gated delta rule, fp64, one head.

TEST INFRASTRUCTURE ONLY. Used by the oracle self-tests to check that the
blockwise algebra equals the token-by-token recurrence; the parity tests never
use it as a reference for the GPU.

Derivation (from the recurrence S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T).
Within a block of n tokens starting from state S0, let G_t = prod_{j<=t} a_j
(gamma_t = log G_t = cumulative sum of g). Writing
u_t = b_t (v_t - a_t S_{t-1} k_t), the state is S_t = G_t S0 + sum_{j<=t} (G_t/G_j) u_j k_j^T.
Substituting into u_t gives a unit lower-triangular system
    (I + A) U_raw = diag(b) V - diag(b G) K S0^T,
    A_ij = b_i (G_i / G_j) k_i . k_j   for j < i, else 0.
With Tm = (I + A)^-1:   U = Tm diag(b) V,   W = Tm diag(b G) K,   U' = U - W S0^T,
    O = diag(G) Q S0^T + ((Q K^T) o M) U',   M_ij = G_i/G_j for j <= i, else 0,
    S_n^T = G_n S0^T + K^T diag(G_n/G_j) U'.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def chunked_head(q, k, v, g, beta, ST0, n: int):
    """q, k: [T, dk]; v: [T, dv]; g, beta: [T]; ST0: [dk, dv]; block length n.

    Returns (o [T, dv], ST [dk, dv])."""
    q, k, v, g, beta = (np.asarray(a, dtype=np.float64) for a in (q, k, v, g, beta))
    T = q.shape[0]
    ST = np.array(ST0, dtype=np.float64, copy=True)
    o = np.zeros((T, v.shape[1]))
    for s in range(0, T, n):
        e = min(T, s + n)
        L = e - s
        Q, K, V, gb, bb = q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e]
        gam = np.cumsum(gb)
        lower = np.tril(np.ones((L, L), dtype=bool))
        diff = np.where(lower, gam[:, None] - gam[None, :], 0.0)   # <= 0 on and below the diagonal
        M = np.where(lower, np.exp(diff), 0.0)
        A = np.tril(bb[:, None] * (K @ K.T) * M, -1)
        I_A = np.eye(L) + A
        U = solve_triangular(I_A, bb[:, None] * V, lower=True, unit_diagonal=True)
        W = solve_triangular(I_A, (bb * np.exp(gam))[:, None] * K, lower=True, unit_diagonal=True)
        Up = U - W @ ST
        o[s:e] = np.exp(gam)[:, None] * (Q @ ST) + ((Q @ K.T) * M) @ Up
        ST = np.exp(gam[-1]) * ST + K.T @ (np.exp(gam[-1] - gam)[:, None] * Up)
    return o, ST
