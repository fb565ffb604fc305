"""Exact rational brute force of the gated delta rule for tiny inputs.

TEST INFRASTRUCTURE ONLY. It evaluates the update exactly as the method states
it, S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T and o_t = S_t q_t,
with explicit matrix products over fractions.Fraction, in the untransposed
orientation (S is d_v x d_k). The decay factor a_t = exp(g_t) is given directly
as a rational, so no transcendental function enters. Keys are whatever the
caller passes (for exactness, rational unit vectors such as axis vectors or
Pythagorean triples).
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Sequence

Mat = List[List[Fraction]]


def _matmul(A: Mat, B: Mat) -> Mat:
    n, m, p = len(A), len(B), len(B[0])
    return [[sum((A[i][r] * B[r][j] for r in range(m)), Fraction(0)) for j in range(p)]
            for i in range(n)]


def brute_recurrence(q: Sequence[Sequence[Fraction]], k: Sequence[Sequence[Fraction]],
                     v: Sequence[Sequence[Fraction]], a: Sequence[Fraction],
                     b: Sequence[Fraction], S0: Mat):
    """One head. q, k: T x dk; v: T x dv; a, b: T; S0: dv x dk.

    Returns (outputs T x dv, final S as dv x dk), all Fractions."""
    dk, dv = len(k[0]), len(v[0])
    S = [list(row) for row in S0]
    outs = []
    for t in range(len(a)):
        kt = [Fraction(x) for x in k[t]]
        # H = I - b k k^T   (dk x dk)
        H = [[(Fraction(1) if i == j else Fraction(0)) - b[t] * kt[i] * kt[j] for j in range(dk)]
             for i in range(dk)]
        SH = _matmul(S, H)
        S = [[a[t] * SH[i][j] + b[t] * Fraction(v[t][i]) * kt[j] for j in range(dk)]
             for i in range(dv)]
        outs.append([sum((S[i][j] * Fraction(q[t][j]) for j in range(dk)), Fraction(0))
                     for i in range(dv)])
    return outs, S
