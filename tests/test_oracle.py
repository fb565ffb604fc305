"""Pins of the fp64 oracle to facts outside itself (no GPU).

Each test fixes part of the oracle against mathematics it must reproduce: closed
forms of the gated delta rule, an exact rational brute force of the update as
the method states it, the chunked (WY/UT) identity, the conv's impulse
response, the L2 norm's closed form and the GQA head map. A plausible slip in
the oracle (a dropped decay factor, a sign, a transposed state, the wrong tap
order or head map) fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit

import oracle
from oracle.brute import brute_recurrence
from oracle.chunked import chunked_head


def _rng(s):
    return np.random.default_rng(s)


def _unit_rows(rng, T, H, d):
    x = rng.standard_normal((T, H, d))
    return (x / np.linalg.norm(x, axis=-1, keepdims=True)).reshape(T, H * d)


# --------------------------------------------------------------------------
# exact rational brute force (update as stated, untransposed state)
# --------------------------------------------------------------------------

def _dyadic(rng, shape, denom=64, lo=-64, hi=64):
    """Random dyadic rationals: exact in fp64 and in Fraction."""
    return rng.integers(lo, hi + 1, size=shape) / denom


@pytest.mark.parametrize("T,dk,dv,Hk,Hv", [(12, 3, 2, 1, 1), (16, 4, 3, 1, 2), (9, 2, 5, 2, 2)])
def test_brute_force_rational(T, dk, dv, Hk, Hv):
    rng = _rng(T * 100 + dk)
    q = _dyadic(rng, (T, Hk * dk))
    k = _dyadic(rng, (T, Hk * dk))
    v = _dyadic(rng, (T, Hv * dv))
    a = rng.integers(1, 17, size=(T, Hv)) / 16.0          # decay in (0, 1]
    b = rng.integers(0, 17, size=(T, Hv)) / 16.0          # beta in [0, 1]
    ST0 = _dyadic(rng, (Hv, dk, dv))
    o, ST = oracle.recurrence(q, k, v, a, b, Hk, Hv, ST0)
    G = Hv // Hk
    for h in range(Hv):
        hk = h // G
        F = lambda arr: [[Fraction(float(x)) for x in row] for row in arr]
        S0 = [[Fraction(float(ST0[h, j, i])) for j in range(dk)] for i in range(dv)]  # dv x dk
        outs, S = brute_recurrence(F(q[:, hk * dk:(hk + 1) * dk]), F(k[:, hk * dk:(hk + 1) * dk]),
                                   F(v[:, h * dv:(h + 1) * dv]),
                                   [Fraction(float(x)) for x in a[:, h]],
                                   [Fraction(float(x)) for x in b[:, h]], S0)
        S_exact = np.array([[float(S[i][j]) for j in range(dk)] for i in range(dv)])
        o_exact = np.array([[float(x) for x in row] for row in outs])
        scale = max(1.0, np.abs(S_exact).max())
        assert np.abs(ST[h].T - S_exact).max() <= 1e-13 * scale
        oscale = max(1.0, np.abs(o_exact).max())
        assert np.abs(o[:, h, :] - o_exact).max() <= 1e-13 * oscale


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def test_beta_zero_pure_decay():
    """beta = 0: S_t = exp(sum g) S_0 and o_t = exp(sum_{<=t} g) S_0 q_t."""
    rng = _rng(1)
    T, Hk, Hv, dk, dv = 40, 1, 2, 6, 5
    q = _unit_rows(rng, T, Hk, dk)
    k = _unit_rows(rng, T, Hk, dk)
    v = rng.standard_normal((T, Hv * dv))
    g = -rng.random((T, Hv)) * 0.3
    ST0 = rng.standard_normal((Hv, dk, dv))
    o, ST = oracle.recurrence(q, k, v, np.exp(g), np.zeros((T, Hv)), Hk, Hv, ST0)
    for h in range(Hv):
        decay = np.exp(np.cumsum(g[:, h]))
        np.testing.assert_allclose(ST[h], decay[-1] * ST0[h], rtol=1e-13)
        expect = decay[:, None] * (q[:, :dk] @ ST0[h])
        np.testing.assert_allclose(o[:, h, :], expect, rtol=1e-12, atol=1e-14)


def test_beta_zero_through_layer():
    """The whole layer with beta = 0 leaves only the decay of the given state."""
    rng = _rng(2)
    T, Hk, Hv, dk, dv = 33, 2, 4, 8, 4
    ch = 2 * Hk * dk + Hv * dv
    xq = rng.standard_normal((T, Hk * dk))
    xk = rng.standard_normal((T, Hk * dk))
    xv = rng.standard_normal((T, Hv * dv))
    g = -rng.random((T, Hv)) * 0.2
    w = rng.standard_normal((ch, 4)) * 0.5
    ST0 = rng.standard_normal((Hv, dk, dv))
    _, ST, _ = oracle.layer(xq, xk, xv, g, np.zeros((T, Hv)), w, Hk, Hv, ST0=ST0)
    np.testing.assert_allclose(ST, np.exp(g.sum(0))[:, None, None] * ST0, rtol=1e-13)


def test_orthonormal_keys_store_and_recall():
    """g = 0, beta = 1, orthonormal keys, S_0 = 0: S = sum v_j k_j^T and S k_j = v_j."""
    rng = _rng(3)
    dk, dv, n = 8, 5, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :n].T                       # n orthonormal rows
    vals = rng.standard_normal((n, dv))
    q = np.concatenate([keys, keys])         # second pass: query each key with beta = 0
    k = np.concatenate([keys, keys])
    v = np.concatenate([vals, np.zeros((n, dv))])
    beta = np.concatenate([np.ones(n), np.zeros(n)])[:, None]
    o, ST = oracle.recurrence(q, k, v, np.ones((2 * n, 1)), beta, 1, 1)
    np.testing.assert_allclose(ST[0], keys.T @ vals, atol=1e-13)
    np.testing.assert_allclose(o[n:, 0, :], vals, atol=1e-13)


def test_delta_rule_overwrites_a_key():
    """Writing key k again with v' (beta = 1, g = 0) makes S k = v'."""
    rng = _rng(4)
    dk, dv = 6, 3
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k1, k2 = Qm[:, 0], Qm[:, 1]
    v1, v2, v1b = rng.standard_normal((3, dv))
    k = np.stack([k1, k2, k1, k1])
    v = np.stack([v1, v2, v1b, np.zeros(dv)])
    beta = np.array([[1.0], [1.0], [1.0], [0.0]])
    o, _ = oracle.recurrence(k, k, v, np.ones((4, 1)), beta, 1, 1)
    np.testing.assert_allclose(o[3, 0], v1b, atol=1e-13)
    # the other key is untouched by the overwrite
    o2, _ = oracle.recurrence(np.stack([k1, k2, k1, k2]), k, v, np.ones((4, 1)), beta, 1, 1)
    np.testing.assert_allclose(o2[3, 0], v2, atol=1e-13)


def test_state_norm_bound_each_step():
    """|S_t|_F <= a_t |S_{t-1}|_F + b_t |v_t| for unit keys and beta in [0, 1]."""
    rng = _rng(5)
    T, dk, dv = 60, 7, 4
    k = _unit_rows(rng, T, 1, dk)
    q = _unit_rows(rng, T, 1, dk)
    v = rng.standard_normal((T, dv)) * 3
    a = np.exp(-rng.random((T, 1)) * 0.1)
    b = rng.random((T, 1))
    ST = rng.standard_normal((1, dk, dv))
    for t in range(T):
        prev = np.linalg.norm(ST)
        _, ST = oracle.recurrence(q[t:t + 1], k[t:t + 1], v[t:t + 1], a[t:t + 1], b[t:t + 1], 1, 1, ST)
        assert np.linalg.norm(ST) <= a[t, 0] * prev + b[t, 0] * np.linalg.norm(v[t]) + 1e-12


def test_householder_special_case():
    """beta = 2, g = 0, v = 0 makes each step a Householder reflection: S_T = S_0 H_1 ... H_T."""
    rng = _rng(6)
    T, dk, dv = 7, 5, 3
    k = _unit_rows(rng, T, 1, dk)
    S0 = rng.standard_normal((dv, dk))
    _, ST = oracle.recurrence(k, k, np.zeros((T, dv)), np.ones((T, 1)), 2 * np.ones((T, 1)), 1, 1,
                              S0.T[None])
    P = np.eye(dk)
    for t in range(T):
        P = P @ (np.eye(dk) - 2 * np.outer(k[t], k[t]))
    np.testing.assert_allclose(ST[0].T, S0 @ P, atol=1e-13)
    # a reflection keeps the Frobenius norm
    assert abs(np.linalg.norm(ST) - np.linalg.norm(S0)) < 1e-12


# --------------------------------------------------------------------------
# chunked (WY/UT) form == recurrence
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 7, 16, 64, 512])
def test_chunked_equals_recurrent(n):
    rng = _rng(7)
    T, dk, dv = 700, 16, 12
    q = _unit_rows(rng, T, 1, dk)
    k = _unit_rows(rng, T, 1, dk)
    v = rng.standard_normal((T, dv))
    g = -np.logaddexp(0, rng.standard_normal(T)) * 0.1
    beta = expit(rng.standard_normal(T))
    ST0 = rng.standard_normal((dk, dv)) * 0.1
    o_r, ST_r = oracle.recurrence(q, k, v, np.exp(g)[:, None], beta[:, None], 1, 1, ST0[None])
    o_c, ST_c = chunked_head(q, k, v, g, beta, ST0, n)
    rel = lambda x, y: np.linalg.norm(x - y) / np.linalg.norm(y)
    assert rel(o_c, o_r[:, 0]) < 1e-12
    assert rel(ST_c, ST_r[0]) < 1e-12


# --------------------------------------------------------------------------
# conv and norm
# --------------------------------------------------------------------------

def test_conv_impulse_gives_taps_in_order():
    """An impulse at position t0 yields y[t0 + i] = w[c, 3 - i]: tap 3 is the current token."""
    rng = _rng(8)
    T, nc, t0 = 12, 3, 4
    w = rng.standard_normal((nc, 4))
    x = np.zeros((T, nc))
    x[t0, 1] = 1.0
    y, _ = oracle.conv(x, w)
    for i in range(4):
        assert y[t0 + i, 1] == w[1, 3 - i]
    mask = np.ones_like(y, dtype=bool)
    mask[t0:t0 + 4, 1] = False
    assert np.all(y[mask] == 0)


def test_conv_zero_weights_and_state_carry():
    rng = _rng(9)
    T, nc = 20, 5
    x = rng.standard_normal((T, nc))
    w = rng.standard_normal((nc, 4))
    y0, _ = oracle.conv(x, np.zeros((nc, 4)))
    assert np.all(y0 == 0)
    y, st = oracle.conv(x, w)
    for cut in range(T + 1):
        ya, sa = oracle.conv(x[:cut], w)
        yb, sb = oracle.conv(x[cut:], w, sa)
        assert np.array_equal(np.concatenate([ya, yb]), y)
        assert np.array_equal(sb, st)
    assert np.array_equal(st, x[-3:])   # the carried state is the last three raw inputs


def test_conv_silu():
    rng = _rng(10)
    x = rng.standard_normal((9, 4))
    w = rng.standard_normal((4, 4))
    z, _ = oracle.conv(x, w, act=0)
    y, _ = oracle.conv(x, w, act=1)
    np.testing.assert_allclose(y, z * expit(z), rtol=1e-14, atol=1e-15)


def test_l2norm_closed_form():
    rng = _rng(11)
    T, H, d, eps, s = 6, 3, 10, 1e-6, 0.7
    y = rng.standard_normal((T, H * d)) * rng.random((T, 1)) * 1e-2
    out = oracle.l2norm(y, H, d, scale=s, eps=eps).reshape(T, H, d)
    yy = y.reshape(T, H, d)
    ny = np.linalg.norm(yy, axis=-1)
    np.testing.assert_allclose(np.linalg.norm(out, axis=-1), s * ny / np.sqrt(ny ** 2 + eps), rtol=1e-13)
    # same direction as y
    cos = (out * yy).sum(-1) / (np.linalg.norm(out, axis=-1) * ny)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-13)


# --------------------------------------------------------------------------
# the composite layer
# --------------------------------------------------------------------------

def _layer_inputs(rng, T, Hk, Hv, dk, dv):
    ch = 2 * Hk * dk + Hv * dv
    return dict(xq=rng.standard_normal((T, Hk * dk)), xk=rng.standard_normal((T, Hk * dk)),
                xv=rng.standard_normal((T, Hv * dv)),
                g=-np.logaddexp(0, rng.standard_normal((T, Hv))) * 0.1,
                beta=expit(rng.standard_normal((T, Hv))), conv_w=rng.standard_normal((ch, 4)) * 0.5)


def test_gqa_equals_duplicated_heads():
    """Hv = 2 Hk with head map h -> h // 2 equals Hk = Hv with q/k heads duplicated (exactly)."""
    rng = _rng(12)
    T, Hk, Hv, d = 40, 2, 4, 6
    a = _layer_inputs(rng, T, Hk, Hv, d, d)
    o, ST, _ = oracle.layer(Hk=Hk, Hv=Hv, **a)
    dup = lambda x: np.concatenate([x[:, (h // 2) * d:(h // 2 + 1) * d] for h in range(Hv)], axis=1)
    w = a["conv_w"]
    wq, wk, wv = w[:Hk * d], w[Hk * d:2 * Hk * d], w[2 * Hk * d:]
    wdup = lambda ww: np.concatenate([ww[(h // 2) * d:(h // 2 + 1) * d] for h in range(Hv)])
    b = dict(a, xq=dup(a["xq"]), xk=dup(a["xk"]), conv_w=np.concatenate([wdup(wq), wdup(wk), wv]))
    o2, ST2, _ = oracle.layer(Hk=Hv, Hv=Hv, **b)
    assert np.array_equal(o, o2) and np.array_equal(ST, ST2)


def test_layer_is_conv_norm_recurrence():
    """The composite routes channels q | k | v and the conv state blocks correctly."""
    rng = _rng(13)
    T, Hk, Hv, dk, dv = 25, 2, 4, 5, 3
    a = _layer_inputs(rng, T, Hk, Hv, dk, dv)
    ch = 2 * Hk * dk + Hv * dv
    cs0 = rng.standard_normal((3, ch))
    o, ST, cs = oracle.layer(Hk=Hk, Hv=Hv, conv_state=cs0, act=1, q_scale=0.5, **a)
    w = a["conv_w"]
    nq = Hk * dk
    yq, sq = oracle.conv(a["xq"], w[:nq], cs0[:, :nq], act=1)
    yk, sk = oracle.conv(a["xk"], w[nq:2 * nq], cs0[:, nq:2 * nq], act=1)
    yv, sv = oracle.conv(a["xv"], w[2 * nq:], cs0[:, 2 * nq:], act=1)
    q = oracle.l2norm(yq, Hk, dk, 0.5)
    k = oracle.l2norm(yk, Hk, dk, 1.0)
    o2, ST2 = oracle.recurrence(q, k, yv, np.exp(a["g"]), a["beta"], Hk, Hv)
    # numpy's exp and libm's exp may differ in the last ulp
    np.testing.assert_allclose(o, o2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(ST, ST2, rtol=1e-13, atol=1e-15)
    assert np.array_equal(cs, np.concatenate([sq, sk, sv], axis=1))


def test_layer_split_invariance():
    """Running [0, a) then [a, T) with the carried state equals one run (exactly, in fp64)."""
    rng = _rng(14)
    T, Hk, Hv, d = 50, 1, 2, 4
    a = _layer_inputs(rng, T, Hk, Hv, d, d)
    o, ST, cs = oracle.layer(Hk=Hk, Hv=Hv, **a)
    for cut in (0, 1, 2, 3, 17, 49, 50):
        p1 = {k_: v_[:cut] if k_ != "conv_w" else v_ for k_, v_ in a.items()}
        p2 = {k_: v_[cut:] if k_ != "conv_w" else v_ for k_, v_ in a.items()}
        oa, STa, csa = oracle.layer(Hk=Hk, Hv=Hv, **p1)
        ob, STb, csb = oracle.layer(Hk=Hk, Hv=Hv, conv_state=csa, ST0=STa, **p2)
        assert np.array_equal(np.concatenate([oa, ob]), o)
        assert np.array_equal(STb, ST) and np.array_equal(csb, cs)


def test_gates_closed_forms():
    """The raw-gate variant's g = -exp(A_log) softplus(a + dt_bias) and beta = sigmoid(b), pinned by values
    known in closed form: softplus(0) = ln 2, softplus(ln(e - 1)) = 1, softplus(x) -> x for large x and
    -> e^x for very negative x; sigmoid(0) = 1/2, sigmoid(+-ln 3) = 3/4, 1/4. Two heads with different
    parameters pin the per-head indexing."""
    L3 = np.log(3.0)
    a = np.array([[0.0 - 0.25, np.log(np.e - 1.0)],     # head 0: x = a + dt_bias = 0
                  [50.0 - 0.25, -50.0],
                  [-0.25, 0.0]])
    b = np.array([[0.0, L3], [-L3, 0.0], [L3, -L3]])
    A_log = np.array([L3, 0.0])                          # exp(A_log) = 3, 1
    dt_bias = np.array([0.25, 0.0])
    g, beta = oracle.gates(a, b, A_log, dt_bias)
    assert g[0, 0] == pytest.approx(-3.0 * np.log(2.0), rel=1e-15)
    assert g[0, 1] == pytest.approx(-1.0, rel=1e-15)
    assert g[1, 0] == pytest.approx(-3.0 * 50.0, rel=1e-15)
    assert g[1, 1] == pytest.approx(-np.exp(-50.0), rel=1e-12)
    assert g[2, 0] == pytest.approx(-3.0 * np.log(2.0), rel=1e-15)
    assert g[2, 1] == pytest.approx(-np.log(2.0), rel=1e-15)
    assert np.all(g < 0)
    assert beta[0, 0] == 0.5 and beta[1, 1] == 0.5
    assert beta[0, 1] == pytest.approx(0.75, rel=1e-15) and beta[2, 0] == pytest.approx(0.75, rel=1e-15)
    assert beta[1, 0] == pytest.approx(0.25, rel=1e-15) and beta[2, 1] == pytest.approx(0.25, rel=1e-15)
