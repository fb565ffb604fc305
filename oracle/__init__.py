"""fp64 CPU oracle of the chunked Gated-DeltaNet layer.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline may import this package; the library and its Python binding never do.
It shares no code with the CUDA path.

Contents
  gdn_oracle.c   conv + L2 norm + the token-by-token gated delta rule in fp64 (C),
                 and the raw-gate variant's g and beta from projections
  chunked.py     the chunked (WY / UT) form in fp64 numpy, used only to check
                 the algebraic identity with the recurrence
  brute.py       exact rational brute force of the recurrence for tiny inputs
  build.py       compiles gdn_oracle.c with gcc

Every entry point takes float64 arrays holding the exact values of the rounded
inputs. Parity is pinned by tests/test_oracle.py (closed forms, brute force,
chunked identity, conv impulse, norm, GQA duplication); no function here is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from .build import build_oracle, library_path

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            build_oracle()
        lib = ctypes.CDLL(path)
        d = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_conv.argtypes = [i64, i64, d, i64, d, d, ctypes.c_int, d, d]
        lib.oracle_conv.restype = None
        lib.oracle_l2norm.argtypes = [i64, i64, i64, d, ctypes.c_double, ctypes.c_double, d]
        lib.oracle_l2norm.restype = None
        ci = ctypes.c_int
        lib.oracle_recurrence.argtypes = [i64, ci, ci, ci, ci, d, d, d, d, d, d, d]
        lib.oracle_recurrence.restype = None
        lib.oracle_layer.argtypes = [i64, ci, ci, ci, ci, ci, ctypes.c_double, ctypes.c_double,
                                     d, d, d, d, d, d, d, d, d]
        lib.oracle_layer.restype = ctypes.c_int
        lib.oracle_gates.argtypes = [i64, ci, d, d, d, d, d, d]
        lib.oracle_gates.restype = None
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _c(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def conv(x: np.ndarray, w: np.ndarray, state: Optional[np.ndarray] = None, act: int = 0):
    """Causal conv, kernel 4. x: [T, nc]; w: [nc, 4]; state: [3, nc]. Returns (y, new_state)."""
    x, w = _c(x), _c(w)
    T, nc = x.shape
    state = np.zeros((3, nc)) if state is None else _c(state)
    y = np.zeros((T, nc))
    so = np.zeros((3, nc))
    _load().oracle_conv(T, nc, _p(x), nc, _p(w), _p(state), act, _p(y), _p(so))
    return y, so


def l2norm(y: np.ndarray, H: int, d: int, scale: float = 1.0, eps: float = 1e-6) -> np.ndarray:
    y = _c(y)
    T = y.shape[0]
    out = np.zeros_like(y)
    _load().oracle_l2norm(T, H, d, _p(y), scale, eps, _p(out))
    return out


def recurrence(q, k, v, alpha, beta, Hk: int, Hv: int, ST0: Optional[np.ndarray] = None):
    """Gated delta rule with decay factors given directly.

    q, k: [T, Hk*dk] (already normalised); v: [T, Hv*dv]; alpha, beta: [T, Hv];
    ST0: [Hv, dk, dv]. Returns (o [T, Hv, dv], ST [Hv, dk, dv])."""
    q, k, v, alpha, beta = map(_c, (q, k, v, alpha, beta))
    T = q.shape[0]
    dk = q.shape[1] // Hk
    dv = v.shape[1] // Hv
    ST = np.zeros((Hv, dk, dv)) if ST0 is None else _c(ST0).copy()
    o = np.zeros((T, Hv, dv))
    _load().oracle_recurrence(T, Hk, Hv, dk, dv, _p(q), _p(k), _p(v), _p(alpha), _p(beta),
                              _p(ST), _p(o))
    return o, ST


def layer(xq, xk, xv, g, beta, conv_w, Hk: int, Hv: int, conv_state=None, ST0=None,
          act: int = 0, q_scale: float = 1.0, eps: float = 1e-6):
    """The whole layer over one run of tokens.

    Returns (o [T, Hv, dv], ST [Hv, dk, dv], conv_state [3, ch])."""
    xq, xk, xv, g, beta, conv_w = map(_c, (xq, xk, xv, g, beta, conv_w))
    T = xq.shape[0]
    dk = xq.shape[1] // Hk
    dv = xv.shape[1] // Hv
    ch = 2 * Hk * dk + Hv * dv
    assert conv_w.shape == (ch, 4)
    cs = np.zeros((3, ch)) if conv_state is None else _c(conv_state).copy()
    ST = np.zeros((Hv, dk, dv)) if ST0 is None else _c(ST0).copy()
    o = np.zeros((T, Hv, dv))
    rc = _load().oracle_layer(T, Hk, Hv, dk, dv, act, q_scale, eps, _p(xq), _p(xk), _p(xv),
                              _p(g), _p(beta), _p(conv_w), _p(cs), _p(ST), _p(o))
    if rc != 0:
        raise RuntimeError(f"oracle_layer failed ({rc})")
    return o, ST, cs


def gates(a, b, A_log, dt_bias):
    """g and beta from raw projections (the raw-gate variant, a reading outside the pages: the usual
    Gated-DeltaNet parametrisation g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)).

    a, b: [T, Hv]; A_log, dt_bias: [Hv]. Returns (g, beta), each [T, Hv]."""
    a, b, A_log, dt_bias = map(_c, (a, b, A_log, dt_bias))
    T, Hv = a.shape
    g = np.zeros((T, Hv))
    beta = np.zeros((T, Hv))
    _load().oracle_gates(T, Hv, _p(a), _p(b), _p(A_log), _p(dt_bias), _p(g), _p(beta))
    return g, beta


def head_columns(Hk: int, Hv: int, dk: int, dv: int, v_heads: Sequence[int]):
    """Column indices (into xq/xk, xv and conv channels) that the given v-heads read.

    Heads are independent, so the oracle can be run on a subset of heads: the
    conv is per channel and each v-head reads only its own q/k head."""
    G = Hv // Hk
    k_heads = sorted({h // G for h in v_heads})
    qk_cols = np.concatenate([np.arange(h * dk, (h + 1) * dk) for h in k_heads])
    v_cols = np.concatenate([np.arange(h * dv, (h + 1) * dv) for h in v_heads])
    return k_heads, qk_cols, v_cols
