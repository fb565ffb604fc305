"""Shared helpers of the GPU tests: run the library on workload tokens and the
fp64 oracle on the same values, and compare them by the tolerance metric
(relative L2 per session and v-head, max over heads)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from chunked_gated_deltanet_gb300 import gdn
from chunked_gated_deltanet_gb300 import workloads as wl

# tolerances: outputs / final state, by input dtype
TOL = {wl.BF16: (2e-3, 1e-3), wl.FP32: (1e-5, 1e-5)}


def desc_of(shape: wl.Shape, out_dtype=gdn.GDN_FP32, act=gdn.GDN_CONV_NONE, q_scale=1.0):
    return gdn.make_desc(shape.n_qk_heads, shape.n_v_heads, shape.d_k, shape.d_v, shape.grid_c,
                         gdn.GDN_BF16 if shape.dtype == wl.BF16 else gdn.GDN_FP32, out_dtype, act, q_scale)


def rel_l2_max(x: np.ndarray, ref: np.ndarray) -> float:
    """x, ref: [..., H, d] or [H, dk, dv]; relative L2 per head (axis chosen by caller layout)."""
    worst = 0.0
    for h in range(ref.shape[0]):
        nr = np.linalg.norm(ref[h])
        err = np.linalg.norm(x[h] - ref[h])
        worst = max(worst, err / nr if nr > 0 else (0.0 if err <= 1e-6 else np.inf))
    return worst


def out_rel(o_gpu: np.ndarray, o_ref: np.ndarray) -> float:
    """outputs [T, H, d]: heads to the front."""
    return rel_l2_max(np.moveaxis(o_gpu, 1, 0), np.moveaxis(o_ref, 1, 0))


class Runner:
    """Device-side copies of one session's tokens and the layer weights."""

    def __init__(self, shape: wl.Shape, tok: wl.Tokens, cw: np.ndarray, device, out_dtype=gdn.GDN_FP32,
                 act=gdn.GDN_CONV_NONE, q_scale=1.0):
        self.shape, self.tok, self.cw, self.dev = shape, tok, cw, device
        self.desc = desc_of(shape, out_dtype, act, q_scale)
        self.x = wl.tokens_to_torch(tok, shape.dtype, device)
        self.cw_t = wl.to_torch(cw, shape.dtype, device)
        self.out_dt = torch.float32 if out_dtype == gdn.GDN_FP32 else torch.bfloat16
        self.ws = gdn.workspace(self.desc, len(tok) + 64, 1, device)

    def new_out(self, T=None):
        T = len(self.tok) if T is None else T
        return torch.full((T, self.shape.n_v_heads, self.shape.d_v), float("nan"), dtype=self.out_dt,
                          device=self.dev)

    def session(self):
        return gdn.Session(self.desc, self.dev)

    def prefill(self, sess, a: int, b: int, out: torch.Tensor, flags: int = 0) -> int:
        """Feed rows [a, b); outputs land in out[a:b] (rows of consumed tokens)."""
        xq, xk, xv, g, beta = (t[a:b] for t in self.x)
        return gdn.gdn_prefill_chunks(self.desc, sess, xq, xk, xv, g, beta, self.cw_t, out[a:b], self.ws,
                                      flags=flags)


def oracle_run(shape: wl.Shape, tok: wl.Tokens, cw: np.ndarray, v_heads=None, conv_state=None, ST0=None,
               act=0, q_scale=1.0):
    """fp64 oracle over `tok` for the given v-heads (whole layer if None).

    Returns (o [T, len(v_heads), dv], ST [len(v_heads), dk, dv], conv_state of the selected channels)."""
    Hk, Hv, dk, dv = shape.n_qk_heads, shape.n_v_heads, shape.d_k, shape.d_v
    f = lambda a: wl.as_f64(a, shape.dtype)
    if v_heads is None:
        return oracle.layer(f(tok.xq), f(tok.xk), f(tok.xv), tok.g.astype(np.float64),
                            tok.beta.astype(np.float64), f(cw), Hk, Hv, conv_state=conv_state, ST0=ST0,
                            act=act, q_scale=q_scale)
    v_heads = list(v_heads)
    k_heads, qk_cols, v_cols = oracle.head_columns(Hk, Hv, dk, dv, v_heads)
    nq = Hk * dk
    chan = np.concatenate([qk_cols, nq + qk_cols, 2 * nq + v_cols])
    cs = None if conv_state is None else np.asarray(conv_state)[:, chan]
    st0 = None if ST0 is None else np.asarray(ST0)[v_heads]
    return oracle.layer(f(tok.xq[:, qk_cols]), f(tok.xk[:, qk_cols]), f(tok.xv[:, v_cols]),
                        tok.g[:, v_heads].astype(np.float64), tok.beta[:, v_heads].astype(np.float64),
                        f(cw[chan]), len(k_heads), len(v_heads), conv_state=cs, ST0=st0, act=act,
                        q_scale=q_scale)


def conv_as_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().double().cpu().numpy()
