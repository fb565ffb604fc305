"""Python binding of libgdn.so (the C ABI in include/gdn.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. PyTorch provides device memory and streams. Functions carry the C
names. Loading fails loudly when the library is missing: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_SHAPE = 2
GDN_ERR_OFF_GRID = 3
GDN_ERR_STATE_MISMATCH = 4
GDN_ERR_WORKSPACE = 5
GDN_ERR_CUDA = 6
GDN_ERR_TIMEOUT = 7
GDN_ERR_NOT_FOUND = 8
GDN_ERR_IO = 9
GDN_FP32 = 0
GDN_BF16 = 1
GDN_CONV_NONE = 0
GDN_CONV_SILU = 1
GDN_ALLOW_PARTIAL = 1
GDN_MAX_SESSIONS = 4096

EXPORTED = ["gdn_desc_tag", "gdn_desc_check", "gdn_state_bytes", "gdn_conv_state_bytes", "gdn_session_init",
            "gdn_workspace_size", "gdn_prefill_chunks", "gdn_prefill_varlen", "gdn_state_capture",
            "gdn_state_restore", "gdn_conv_state", "gdn_decode_step", "gdn_timing_begin", "gdn_timing_end",
            "gdn_prefill_chunks_noalloc", "gdn_device_status", "gdn_debug_inject_wait_timeout", "gdn_gates",
            "gdn_last_error", "gdn_status_string", "gdn_state_blob_bytes", "gdn_state_serialize",
            "gdn_state_deserialize", "gdn_state_save", "gdn_state_load", "gdn_prefill_branches",
            "gdn_prefill_chunks_checkpoint", "gdn_prefill_varlen_checkpoint"]


class gdn_layer_desc(ctypes.Structure):
    _fields_ = [("n_qk_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("grid_c", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("conv_act", ctypes.c_int32), ("q_scale", ctypes.c_float),
                ("l2_eps", ctypes.c_float)]


class gdn_session(ctypes.Structure):
    _fields_ = [("S", ctypes.c_void_p), ("conv", ctypes.c_void_p), ("committed", ctypes.c_int64),
                ("tag", ctypes.c_uint64)]


class gdn_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64), ("timed", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


class GdnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_status_name(status)}: {msg}")
        self.status = status


_lib = None


def load_library(path: Optional[str] = None):
    """Load libgdn.so (raises if it is missing or lacks a symbol)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libgdn.so not built at {p}: run __graft_entry__.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(p)
    vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    D = ctypes.POINTER(gdn_layer_desc)
    Sp = ctypes.POINTER(gdn_session)
    I64p = ctypes.POINTER(ctypes.c_int64)
    sig = {
        "gdn_desc_tag": (ctypes.c_uint64, [D]),
        "gdn_desc_check": (ctypes.c_int, [D]),
        "gdn_state_bytes": (ctypes.c_size_t, [D]),
        "gdn_conv_state_bytes": (ctypes.c_size_t, [D]),
        "gdn_session_init": (ctypes.c_int, [D, Sp, vp, vp, vp]),
        "gdn_workspace_size": (ctypes.c_size_t, [D, i64, i32]),
        "gdn_prefill_chunks": (ctypes.c_int, [D, Sp, vp, vp, vp, vp, vp, vp, i64, u32, vp, I64p, vp,
                                              ctypes.c_size_t, vp]),
        "gdn_prefill_varlen": (ctypes.c_int, [D, Sp, i32, I64p, vp, vp, vp, vp, vp, vp, u32, vp, I64p, vp,
                                              ctypes.c_size_t, vp]),
        "gdn_prefill_chunks_noalloc": (ctypes.c_int, [D, Sp, vp, vp, vp, vp, vp, vp, i64, u32, vp, I64p, vp]),
        "gdn_prefill_branches": (ctypes.c_int, [D, Sp, Sp, i32, I64p, vp, vp, vp, vp, vp, vp, u32, vp, I64p, vp,
                                                ctypes.c_size_t, vp]),
        "gdn_prefill_chunks_checkpoint": (ctypes.c_int, [D, Sp, Sp, vp, vp, vp, vp, vp, vp, i64, u32, vp, I64p, vp,
                                                         ctypes.c_size_t, vp]),
        "gdn_prefill_varlen_checkpoint": (ctypes.c_int, [D, Sp, Sp, i32, I64p, vp, vp, vp, vp, vp, vp, u32, vp, I64p,
                                                         vp, ctypes.c_size_t, vp]),
        "gdn_state_capture": (ctypes.c_int, [D, Sp, Sp, vp]),
        "gdn_state_restore": (ctypes.c_int, [D, Sp, Sp, vp]),
        "gdn_conv_state": (ctypes.c_int, [D, Sp, vp, vp]),
        "gdn_decode_step": (ctypes.c_int, [D, Sp, i32, vp, vp, vp, vp, vp, vp, vp, vp]),
        "gdn_timing_begin": (ctypes.c_int, [i32]),
        "gdn_timing_end": (ctypes.c_int, [ctypes.POINTER(gdn_kernel_time), i32, ctypes.POINTER(i32)]),
        "gdn_device_status": (ctypes.c_int, [vp]),
        "gdn_debug_inject_wait_timeout": (ctypes.c_int, [i32, i64]),
        "gdn_gates": (ctypes.c_int, [D, vp, vp, vp, vp, i64, vp, vp, vp]),
        "gdn_last_error": (ctypes.c_char_p, []),
        "gdn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "gdn_state_blob_bytes": (ctypes.c_size_t, [D]),
        "gdn_state_serialize": (ctypes.c_int, [D, Sp, vp, ctypes.c_size_t, vp]),
        "gdn_state_deserialize": (ctypes.c_int, [D, vp, ctypes.c_size_t, Sp, vp]),
        "gdn_state_save": (ctypes.c_int, [D, Sp, ctypes.c_char_p, vp]),
        "gdn_state_load": (ctypes.c_int, [D, ctypes.c_char_p, Sp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _status_name(st: int) -> str:
    try:
        return load_library().gdn_status_string(st).decode()
    except Exception:
        return f"status {st}"


def _check(st: int):
    if st != GDN_OK:
        raise GdnError(st, load_library().gdn_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


_TORCH_DT = {GDN_BF16: torch.bfloat16, GDN_FP32: torch.float32}


def make_desc(n_qk_heads: int, n_v_heads: int, d_k: int, d_v: int, grid_c: int, in_dtype: int = GDN_BF16,
              out_dtype: int = GDN_FP32, conv_act: int = GDN_CONV_NONE, q_scale: float = 1.0,
              l2_eps: float = 1e-6) -> gdn_layer_desc:
    return gdn_layer_desc(n_qk_heads, n_v_heads, d_k, d_v, grid_c, in_dtype, out_dtype, conv_act, q_scale, l2_eps)


def channels(desc: gdn_layer_desc) -> int:
    return 2 * desc.n_qk_heads * desc.d_k + desc.n_v_heads * desc.d_v


class Session:
    """A session (or checkpoint slot): device buffers held by PyTorch plus the C struct."""

    def __init__(self, desc: gdn_layer_desc, device=None, stream=None, init: bool = True):
        device = torch.device(device or "cuda")
        self.desc = desc
        self.S = torch.empty((desc.n_v_heads, desc.d_k, desc.d_v), dtype=torch.float32, device=device)
        self.conv = torch.empty((3, channels(desc)), dtype=_TORCH_DT[desc.in_dtype], device=device)
        self.c = gdn_session(self.S.data_ptr(), self.conv.data_ptr(), -1, 0)
        if init:
            gdn_session_init(desc, self, stream)

    @property
    def committed(self) -> int:
        return int(self.c.committed)

    @property
    def tag(self) -> int:
        return int(self.c.tag)


def gdn_desc_tag(desc: gdn_layer_desc) -> int:
    return int(load_library().gdn_desc_tag(ctypes.byref(desc)))


def gdn_desc_check(desc: gdn_layer_desc) -> int:
    return int(load_library().gdn_desc_check(ctypes.byref(desc)))


def gdn_state_bytes(desc: gdn_layer_desc) -> int:
    return int(load_library().gdn_state_bytes(ctypes.byref(desc)))


def gdn_conv_state_bytes(desc: gdn_layer_desc) -> int:
    return int(load_library().gdn_conv_state_bytes(ctypes.byref(desc)))


def gdn_session_init(desc: gdn_layer_desc, sess: Session, stream=None):
    _check(load_library().gdn_session_init(ctypes.byref(desc), ctypes.byref(sess.c), _ptr(sess.S),
                                           _ptr(sess.conv), _stream(stream)))


def gdn_workspace_size(desc: gdn_layer_desc, max_tokens: int, max_sessions: int = 1) -> int:
    return int(load_library().gdn_workspace_size(ctypes.byref(desc), max_tokens, max_sessions))


def workspace(desc: gdn_layer_desc, max_tokens: int, max_sessions: int = 1, device=None) -> torch.Tensor:
    n = gdn_workspace_size(desc, max_tokens, max_sessions)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def gdn_prefill_chunks(desc, sess: Session, xq, xk, xv, g, beta, conv_w, out, ws: torch.Tensor,
                       flags: int = 0, n_tokens: Optional[int] = None, stream=None) -> int:
    """Returns the number of tokens consumed (a multiple of grid_c unless GDN_ALLOW_PARTIAL)."""
    n = int(g.shape[0]) if n_tokens is None else int(n_tokens)
    nc = ctypes.c_int64(0)
    _check(load_library().gdn_prefill_chunks(
        ctypes.byref(desc), ctypes.byref(sess.c), _ptr(xq), _ptr(xk), _ptr(xv), _ptr(g), _ptr(beta),
        _ptr(conv_w), n, flags, _ptr(out), ctypes.byref(nc), _ptr(ws), ws.numel() if ws is not None else 0,
        _stream(stream)))
    return int(nc.value)


GDN_NOALLOC_SCRATCH_BYTES = 32 << 20


def gdn_prefill_chunks_noalloc(desc, sess: Session, xq, xk, xv, g, beta, conv_w, out, flags: int = 0,
                               n_tokens: Optional[int] = None, stream=None) -> int:
    """gdn_prefill_chunks with the library's built-in scratch (no workspace argument, no allocation)."""
    n = int(g.shape[0]) if n_tokens is None else int(n_tokens)
    nc = ctypes.c_int64(0)
    _check(load_library().gdn_prefill_chunks_noalloc(
        ctypes.byref(desc), ctypes.byref(sess.c), _ptr(xq), _ptr(xk), _ptr(xv), _ptr(g), _ptr(beta),
        _ptr(conv_w), n, flags, _ptr(out), ctypes.byref(nc), _stream(stream)))
    return int(nc.value)


def gdn_prefill_varlen(desc, sessions: Sequence[Session], cu_seqlens: Sequence[int], xq, xk, xv, g, beta,
                       conv_w, out, ws: torch.Tensor, flags: int = 0, stream=None) -> List[int]:
    n = len(sessions)
    arr = (gdn_session * n)(*[s.c for s in sessions])
    cu = (ctypes.c_int64 * (n + 1))(*[int(x) for x in cu_seqlens])
    nc = (ctypes.c_int64 * n)()
    st = load_library().gdn_prefill_varlen(
        ctypes.byref(desc), arr, n, cu, _ptr(xq), _ptr(xk), _ptr(xv), _ptr(g), _ptr(beta), _ptr(conv_w),
        flags, _ptr(out), nc, _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream))
    for i, s in enumerate(sessions):   # the library updated the copies in `arr`
        s.c.committed = arr[i].committed
    _check(st)
    return [int(x) for x in nc]


def gdn_prefill_chunks_checkpoint(desc, sess: Session, slot: Session, xq, xk, xv, g, beta, conv_w, out,
                                  ws: torch.Tensor, flags: int = 0, n_tokens: Optional[int] = None, stream=None) -> int:
    """gdn_prefill_chunks, with the result also written into `slot` in the same pass."""
    n_tokens = xq.shape[0] if n_tokens is None else n_tokens
    nc = ctypes.c_int64(0)
    st = load_library().gdn_prefill_chunks_checkpoint(
        ctypes.byref(desc), ctypes.byref(sess.c), ctypes.byref(slot.c), _ptr(xq), _ptr(xk), _ptr(xv), _ptr(g),
        _ptr(beta), _ptr(conv_w), n_tokens, flags, _ptr(out), ctypes.byref(nc), _ptr(ws),
        ws.numel() if ws is not None else 0, _stream(stream))
    _check(st)
    return int(nc.value)


def gdn_prefill_varlen_checkpoint(desc, sessions: Sequence[Session], slots: Sequence[Session],
                                  cu_seqlens: Sequence[int], xq, xk, xv, g, beta, conv_w, out, ws: torch.Tensor,
                                  flags: int = 0, stream=None) -> List[int]:
    n = len(sessions)
    arr = (gdn_session * n)(*[s.c for s in sessions])
    sarr = (gdn_session * n)(*[s.c for s in slots])
    cu = (ctypes.c_int64 * (n + 1))(*[int(x) for x in cu_seqlens])
    nc = (ctypes.c_int64 * n)()
    st = load_library().gdn_prefill_varlen_checkpoint(
        ctypes.byref(desc), arr, sarr, n, cu, _ptr(xq), _ptr(xk), _ptr(xv), _ptr(g), _ptr(beta), _ptr(conv_w),
        flags, _ptr(out), nc, _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream))
    for i in range(n):
        sessions[i].c.committed = arr[i].committed
        slots[i].c.committed, slots[i].c.tag = sarr[i].committed, sarr[i].tag
    _check(st)
    return [int(x) for x in nc]


def gdn_prefill_branches(desc, prefix: Session, branches: Sequence[Session], cu_seqlens: Sequence[int], xq, xk, xv,
                         g, beta, conv_w, out, ws: torch.Tensor, flags: int = 0, stream=None) -> List[int]:
    """Every branch continues `prefix` (read in place, unchanged) with its own packed rows."""
    n = len(branches)
    arr = (gdn_session * n)(*[s.c for s in branches])
    cu = (ctypes.c_int64 * (n + 1))(*[int(x) for x in cu_seqlens])
    nc = (ctypes.c_int64 * n)()
    st = load_library().gdn_prefill_branches(
        ctypes.byref(desc), ctypes.byref(prefix.c), arr, n, cu, _ptr(xq), _ptr(xk), _ptr(xv), _ptr(g), _ptr(beta),
        _ptr(conv_w), flags, _ptr(out), nc, _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream))
    for i, s in enumerate(branches):
        s.c.committed = arr[i].committed
    _check(st)
    return [int(x) for x in nc]


def gdn_state_capture(desc, src: Session, slot: Session, stream=None):
    st = load_library().gdn_state_capture(ctypes.byref(desc), ctypes.byref(src.c), ctypes.byref(slot.c),
                                          _stream(stream))
    _check(st)


def gdn_state_restore(desc, dst: Session, slot: Session, stream=None):
    _check(load_library().gdn_state_restore(ctypes.byref(desc), ctypes.byref(dst.c), ctypes.byref(slot.c),
                                            _stream(stream)))


def gdn_conv_state(desc, sess: Session, out: torch.Tensor, stream=None):
    _check(load_library().gdn_conv_state(ctypes.byref(desc), ctypes.byref(sess.c), _ptr(out), _stream(stream)))


def gdn_decode_step(desc, sessions: Sequence[Session], xq, xk, xv, g, beta, conv_w, out, stream=None):
    n = len(sessions)
    arr = (gdn_session * n)(*[s.c for s in sessions])
    st = load_library().gdn_decode_step(ctypes.byref(desc), arr, n, _ptr(xq), _ptr(xk), _ptr(xv), _ptr(g),
                                        _ptr(beta), _ptr(conv_w), _ptr(out), _stream(stream))
    for i, s in enumerate(sessions):
        s.c.committed = arr[i].committed
    _check(st)


def gdn_gates(desc, a: torch.Tensor, b: torch.Tensor, A_log: torch.Tensor, dt_bias: torch.Tensor,
              g: torch.Tensor, beta: torch.Tensor, stream=None):
    """g, beta [n][Hv] from raw projections a, b [n][Hv] and per-head A_log, dt_bias [Hv] (fp32, on the GPU)."""
    n = a.shape[0]
    for t in (a, b, g, beta):
        if t.dtype != torch.float32 or tuple(t.shape) != (n, desc.n_v_heads):
            raise ValueError("a, b, g, beta must be fp32 [n_tokens][n_v_heads]")
    for t in (A_log, dt_bias):
        if t.dtype != torch.float32 or t.numel() != desc.n_v_heads:
            raise ValueError("A_log, dt_bias must be fp32 [n_v_heads]")
    _check(load_library().gdn_gates(ctypes.byref(desc), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), n, _ptr(g),
                                    _ptr(beta), _stream(stream)))


def gdn_state_blob_bytes(desc) -> int:
    return int(load_library().gdn_state_blob_bytes(ctypes.byref(desc)))


def gdn_state_serialize(desc, session: Session, blob: torch.Tensor, stream=None):
    """Serialise into `blob` (a uint8 host tensor, pinned for an asynchronous copy)."""
    _check(load_library().gdn_state_serialize(ctypes.byref(desc), ctypes.byref(session.c), _ptr(blob),
                                              blob.numel() * blob.element_size(), _stream(stream)))


def gdn_state_deserialize(desc, blob: torch.Tensor, dst: Session, stream=None):
    lib = load_library()
    st = lib.gdn_state_deserialize(ctypes.byref(desc), _ptr(blob), blob.numel() * blob.element_size(),
                                   ctypes.byref(dst.c), _stream(stream))
    _check(st)


def gdn_state_save(desc, session: Session, path: str, stream=None):
    _check(load_library().gdn_state_save(ctypes.byref(desc), ctypes.byref(session.c), os.fsencode(path),
                                         _stream(stream)))


def gdn_state_load(desc, path: str, dst: Session, stream=None):
    _check(load_library().gdn_state_load(ctypes.byref(desc), os.fsencode(path), ctypes.byref(dst.c),
                                         _stream(stream)))


def gdn_timing_begin(max_launches: int):
    _check(load_library().gdn_timing_begin(max_launches))


def gdn_timing_end() -> dict:
    """{kind: (launches, timed launches, total device ms)} since gdn_timing_begin."""
    arr = (gdn_kernel_time * 8)()
    n = ctypes.c_int32(0)
    _check(load_library().gdn_timing_end(arr, 8, ctypes.byref(n)))
    return {arr[i].name.decode(): (int(arr[i].launches), int(arr[i].timed), float(arr[i].total_ms))
            for i in range(min(n.value, 8))}


def gdn_device_status(stream=None) -> int:
    """GDN_OK, or GDN_ERR_TIMEOUT if a kernel gave up a bounded wait since the last check (synchronises)."""
    return int(load_library().gdn_device_status(_stream(stream)))


def gdn_debug_inject_wait_timeout(enable: int, wait_limit: int = 1000):
    """enable: 0 off, 1 the state kernel, 2 the tcgen05 prologue skips its first copy."""
    _check(load_library().gdn_debug_inject_wait_timeout(int(enable), wait_limit))
