"""Seeded synthetic inputs for the chunked Gated-DeltaNet prefill.

This module is shared by the tests, the benchmark and the oracle's callers. It
holds the workload definitions and the random draws only: none of the layer's
arithmetic (convolution, normalisation, recurrence) lives here.

The pages measure on private conversations of a Qwen3.5 0.8B reader
("The shadow reader", section "Exact on a grid": 41,802 and 58,278 tokens) and
on random-token prompts ("qwen3_5: run prompts that share prefixes once per
prefix", section "Test Plan"). Neither is available, so activations drawn here
stand in for them, with the shapes of those workloads:

* q, k, v activations ~ N(0, 1), rounded to the input dtype (bf16 by
  round-to-nearest-even, or fp32).
* beta = sigmoid(N(0, 1)); log-decay g = -softplus(N(mu, 1)) * scale
  (mu = 0, scale = 0.1 by default; the long-session workload uses mu = -2,
  scale = 1).
* conv weights ~ N(0, 0.5^2), kernel 4, rounded to the input dtype.
* raw-gate inputs (the optional variant that computes g and beta from
  projections): a ~ N(0, 1), b ~ N(0, 1) per token and v-head; per head
  A_log = ln U(0.05, 0.5) and dt_bias ~ N(-2, 0.5), so that the resulting
  log-decays stay moderate (about -0.5 to -0.003), like the drawn g above.

All draws use numpy's PCG64 through independent SeedSequence streams:
stream (seed, 0) for layer weights, (seed, 1 + i) for session i's tokens,
(seed, 10_000 + j) for question/branch j's tokens, and (seed, 99_999) for
lengths and cut points. Rows are drawn in the fixed order x_q, x_k, x_v,
g-noise, beta-noise, so any slice of a session sees the same values however the
session is later split into calls.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

BF16 = "bf16"
FP32 = "fp32"

_ROW_CHUNK = 8192  # rows drawn per numpy call; draws are sequential, so chunking does not change values


# ---------------------------------------------------------------------------
# bf16 helpers (bit patterns held in uint16 arrays)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not np.isfinite(x).all():
        raise ValueError("bf16 rounding of non-finite values is not supported")
    b = x.view(np.uint32)
    # finite values have bits <= 0xFF7FFFFF, so adding at most 0x8000 stays inside uint32
    r = b >> np.uint32(16)
    r &= np.uint32(1)
    r += np.uint32(0x7FFF)
    r += b
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 view of stored input values (bf16 bits or float32)."""
    if dtype == BF16:
        return bf16_bits_to_f32(arr).astype(np.float64)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


def _round(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype != BF16:
        return np.ascontiguousarray(x32, dtype=np.float32)
    try:   # torch's float32 -> bfloat16 cast is round-to-nearest-even too, and vectorised
        import torch
        t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    except ImportError:
        return f32_to_bf16_bits(x32)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _softplus(x):
    return np.logaddexp(0.0, x)


# ---------------------------------------------------------------------------
# Layer shape and a block of tokens
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Shape:
    n_qk_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    grid_c: int
    dtype: str = BF16

    @property
    def channels(self) -> int:
        return 2 * self.n_qk_heads * self.d_k + self.n_v_heads * self.d_v


@dataclasses.dataclass
class Tokens:
    """Per-token layer inputs of one contiguous run of positions.

    xq, xk: [T, Hk*d_k]; xv: [T, Hv*d_v] (uint16 bf16 bits or float32);
    g, beta: [T, Hv] float32.
    """
    xq: np.ndarray
    xk: np.ndarray
    xv: np.ndarray
    g: np.ndarray
    beta: np.ndarray

    def __len__(self) -> int:
        return int(self.g.shape[0])

    def slice(self, a: int, b: int) -> "Tokens":
        return Tokens(self.xq[a:b], self.xk[a:b], self.xv[a:b], self.g[a:b], self.beta[a:b])

    @staticmethod
    def concat(parts: Sequence["Tokens"]) -> "Tokens":
        return Tokens(*(np.concatenate([getattr(p, f) for p in parts], axis=0)
                        for f in ("xq", "xk", "xv", "g", "beta")))


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def draw_conv_weights(shape: Shape, seed: int, std: float = 0.5) -> np.ndarray:
    """conv weights [channels, 4]; tap 3 multiplies the current token."""
    rng = _rng(seed, 0)
    w = (rng.standard_normal((shape.channels, 4)) * std).astype(np.float32)
    return _round(w, shape.dtype)


def _draw_matrix(rng, rows: int, cols: int, dtype: str, prenorm_head: int = 0) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.uint16 if dtype == BF16 else np.float32)
    for a in range(0, rows, _ROW_CHUNK):
        b = min(rows, a + _ROW_CHUNK)
        x = rng.standard_normal((b - a, cols), dtype=np.float32)
        if prenorm_head:
            # input recipe of the small fp32 workload: q and k arrive unit-norm per head
            xs = x.reshape(b - a, cols // prenorm_head, prenorm_head).astype(np.float64)
            xs = xs / np.linalg.norm(xs, axis=-1, keepdims=True)
            x = xs.reshape(b - a, cols).astype(np.float32)
        out[a:b] = _round(x, dtype)
    return out


def draw_tokens(shape: Shape, T: int, seed: int, stream: int, g_mu: float = 0.0,
                g_scale: float = 0.1, prenorm_qk: bool = False) -> Tokens:
    rng = _rng(seed, stream)
    Hk, Hv = shape.n_qk_heads, shape.n_v_heads
    pn = shape.d_k if prenorm_qk else 0
    xq = _draw_matrix(rng, T, Hk * shape.d_k, shape.dtype, pn)
    xk = _draw_matrix(rng, T, Hk * shape.d_k, shape.dtype, pn)
    xv = _draw_matrix(rng, T, Hv * shape.d_v, shape.dtype)
    gn = rng.standard_normal((T, Hv)) + g_mu
    bn = rng.standard_normal((T, Hv))
    g = (-_softplus(gn) * g_scale).astype(np.float32)
    beta = _sigmoid(bn).astype(np.float32)
    return Tokens(xq, xk, xv, g, beta)


# ---------------------------------------------------------------------------
# Turn / length recipes
# ---------------------------------------------------------------------------

def draw_raw_gates(T: int, n_v_heads: int, seed: int):
    """Raw-gate inputs (fp32): a, b [T, Hv] and per-head A_log, dt_bias [Hv]; stream (seed, 20_000)."""
    rng = _rng(seed, 20_000)
    a = rng.standard_normal((T, n_v_heads)).astype(np.float32)
    b = rng.standard_normal((T, n_v_heads)).astype(np.float32)
    A_log = np.log(rng.uniform(0.05, 0.5, n_v_heads)).astype(np.float32)
    dt_bias = rng.normal(-2.0, 0.5, n_v_heads).astype(np.float32)
    return a, b, A_log, dt_bias


def split_turns(total: int, n_turns: int, rng: np.random.Generator, lo: int = 0,
                hi: Optional[int] = None, max_tries: int = 100000) -> List[int]:
    """Split `total` tokens into `n_turns` positive turns.

    Each turn gets `lo` tokens plus a share of the rest cut at n_turns-1 sorted
    uniform points; redrawn until every turn is <= hi (when given).
    """
    rest = total - lo * n_turns
    assert rest >= 0
    for _ in range(max_tries):
        cuts = np.sort(rng.integers(0, rest + 1, size=n_turns - 1))
        parts = np.diff(np.concatenate([[0], cuts, [rest]])) + lo
        if parts.min() >= 1 and (hi is None or parts.max() <= hi):
            return [int(p) for p in parts]
    raise RuntimeError("could not draw turns within bounds")


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    shape: Shape
    seed: int = 0
    g_mu: float = 0.0
    g_scale: float = 0.1
    prenorm_qk: bool = False
    # single/varlen sessions: session lengths and per-session turn lengths
    session_lengths: List[int] = dataclasses.field(default_factory=list)
    turns: List[List[int]] = dataclasses.field(default_factory=list)
    n_slots: int = 0
    # forks over a session's committed state: question lengths
    fork_questions: List[int] = dataclasses.field(default_factory=list)
    # shared prefix: request prefix, group prefixes, branch lengths per group
    request_prefix: int = 0
    group_prefixes: List[int] = dataclasses.field(default_factory=list)
    branches: List[List[int]] = dataclasses.field(default_factory=list)

    def conv_weights(self) -> np.ndarray:
        return draw_conv_weights(self.shape, self.seed)

    def session_tokens(self, i: int, T: Optional[int] = None) -> Tokens:
        n = self.session_lengths[i] if T is None else T
        return draw_tokens(self.shape, n, self.seed, 1 + i, self.g_mu, self.g_scale, self.prenorm_qk)

    def extra_tokens(self, j: int, T: int) -> Tokens:
        """Tokens of question / branch / group segment j (independent stream)."""
        return draw_tokens(self.shape, T, self.seed, 10_000 + j, self.g_mu, self.g_scale, self.prenorm_qk)


def small_fp32(seed: int = 0) -> Workload:
    """Single layer, fp32 inputs: T=2048, 2 heads, d=64, C=64, one call."""
    return Workload("fp32_T2048_H2_d64_C64", Shape(2, 2, 64, 64, 64, FP32), seed=seed,
                    prenorm_qk=True, session_lengths=[2048], turns=[[2048]])


def qwen08b_replay(seed: int = 0) -> Workload:
    """Qwen3.5-0.8B-shaped layer: 16 heads, d=128, C=512, 41,802 tokens in 30 turns of 200..4000."""
    rng = _rng(seed, 99_999)
    turns = split_turns(41_802, 30, rng, lo=200, hi=4000)
    return Workload("bf16_T41802_H16_d128_C512_30turns", Shape(16, 16, 128, 128, 512, BF16),
                    seed=seed, session_lengths=[41_802], turns=[turns], n_slots=6,
                    fork_questions=[290])


def varlen8(seed: int = 0, scale: float = 1.0) -> Workload:
    """8 sessions, Hk=16, Hv=32, d=128, C=512, lengths log-uniform 4096..65536, 6 turns each."""
    rng = _rng(seed, 99_999)
    lens = [int(round(math.exp(rng.uniform(math.log(4096), math.log(65536))) * scale)) for _ in range(8)]
    lens = [max(l, 6) for l in lens]
    turns = [split_turns(l, 6, rng) for l in lens]
    return Workload("bf16_varlen8_Hk16_Hv32_d128_C512", Shape(16, 32, 128, 128, 512, BF16),
                    seed=seed, session_lengths=lens, turns=turns, n_slots=6)


def shared_prefix(seed: int = 0) -> Workload:
    """Request prefix 1,000; groups with prefixes 0/1/70/128; 4 branches per group of 1..200 tokens; C=64."""
    rng = _rng(seed, 99_999)
    branches = [[int(x) for x in rng.integers(1, 201, size=4)] for _ in range(4)]
    return Workload("bf16_shared_prefix_H16_d128_C64", Shape(16, 16, 128, 128, 64, BF16),
                    seed=seed, request_prefix=1000, group_prefixes=[0, 1, 70, 128],
                    branches=branches)


def long_session(seed: int = 0) -> Workload:
    """100,000 tokens, Hk=16, Hv=32, d=128, C=512, slow decay, 6 turns, 64 forks of 20..200 tokens."""
    rng = _rng(seed, 99_999)
    turns = split_turns(100_000, 6, rng)
    questions = [int(x) for x in rng.integers(20, 201, size=64)]
    return Workload("bf16_T100000_Hk16_Hv32_d128_C512_forks", Shape(16, 32, 128, 128, 512, BF16),
                    seed=seed, g_mu=-2.0, g_scale=1.0, session_lengths=[100_000], turns=[turns],
                    n_slots=6, fork_questions=questions)


WORKLOADS = {
    "small_fp32": small_fp32,
    "qwen08b_replay": qwen08b_replay,
    "varlen8": varlen8,
    "shared_prefix": shared_prefix,
    "long_session": long_session,
}


def grid_floor(n: int, c: int) -> int:
    return (n // c) * c


# ---------------------------------------------------------------------------
# Host arrays -> torch tensors (data movement only)
# ---------------------------------------------------------------------------

def to_torch(a: np.ndarray, dtype: str, device=None, pin: bool = False):
    """Stored input values as a torch tensor (bf16 bits -> torch.bfloat16, else float32)."""
    import torch
    a = np.ascontiguousarray(a)
    if dtype == BF16 and a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a.astype(np.float32, copy=False))
    if pin:
        t = t.pin_memory()
    return t.to(device) if device is not None else t


def tokens_to_torch(tok: Tokens, dtype: str, device=None, pin: bool = False):
    """(xq, xk, xv, g, beta) as torch tensors."""
    return (to_torch(tok.xq, dtype, device, pin), to_torch(tok.xk, dtype, device, pin),
            to_torch(tok.xv, dtype, device, pin), to_torch(tok.g, FP32, device, pin),
            to_torch(tok.beta, FP32, device, pin))
