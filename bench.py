#!/usr/bin/env python
"""Benchmark: chunked Gated-DeltaNet prefill tokens/s per layer on one GB300.

Default workload: the Qwen3.5-0.8B-shaped layer (16 heads, d_k = d_v = 128,
grid C = 512, bf16 inputs, fp32 state and outputs), one session of 41,802
synthetic tokens fed as 30 turns of 200..4,000 tokens with the sub-grid tail
held pending, a checkpoint of every turn's end state (6 rotating slots, written
by the turn's own prefill call), and at the end one fork that prefills the
330-token pending tail plus a 290-token question and restores the state from
the last turn's checkpoint ("The shadow reader", sections "One session's
state", "Exact on a grid" and "Who asks"). One step = that whole sequence.

Prints one JSON line. `value` = tokens processed per second with inputs
resident in HBM (CUDA events on the launching stream, K timed steps after W
warm-ups); `e2e` = the same with inputs copied from pinned host memory and the
outputs copied back inside the timed region; `roofline` = the dominant
kernel's achieved HBM bandwidth (algorithmic bytes / average launch time)
against the measured copy peak; `cpu_baseline` = the fp64 oracle on the host
cores over a bounded sample of the same workload.

`--impl reference` times the oracle itself (the reference arm of this method).
Several GPUs run independent replicas (the layer needs no exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s per layer on 1 GB300 + % of tensor-pipe/HBM roofline"
UNIT = "tokens/s"
# the arithmetic of the bf16-input path: what each stage computes in
PRECISION = {"inputs": "bf16", "conv_norm_gates": "fp32",
             "prologue_products": "tcgen05 kind::f16, fp32 accumulate: [q; k] k^T on bf16 hi/lo operand pairs "
                                  "(hi*hi + hi*lo + lo*hi); P T and [T; P T] [beta e^gamma k | beta v] on single fp16 "
                                  "operands",
             "triangular_inverse": "fp32 substitution + tf32 products",
             "record": "fp16 (W, Qe, K_tilde, U, O_intra) and fp32 e^gamma",
             "state_pass_products": "tcgen05 kind::f16: fp16 operands (record, state copy, U'), fp32 accumulate",
             "state": "fp32", "outputs": "fp32"}
FALLBACK_HBM_GBS = 6800.0

# Algorithmic HBM bytes per token of the fused layer: q and k per q/k head
# (2 d_k inputs), v per v-head, the output per v-head, g and beta per v-head.
def algorithmic_bytes_per_token(Hk, Hv, d, in_bytes, out_bytes):
    return Hk * 2 * d * in_bytes + Hv * d * in_bytes + Hv * d * out_bytes + Hv * 8


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group("gloo")
    return dist.get_rank(), dist.get_world_size(), int(os.environ.get("LOCAL_RANK", "0"))


def reduce_max_sum(ms: float, units: float):
    """(max of ms, sum of units) over ranks; identity on one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return ms, units
    t = torch.tensor([ms], dtype=torch.float64)
    u = torch.tensor([units], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tf32_tflops_probe(dev, n: int = 8192, reps: int = 10) -> float:
    """Dense tf32 matmul rate of this GPU, measured now (the state kernel's contractions run on tf32)."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(n, n, device=dev)
        b = torch.randn(n, n, device=dev)
        for _ in range(3):
            a @ b
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            a @ b
        e1.record()
        torch.cuda.synchronize()
        return 2.0 * n ** 3 * reps / (e0.elapsed_time(e1) / 1e3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.3)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + float("0." + f[0].split(".")[1])
            except Exception:
                ts = None
            rows.append((ts, f))
        inside = [f for ts, f in rows if ts is not None and self.t0 - 0.2 <= ts <= self.t1 + 0.2] or [f for _, f in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for f in inside for i in range(4) if f[6 + i].lower().startswith("active")})
        sm = [float(f[2]) for f in inside if re.match(r"^[0-9.]+$", f[2])]
        mx = [float(f[3]) for f in inside if re.match(r"^[0-9.]+$", f[3])]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------
# the workload step
# ---------------------------------------------------------------------------

class CudaRuntime:
    """The few CUDA runtime calls the end-to-end step needs, called directly (a torch copy per slice costs
    ~15 us of host time; these cost ~1-2 us): async copies, events without timing, stream waits."""

    def __init__(self):
        import ctypes
        path = None
        for line in open("/proc/self/maps"):
            if "libcudart.so" in line:
                path = line.split()[-1]
                break
        self.lib = ctypes.CDLL(path or "libcudart.so")
        self.c = ctypes
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        self.lib.cudaMemcpyAsync.argtypes = [vp, vp, sz, ctypes.c_int, vp]
        self.lib.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
        self.lib.cudaEventRecord.argtypes = [vp, vp]
        self.lib.cudaStreamWaitEvent.argtypes = [vp, vp, ctypes.c_uint]

    def _ok(self, r):
        if r != 0:
            raise RuntimeError(f"CUDA runtime error {r}")

    def event(self):
        e = self.c.c_void_p()
        self._ok(self.lib.cudaEventCreateWithFlags(self.c.byref(e), 2))   # cudaEventDisableTiming
        return e

    def h2d(self, dst, src, n, stream):
        self._ok(self.lib.cudaMemcpyAsync(dst, src, n, 1, stream))

    def d2h(self, dst, src, n, stream):
        self._ok(self.lib.cudaMemcpyAsync(dst, src, n, 2, stream))

    def record(self, ev, stream):
        self._ok(self.lib.cudaEventRecord(ev, stream))

    def wait(self, stream, ev):
        self._ok(self.lib.cudaStreamWaitEvent(stream, ev, 0))


class ReplayStep:
    """30 turns with checkpoints, then one fork over the pending tail plus a question."""

    def __init__(self, w, device):
        import torch
        from chunked_gated_deltanet_gb300 import gdn
        from chunked_gated_deltanet_gb300 import workloads as wl
        self.gdn, self.torch = gdn, torch
        self.w = w
        sh = w.shape
        self.T = w.session_lengths[0]
        self.Q = w.fork_questions[0]
        tok = wl.Tokens.concat([w.session_tokens(0), w.extra_tokens(0, self.Q)])
        self.rows = len(tok)
        self.desc = gdn.make_desc(sh.n_qk_heads, sh.n_v_heads, sh.d_k, sh.d_v, sh.grid_c, gdn.GDN_BF16, gdn.GDN_FP32)
        self.host = wl.tokens_to_torch(tok, sh.dtype, None, pin=True)
        self.host_cw = wl.to_torch(w.conv_weights(), sh.dtype, None, pin=True)
        self.x = [t.to(device) for t in self.host]
        self.cw = self.host_cw.to(device)
        self.out = torch.empty((self.rows, sh.n_v_heads, sh.d_v), dtype=torch.float32, device=device)
        self.host_out = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        C = sh.grid_c
        self.calls, end, committed = [], 0, 0
        for n in w.turns[0]:
            end += n
            take = (end - committed) // C * C
            self.calls.append((committed, end, take))
            committed += take
        self.committed = committed
        self.fork = (committed, self.rows)
        max_call = max([e - s for s, e, _ in self.calls] + [self.rows - committed])
        self.ws = gdn.workspace(self.desc, max_call, 1, device)
        self.sess = gdn.Session(self.desc, device)
        self.slots = [gdn.Session(self.desc, device) for _ in range(w.n_slots)]
        self.tokens_per_step = committed + (self.rows - committed)
        # dependent 64-token block steps of one head's state pass per bench step
        self.block_steps_per_step = sum(-(-take // 64) for _, _, take in self.calls) + -(-(self.rows - committed) // 64)
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.host) + \
            self.host_cw.numel() * self.host_cw.element_size()
        self.d2h_bytes = self.out.numel() * self.out.element_size()

    def step(self):
        g = self.gdn
        d, s, x, cw, out, ws = self.desc, self.sess, self.x, self.cw, self.out, self.ws
        g.gdn_session_init(d, s)
        for k, (a, b, take) in enumerate(self.calls):   # each turn keeps a checkpoint of its end state
            slot = self.slots[k % len(self.slots)]
            n = g.gdn_prefill_chunks_checkpoint(d, s, slot, x[0][a:b], x[1][a:b], x[2][a:b], x[3][a:b], x[4][a:b],
                                                cw, out[a:b], ws)
            assert n == take
        # the fork: tail + question above the committed rows, then back to the last turn's checkpoint
        a, b = self.fork
        g.gdn_prefill_chunks(d, s, x[0][a:b], x[1][a:b], x[2][a:b], x[3][a:b], x[4][a:b], cw, out[a:b], ws,
                             flags=g.GDN_ALLOW_PARTIAL)
        g.gdn_state_restore(d, s, slot)

    # call groups of the end-to-end copies (calls per copy; chosen by a sweep on the GB300 machine with the two
    # buffer sets: 8 calls per upload and 4 per download gave the shortest step, 2.998 ms against 3.17 ms
    # for 2 and 2 or for one copy per tensor of the whole step)
    up_group = 8
    down_group = 4

    def up_sizes(self, n):
        return [self.up_group] * (-(-n // self.up_group))

    def down_sizes(self, n):
        return [self.down_group] * (-(-n // self.down_group))

    def _e2e_setup(self):
        """Copy plan of the end-to-end step. Every copy costs a few microseconds of idle host link, so inputs
        go up in fewer, larger copies: the gates and conv weights of the whole step first, then the q/k/v rows
        of groups of calls (a call waits only for its group); outputs come down by groups of calls. Groups
        that are too large make the compute wait for the link. Two sets of device buffers take turns, so
        that the next step's inputs go up while this step computes, as in a serving loop; a set is refilled
        once the compute of the step before last no longer reads it, and its outputs are overwritten once
        their download is done. Raw pointers, two copy streams and the events that order them."""
        torch = self.torch
        self.rt = CudaRuntime()
        self.h2d, self.d2h = torch.cuda.Stream(), torch.cuda.Stream()
        self.sets = [(self.x, self.cw, self.out),
                     ([torch.empty_like(t) for t in self.x], torch.empty_like(self.cw), torch.empty_like(self.out))]
        spans = [(a, b, take) for a, b, take in self.calls] + [(self.fork[0], self.fork[1], self.fork[1] - self.fork[0])]
        n = len(spans)

        def groups(sizes):
            out, k = [], 0
            for g in sizes:
                if k >= n:
                    break
                out.append((k, min(n, k + g)))
                k += g
            if k < n:
                out.append((k, n))
            return out

        up_groups, self.up_of = groups(self.up_sizes(n)), [0] * n
        for gi, (k0, k1) in enumerate(up_groups):
            for k in range(k0, k1):
                self.up_of[k] = gi
        down_groups = groups(self.down_sizes(n))
        self.plans = []
        for x, cw, out in self.sets:
            row_bytes = [(t.stride(0) * t.element_size(), d.data_ptr(), t.data_ptr()) for d, t in zip(x, self.host)]
            out_row = out.stride(0) * out.element_size()
            # uploads: whole-step gates and weights, then q, k, v rows by call group
            first = [(dp, hp, self.rows * rb) for rb, dp, hp in row_bytes[3:]]
            first.append((cw.data_ptr(), self.host_cw.data_ptr(), cw.numel() * cw.element_size()))
            ups = []
            for k0, k1 in up_groups:
                r0 = spans[k0 - 1][1] if k0 > 0 else 0
                r1 = spans[k1 - 1][1]
                ups.append([(dp + r0 * rb, hp + r0 * rb, (r1 - r0) * rb) for rb, dp, hp in row_bytes[:3]])
            # downloads: committed output rows by call group, issued after the group's last call
            downs = {}
            for k0, k1 in down_groups:
                r0, r1 = spans[k0][0], spans[k1 - 1][0] + spans[k1 - 1][2]
                downs[k1 - 1] = (self.host_out.data_ptr() + r0 * out_row, out.data_ptr() + r0 * out_row,
                                 (r1 - r0) * out_row)
            ev = {"up": [self.rt.event() for _ in ups], "call": [self.rt.event() for _ in range(n)],
                  "in_free": self.rt.event(), "out_free": self.rt.event()}
            self.plans.append((first, ups, downs, ev))
        self.n_copies = len(self.plans[0][0]) + 3 * len(self.plans[0][1]) + len(self.plans[0][2])
        self.gate_ev = self.rt.event()
        self.k_e2e = 0

    def e2e_gate(self, steps: int = 2):
        """The uploads of the next `steps` steps wait for the compute stream's current position (the start
        of a timed region), so that none of their copies runs before it."""
        if not hasattr(self, "plans"):
            self._e2e_setup()
        self.rt.record(self.gate_ev, self.torch.cuda.current_stream().cuda_stream)
        self.gate_left = steps

    def e2e_step(self):
        """The step through host buffers on the next set of device buffers: inputs go up on a copy stream
        ahead of the compute (each call waits for the upload group that holds its rows), outputs come back
        on another copy stream by call group. e2e_finish() makes the compute stream wait for the outstanding
        downloads."""
        g, torch = self.gdn, self.torch
        if not hasattr(self, "plans"):
            self._e2e_setup()
        rt = self.rt
        si = self.k_e2e % 2
        self.k_e2e += 1
        (x, cw, out), (first, ups, downs, ev) = self.sets[si], self.plans[si]
        comp = torch.cuda.current_stream().cuda_stream
        h2d, d2h = self.h2d.cuda_stream, self.d2h.cuda_stream
        if getattr(self, "gate_left", 0) > 0:
            rt.wait(h2d, self.gate_ev)
            self.gate_left -= 1
        rt.wait(h2d, ev["in_free"])          # the step before last no longer reads this set's inputs
        for dst, src, nb in first:
            rt.h2d(dst, src, nb, h2d)
        for gi, grp in enumerate(ups):
            for dst, src, nb in grp:
                rt.h2d(dst, src, nb, h2d)
            rt.record(ev["up"][gi], h2d)
        rt.wait(comp, ev["out_free"])        # this set's outputs of the step before last are downloaded
        d, s, ws = self.desc, self.sess, self.ws

        def after(k):
            spec = downs.get(k)
            if spec is not None:
                rt.record(ev["call"][k], comp)
                rt.wait(d2h, ev["call"][k])
                rt.d2h(*spec, d2h)

        g.gdn_session_init(d, s)
        for k, (a, b, take) in enumerate(self.calls):
            rt.wait(comp, ev["up"][self.up_of[k]])
            slot = self.slots[k % len(self.slots)]
            n = g.gdn_prefill_chunks_checkpoint(d, s, slot, x[0][a:b], x[1][a:b], x[2][a:b], x[3][a:b], x[4][a:b],
                                                cw, out[a:b], ws)
            assert n == take
            after(k)
        a, b = self.fork
        k = len(self.calls)
        rt.wait(comp, ev["up"][self.up_of[k]])
        g.gdn_prefill_chunks(d, s, x[0][a:b], x[1][a:b], x[2][a:b], x[3][a:b], x[4][a:b], cw, out[a:b], ws,
                             flags=g.GDN_ALLOW_PARTIAL)
        g.gdn_state_restore(d, s, slot)
        rt.record(ev["in_free"], comp)
        after(k)
        rt.record(ev["out_free"], d2h)
        self.last_out = out

    def e2e_finish(self):
        """The compute stream waits for every download issued so far."""
        comp = self.torch.cuda.current_stream().cuda_stream
        for _, _, _, ev in self.plans:
            self.rt.wait(comp, ev["out_free"])

    def config(self):
        sh = self.w.shape
        return {"workload": self.w.name, "sessions": 1, "session_tokens": self.T, "turns": len(self.w.turns[0]),
                "checkpoint_slots": len(self.slots), "fork_tokens": self.rows - self.committed,
                "tokens_per_step": self.tokens_per_step, "n_qk_heads": sh.n_qk_heads, "n_v_heads": sh.n_v_heads,
                "d_k": sh.d_k, "d_v": sh.d_v, "grid_c": sh.grid_c, "inputs": "bf16", "state": "fp32",
                "outputs": "fp32",
                "l2": f"inputs larger than L2 ({self.h2d_bytes / 1e6:.0f} MB read per step vs 129 MB L2)",
                "parallelism": "replicas"}


class VarlenStep:
    """8 sessions (Hk 16, Hv 32, grid 512) fed in 6 turn rounds: one varlen call per round, which also writes
    every session's round checkpoint into that round's slot; pending tails carried between rounds."""

    def __init__(self, w, device):
        import torch
        from chunked_gated_deltanet_gb300 import gdn
        from chunked_gated_deltanet_gb300 import workloads as wl
        self.gdn, self.w = gdn, w
        sh = w.shape
        self.desc = gdn.make_desc(sh.n_qk_heads, sh.n_v_heads, sh.d_k, sh.d_v, sh.grid_c, gdn.GDN_BF16, gdn.GDN_FP32)
        n, C, R = len(w.session_lengths), sh.grid_c, len(w.turns[0])
        toks = [w.session_tokens(i) for i in range(n)]
        ends, committed = [0] * n, [0] * n
        self.rounds, max_rows, self.block_steps_per_step = [], 0, 0
        for r in range(R):
            parts, cu, longest = [], [0], 0
            for i in range(n):
                ends[i] += w.turns[i][r]
                parts.append(toks[i].slice(committed[i], ends[i]))
                cu.append(cu[-1] + ends[i] - committed[i])
                take = (ends[i] - committed[i]) // C * C
                longest = max(longest, -(-take // 64))
                committed[i] += take
            x = wl.tokens_to_torch(wl.Tokens.concat(parts), sh.dtype, device)
            out = torch.empty((cu[-1], sh.n_v_heads, sh.d_v), dtype=torch.float32, device=device)
            self.rounds.append((cu, x, out))
            max_rows = max(max_rows, cu[-1])
            self.block_steps_per_step += longest
        self.tokens_per_step = sum(committed)
        self.cw = wl.to_torch(w.conv_weights(), sh.dtype, device)
        self.ws = gdn.workspace(self.desc, max_rows + 64 * n, n, device)
        self.sess = [gdn.Session(self.desc, device) for _ in range(n)]
        self.slots = [[gdn.Session(self.desc, device) for _ in range(n)] for _ in range(R)]
        self.n = n

    def step(self):
        g = self.gdn
        for s in self.sess:
            g.gdn_session_init(self.desc, s)
        for r, (cu, x, out) in enumerate(self.rounds):
            g.gdn_prefill_varlen_checkpoint(self.desc, self.sess, self.slots[r], cu, *x, self.cw, out, self.ws)

    def config(self):
        sh = self.w.shape
        return {"workload": self.w.name, "sessions": self.n, "session_tokens": list(self.w.session_lengths),
                "turn_rounds": len(self.rounds), "checkpoint_slots": len(self.slots), "tokens_per_step":
                self.tokens_per_step, "n_qk_heads": sh.n_qk_heads, "n_v_heads": sh.n_v_heads, "d_k": sh.d_k,
                "d_v": sh.d_v, "grid_c": sh.grid_c, "inputs": "bf16", "state": "fp32", "outputs": "fp32",
                "l2": "inputs larger than L2", "parallelism": "replicas"}


class LongStep:
    """One 100,000-token session (Hk 16, Hv 32, slow decay) in 6 turns, each writing its checkpoint, then
    64 forks of 20..200 question tokens over the committed state. The forks run as one branches call:
    each branch is the pending tail plus its question, starting from the committed state read in place
    (so the state needs no restore afterwards)."""

    def __init__(self, w, device):
        import torch
        from chunked_gated_deltanet_gb300 import gdn
        from chunked_gated_deltanet_gb300 import workloads as wl
        self.gdn, self.w = gdn, w
        sh = w.shape
        C = sh.grid_c
        self.desc = gdn.make_desc(sh.n_qk_heads, sh.n_v_heads, sh.d_k, sh.d_v, sh.grid_c, gdn.GDN_BF16, gdn.GDN_FP32)
        T = w.session_lengths[0]
        tok = w.session_tokens(0)
        self.x = wl.tokens_to_torch(tok, sh.dtype, device)
        self.out = torch.empty((T, sh.n_v_heads, sh.d_v), dtype=torch.float32, device=device)
        self.calls, end, committed = [], 0, 0
        for n in w.turns[0]:
            end += n
            take = (end - committed) // C * C
            self.calls.append((committed, end, take))
            committed += take
        tail = tok.slice(committed, T)
        forks = [wl.Tokens.concat([tail, w.extra_tokens(j, q)]) for j, q in enumerate(w.fork_questions)]
        self.cu = [0]
        for f in forks:
            self.cu.append(self.cu[-1] + len(f))
        self.xf = wl.tokens_to_torch(wl.Tokens.concat(forks), sh.dtype, device)
        self.outf = torch.empty((self.cu[-1], sh.n_v_heads, sh.d_v), dtype=torch.float32, device=device)
        self.cw = wl.to_torch(w.conv_weights(), sh.dtype, device)
        max_call = max([e - s for s, e, _ in self.calls] + [self.cu[-1]])
        self.ws = gdn.workspace(self.desc, max_call + 64 * len(forks), len(forks), device)
        self.sess = gdn.Session(self.desc, device)
        self.slots = [gdn.Session(self.desc, device) for _ in range(w.n_slots)]
        self.branches = [gdn.Session(self.desc, device) for _ in forks]
        self.committed, self.n_forks = committed, len(forks)
        self.tokens_per_step = committed + self.cu[-1]
        self.block_steps_per_step = sum(-(-t // 64) for _, _, t in self.calls) + max(-(-len(f) // 64) for f in forks)

    def step(self):
        g, d, x, cw = self.gdn, self.desc, self.x, self.cw
        g.gdn_session_init(d, self.sess)
        for k, (a, b, take) in enumerate(self.calls):
            n = g.gdn_prefill_chunks_checkpoint(d, self.sess, self.slots[k % len(self.slots)], *(t[a:b] for t in x), cw,
                                                self.out[a:b], self.ws)
            assert n == take
        g.gdn_prefill_branches(d, self.sess, self.branches, self.cu, *self.xf, cw, self.outf, self.ws,
                               flags=g.GDN_ALLOW_PARTIAL)

    def config(self):
        sh = self.w.shape
        return {"workload": self.w.name, "sessions": 1, "session_tokens": self.w.session_lengths[0],
                "turns": len(self.calls), "checkpoint_slots": len(self.slots), "forks": self.n_forks,
                "fork_tokens": self.cu[-1], "forks_as": "one branches call from the committed state",
                "tokens_per_step": self.tokens_per_step, "n_qk_heads": sh.n_qk_heads, "n_v_heads": sh.n_v_heads,
                "d_k": sh.d_k, "d_v": sh.d_v, "grid_c": sh.grid_c, "inputs": "bf16", "state": "fp32",
                "outputs": "fp32", "l2": "inputs larger than L2", "parallelism": "replicas"}


class SmallStep:
    """The small fp32 layer (T = 2,048, 2 heads, d = 64, grid 64): one call from a zero state."""

    def __init__(self, w, device):
        import torch
        from chunked_gated_deltanet_gb300 import gdn
        from chunked_gated_deltanet_gb300 import workloads as wl
        self.gdn, self.w = gdn, w
        sh = w.shape
        self.desc = gdn.make_desc(sh.n_qk_heads, sh.n_v_heads, sh.d_k, sh.d_v, sh.grid_c, gdn.GDN_FP32, gdn.GDN_FP32)
        T = w.session_lengths[0]
        self.x = wl.tokens_to_torch(w.session_tokens(0), sh.dtype, device)
        self.cw = wl.to_torch(w.conv_weights(), sh.dtype, device)
        self.out = torch.empty((T, sh.n_v_heads, sh.d_v), dtype=torch.float32, device=device)
        self.ws = gdn.workspace(self.desc, T, 1, device)
        self.sess = gdn.Session(self.desc, device)
        self.tokens_per_step = T
        self.block_steps_per_step = -(-T // 64)

    def step(self):
        g = self.gdn
        g.gdn_session_init(self.desc, self.sess)
        assert g.gdn_prefill_chunks(self.desc, self.sess, *self.x, self.cw, self.out, self.ws) == self.tokens_per_step

    def config(self):
        sh = self.w.shape
        return {"workload": self.w.name, "sessions": 1, "session_tokens": self.tokens_per_step, "calls": 1,
                "n_qk_heads": sh.n_qk_heads, "n_v_heads": sh.n_v_heads, "d_k": sh.d_k, "d_v": sh.d_v,
                "grid_c": sh.grid_c, "inputs": "fp32", "state": "fp32", "outputs": "fp32",
                "l2": "inputs smaller than L2 (the whole layer is 2,048 tokens)", "parallelism": "replicas"}


def kernel_split(ktimes: dict, steps: int) -> dict:
    return {k: {"launches_per_step": v[0] / steps, "ms_per_step": round(v[2] / steps, 4),
                "share": round(v[2] / max(sum(x[2] for x in ktimes.values()), 1e-12), 4)} for k, v in ktimes.items()}


def measure_step(step, steps: int, warmup: int):
    """Device time of `steps` steps (CUDA events on the current stream, after `warmup` steps), then the same
    steps again with an event pair around every launch for the per-kernel split."""
    import torch
    from chunked_gated_deltanet_gb300 import gdn
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        step.step()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step.step()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    gdn.gdn_timing_begin(100_000)
    for _ in range(steps):
        step.step()
    torch.cuda.synchronize()
    return ms, gdn.gdn_timing_end()


def other_config_measure(name: str, w, dev, steps: int, warmup: int = 3) -> dict:
    """Tokens/s, HBM roofline fractions (step and dominant kernel) and the kernel split of one of the other
    workloads, in the line of the headline one."""
    cls = {"varlen8": VarlenStep, "long_session": LongStep, "small_fp32": SmallStep}[name]
    step = cls(w, dev)
    ms, kt = measure_step(step, steps, warmup)
    sh = w.shape
    in_b = 2 if sh.dtype == "bf16" else 4
    bpt = algorithmic_bytes_per_token(sh.n_qk_heads, sh.n_v_heads, sh.d_k, in_b, 4)
    peak, peak_src = measured_peaks()
    rt = dict(kt)
    if "prep_wy_tail" in rt and "prep_wy" in rt:
        a, b = rt.pop("prep_wy_tail"), rt["prep_wy"]
        rt["prep_wy"] = (a[0] + b[0], a[1] + b[1], a[2] + b[2])
    prefill = {k: v for k, v in rt.items() if k in ("prep_wy", "state_output", "prefill_fused")}
    dom_name, (launches, timed, tot) = max(prefill.items(), key=lambda kv: kv[1][2])
    tokens_per_launch = step.tokens_per_step / (launches / steps)
    avg_ms = tot / max(timed, 1)
    ms_step = ms / steps
    out = {"config": step.config(), "steps": steps, "warmup": warmup, "ms_per_step": round(ms_step, 4),
           "tokens_per_step": step.tokens_per_step, "value": round(step.tokens_per_step / (ms_step / 1e3), 1),
           "unit": UNIT, "algorithmic_bytes_per_token": bpt,
           "step_frac": round(bpt * step.tokens_per_step / (ms_step / 1e3) / 1e9 / peak, 4),
           "dominant_kernel": {"kernel": dom_name, "avg_launch_ms": round(avg_ms, 4),
                               "frac": round(bpt * tokens_per_launch / (avg_ms / 1e3) / 1e9 / peak, 4)},
           "peak_gbs": peak, "peak_source": peak_src, "kernels": kernel_split(kt, steps),
           "gpu_launches_per_step": sum(v[0] for v in kt.values()) / steps}
    if "state_output" in kt:
        out["state_pass_us_per_block_step"] = round(kt["state_output"][2] * 1e3 / (step.block_steps_per_step * steps), 3)
    return out


# ---------------------------------------------------------------------------
# Batched decode (one token for each of n sessions), captured once in a CUDA graph
# ---------------------------------------------------------------------------

L2_BYTES = 129 * 1024 * 1024


def decode_measure(w, dev, n_sess: int = 64, steps: int = 50):
    """Replays of one captured decode step over n_sess sessions of the bench layer; HBM roofline of the
    step = every state read and written once, plus the conv states, inputs and outputs."""
    import torch
    from chunked_gated_deltanet_gb300 import gdn
    sh = w.shape
    desc = gdn.make_desc(sh.n_qk_heads, sh.n_v_heads, sh.d_k, sh.d_v, sh.grid_c, gdn.GDN_BF16, gdn.GDN_FP32)
    sessions = [gdn.Session(desc, dev) for _ in range(n_sess)]
    gen = torch.Generator(device=dev).manual_seed(5)
    bf = lambda *shape: torch.randn(*shape, generator=gen, device=dev).to(torch.bfloat16)
    nq, nv = sh.n_qk_heads * sh.d_k, sh.n_v_heads * sh.d_v
    xq, xk, xv = bf(n_sess, nq), bf(n_sess, nq), bf(n_sess, nv)
    g = -0.1 * torch.nn.functional.softplus(torch.randn(n_sess, sh.n_v_heads, generator=gen, device=dev))
    beta = torch.sigmoid(torch.randn(n_sess, sh.n_v_heads, generator=gen, device=dev))
    cw = bf(2 * nq + nv, 4)
    out = torch.empty((n_sess, sh.n_v_heads, sh.d_v), device=dev)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.gdn_decode_step(desc, sessions, xq, xk, xv, g, beta, cw, out)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / steps
    state = n_sess * sh.n_v_heads * sh.d_k * sh.d_v * 4
    conv = n_sess * 3 * (2 * nq + nv) * 2
    io = n_sess * ((2 * nq + nv) * 2 + sh.n_v_heads * 8 + sh.n_v_heads * sh.d_v * 4)
    bytes_step = 2 * state + 2 * conv + io
    peak, _ = measured_peaks()
    gbs = bytes_step / (us / 1e6) / 1e9
    l2 = "state larger than L2" if state > L2_BYTES else "state fits L2 (replays may hit it)"
    return {"sessions": n_sess, "launch": "CUDA graph replay of one gdn_decode_step", "l2": l2, "us_per_step": round(us, 2),
            "tokens_per_s": round(n_sess / (us / 1e6), 1), "bytes_per_step": bytes_step,
            "achieved_gbs": round(gbs, 1), "peak_gbs": peak, "frac": round(gbs / peak, 4), "bound": "hbm"}


def host_link_measure(step, reps: int = 3):
    """Host link speed on this machine, with the step's own pinned buffers: every input tensor up, the output
    down, and both at once (one large copy per tensor, copy streams timed by events); the step's copy floor
    is its bytes over those speeds."""
    import torch
    ups = [(d, h) for d, h in zip(step.x, step.host)]
    down = (step.host_out, step.out)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        torch.cuda.synchronize()
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    def up():
        with torch.cuda.stream(s1):
            for d, h in ups:
                d.copy_(h, non_blocking=True)

    def dn():
        with torch.cuda.stream(s2):
            down[0].copy_(down[1], non_blocking=True)

    def both():
        up()
        dn()

    hb = sum(h.numel() * h.element_size() for _, h in ups)
    db = down[1].numel() * down[1].element_size()
    t_up, t_dn, t_both = timed(up), timed(dn), timed(both)
    floor_ms = max(t_up * step.h2d_bytes / hb, t_dn * step.d2h_bytes / db,
                   t_both * (step.h2d_bytes + step.d2h_bytes) / (hb + db)) * 1e3
    return {"h2d_gbs": round(hb / t_up / 1e9, 1), "d2h_gbs": round(db / t_dn / 1e9, 1),
            "both_gbs": round((hb + db) / t_both / 1e9, 1), "copy_floor_ms": round(floor_ms, 4)}


# ---------------------------------------------------------------------------
# Branches of one shared prefix: one call reading the prefix state in place vs restore + prefill per branch
# ---------------------------------------------------------------------------

def branches_measure(dev, reps: int = 20):
    import torch
    from chunked_gated_deltanet_gb300 import gdn
    from chunked_gated_deltanet_gb300 import workloads as wl
    w = wl.shared_prefix()
    sh = w.shape
    desc = gdn.make_desc(sh.n_qk_heads, sh.n_v_heads, sh.d_k, sh.d_v, sh.grid_c, gdn.GDN_BF16, gdn.GDN_FP32)
    cut = wl.grid_floor(w.request_prefix, sh.grid_c)
    x_req = wl.tokens_to_torch(w.session_tokens(0, cut), sh.dtype, dev)
    cw = wl.to_torch(w.conv_weights(), sh.dtype, dev)
    lengths = [n for br in w.branches for n in br]
    tails = [w.extra_tokens(200 + i, n) for i, n in enumerate(lengths)]
    cu = [0]
    for t in tails:
        cu.append(cu[-1] + len(t))
    x = wl.tokens_to_torch(wl.Tokens.concat(tails), sh.dtype, dev)
    out = torch.empty((cu[-1], sh.n_v_heads, sh.d_v), device=dev)
    ws = gdn.workspace(desc, cu[-1] + 64 * len(tails) + cut, len(tails), dev)
    prefix = gdn.Session(desc, dev)
    gdn.gdn_prefill_chunks(desc, prefix, *x_req, cw, torch.empty((cut, sh.n_v_heads, sh.d_v), device=dev), ws)
    branches = [gdn.Session(desc, dev) for _ in tails]

    def per_branch():
        for i, b in enumerate(branches):
            gdn.gdn_state_restore(desc, b, prefix)
            a, e = cu[i], cu[i + 1]
            gdn.gdn_prefill_chunks(desc, b, *(t[a:e] for t in x), cw, out[a:e], ws, flags=gdn.GDN_ALLOW_PARTIAL)

    def one_call():
        gdn.gdn_prefill_branches(desc, prefix, branches, cu, *x, cw, out, ws, flags=gdn.GDN_ALLOW_PARTIAL)

    res = {}
    for name, fn in (("restore_and_prefill_per_branch", per_branch), ("one_branches_call", one_call)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        res[name] = round(e0.elapsed_time(e1) * 1e3 / reps, 1)
    return {"workload": f"{len(tails)} branches of {min(lengths)}-{max(lengths)} tokens ({cu[-1]} in all) from a "
                        f"{cut}-token prefix state, {sh.n_v_heads} heads, d={sh.d_k}, grid {sh.grid_c}",
            "us_per_round": res, "tokens_per_s_one_call": round(cu[-1] / (res["one_branches_call"] / 1e6), 1),
            "speedup": round(res["restore_and_prefill_per_branch"] / res["one_branches_call"], 2)}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle over a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample(w, n_tokens: int):
    import numpy as np
    import oracle
    from chunked_gated_deltanet_gb300 import workloads as wl
    tok = w.session_tokens(0).slice(0, n_tokens)
    f = lambda a: wl.as_f64(a, w.shape.dtype)
    args = (f(tok.xq), f(tok.xk), f(tok.xv), tok.g.astype(np.float64), tok.beta.astype(np.float64),
            f(w.conv_weights()))
    sh = w.shape

    def run():
        oracle.layer(*args, sh.n_qk_heads, sh.n_v_heads)

    return run


def oracle_one_thread() -> dict:
    """The oracle on one host thread (measured in a child process started with OMP_NUM_THREADS=1): the
    2,048-token fp32 layer (2 heads, d = 64) whole, and one v-head of the 41,802-token replay session's
    first 41,472 tokens."""
    import numpy as np
    import oracle
    from chunked_gated_deltanet_gb300 import workloads as wl
    out = {}
    w = wl.small_fp32()
    t0 = time.time()
    oracle_sample(w, w.session_lengths[0])()
    dt = time.time() - t0
    out["fp32_T2048_H2_d64"] = {"tokens_per_s": round(w.session_lengths[0] / dt, 1), "seconds": round(dt, 3)}
    w = wl.qwen08b_replay()
    sh = w.shape
    n = wl.grid_floor(w.session_lengths[0], sh.grid_c)
    tok = w.session_tokens(0).slice(0, n)
    k_heads, qk_cols, v_cols = oracle.head_columns(sh.n_qk_heads, sh.n_v_heads, sh.d_k, sh.d_v, [0])
    f = lambda a: wl.as_f64(a, sh.dtype)
    cw = w.conv_weights()
    chan = np.concatenate([qk_cols, sh.n_qk_heads * sh.d_k + qk_cols, 2 * sh.n_qk_heads * sh.d_k + v_cols])
    t0 = time.time()
    oracle.layer(f(tok.xq[:, qk_cols]), f(tok.xk[:, qk_cols]), f(tok.xv[:, v_cols]), tok.g[:, [0]].astype(np.float64),
                 tok.beta[:, [0]].astype(np.float64), f(cw[chan]), 1, 1)
    dt = time.time() - t0
    out["replay_one_head"] = {"tokens_per_s": round(n / dt, 1), "seconds": round(dt, 3), "tokens": n}
    return out


def oracle_one_thread_child():
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-thread"], env=env,
                           capture_output=True, text=True, timeout=300, cwd=ROOT)
        return json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else None
    except Exception:
        return None


def cpu_threads(n_heads: int) -> int:
    try:
        c = len(os.sched_getaffinity(0))
    except Exception:
        c = os.cpu_count() or 1
    return max(1, min(c, n_heads))


# kernel kind -> (the sources that define its code, its ncu summary); the summary's figures are used only
# while the sha256 over those sources matches the one it records
PROFILED = {"prefill_fused": (("prefill_fused.cu", "chain_umma.cuh", "prologue_umma.cuh", "umma.cuh", "mma.cuh", "common.cuh"),
                              "prefill_fused_qwen08b_replay.md"),
            "prep_wy": (("prep_umma.cu", "prologue_umma.cuh", "umma.cuh", "mma.cuh", "common.cuh"),
                        "prep_umma_long_session_branches.md"),
            "state_output": (("chain_umma.cu", "chain_umma.cuh", "umma.cuh", "mma.cuh", "common.cuh"),
                             "state_output_long_session_branches.md")}


def source_sha16(names) -> str:
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "chunked_gated_deltanet_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def traffic_record(kind: str):
    """DRAM bytes per token of a kernel from its committed ncu summary, if its source is unchanged since."""
    if kind not in PROFILED:
        return None
    src_names, prof_name = PROFILED[kind]
    prof = os.path.join(ROOT, "profiles", prof_name)
    try:
        sha = source_sha16(src_names)
        txt = open(prof).read()
        m_sha = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
        m_b = re.search(r"dram_bytes_per_token:\s*([0-9.]+)", txt)
        if m_sha and m_b and m_sha.group(1) == sha:
            return float(m_b.group(1))
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode and branch measurements")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the other workloads' lines (8-session batch, 100k session, small fp32 layer)")
    ap.add_argument("--cpu-sample-tokens", type=int, default=41472)
    ap.add_argument("--oracle-one-thread", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--workload", choices=["replay", "varlen8", "long_session"], default="replay",
                    help="replay: the headline (default); varlen8 / long_session: the batch and long-session "
                         "configurations, reported without e2e")
    args = ap.parse_args()
    if args.oracle_one_thread:   # child mode of oracle_one_thread_child (host only)
        print(json.dumps(oracle_one_thread()), flush=True)
        return
    if args.warmup < 3:
        print("note: fewer than 3 warm-up steps", file=sys.stderr)

    rank, world, local = _dist()
    from chunked_gated_deltanet_gb300 import workloads as wl
    w = {"replay": wl.qwen08b_replay, "varlen8": wl.varlen8, "long_session": wl.long_session}[args.workload]()

    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    import torch
    from chunked_gated_deltanet_gb300 import gdn
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gdn.load_library()
    step = {"replay": ReplayStep, "varlen8": VarlenStep, "long_session": LongStep}[args.workload](w, dev)
    if args.workload != "replay":   # the e2e, decode, branch and other-config figures belong to the headline run
        args.no_e2e = args.no_decode = args.no_other_configs = True
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        step.step()
    torch.cuda.synchronize()

    # --- device-resident timed region ---
    clk = ClockSampler(local)
    clk.start()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk.mark("t0")
    ev0.record(stream)
    for _ in range(args.steps):
        step.step()
    ev1.record(stream)
    torch.cuda.synchronize()
    clk.mark("t1")
    barrier()
    ms = ev0.elapsed_time(ev1)
    # --- the same steps again with an event pair around every launch (per-kernel times; kept out of the
    #     region above, whose step time the extra event records would lengthen) ---
    gdn.gdn_timing_begin(100_000)
    for _ in range(args.steps):
        step.step()
    torch.cuda.synchronize()
    ktimes = gdn.gdn_timing_end()
    clocks = clk.stop()
    ms_max, tokens_all = reduce_max_sum(ms, step.tokens_per_step * args.steps)
    config = step.config()
    value = tokens_all / (ms_max / 1e3)

    # --- end to end through host buffers ---
    e2e = None
    if not args.no_e2e:
        for _ in range(2):
            step.e2e_step()
        step.e2e_finish()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step.e2e_gate(2)   # the first two steps' uploads start inside the timed region
        for _ in range(args.steps):
            step.e2e_step()
        step.e2e_finish()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems, etok = reduce_max_sum(e0.elapsed_time(e1), step.tokens_per_step * args.steps)
        # the downloaded outputs are the device's, row for row
        assert torch.equal(step.host_out, step.last_out.cpu()), "host outputs differ from the device outputs"
        e2e = {"value": etok / (ems / 1e3), "unit": UNIT, "h2d_bytes_per_step": step.h2d_bytes,
               "d2h_bytes_per_step": step.d2h_bytes, "ms_per_step": round(ems / args.steps, 4)}
        if hasattr(step, "n_copies"):
            e2e["copies"] = (f"{step.n_copies} copies per step: gates and weights, then input rows by groups of "
                             f"{step.up_group} calls on one copy stream ahead of the compute; output rows by groups "
                             f"of {step.down_group} calls on another as soon as a group is done; two sets of device "
                             "buffers take turns, so the next step's inputs go up while this step computes")
        e2e["host_link"] = host_link_measure(step)

    # --- roofline of the dominant kernel ---
    sh = w.shape
    bpt = algorithmic_bytes_per_token(sh.n_qk_heads, sh.n_v_heads, sh.d_k, 2, 4)
    # the prologue of a call's last blocks (run beside the state pass of its first ones) is the same kernel
    # over the rest of the call's tokens: merged with the others for the roofline
    rtimes = dict(ktimes)
    if "prep_wy_tail" in rtimes and "prep_wy" in rtimes:
        a, b = rtimes.pop("prep_wy_tail"), rtimes["prep_wy"]
        rtimes["prep_wy"] = (a[0] + b[0], a[1] + b[1], a[2] + b[2])
    dom = max(rtimes.items(), key=lambda kv: kv[1][2])
    name, (launches, timed, tot_ms) = dom
    avg_ms = tot_ms / max(timed, 1)
    # tokens one launch of the dominant kernel processes (prefill kernels: every consumed token of the step)
    prefill_launches = launches / args.steps
    tokens_per_launch = step.tokens_per_step / prefill_launches
    achieved = bpt * tokens_per_launch / (avg_ms / 1e3) / 1e9
    peak, peak_src = measured_peaks()
    traffic_bpt = traffic_record(name) if args.workload == "replay" else None   # profiled on the replay
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_src, "kernel": name,
                "algorithmic_bytes_per_token": bpt, "tokens_per_launch": round(tokens_per_launch, 1),
                "avg_launch_ms": round(avg_ms, 4),
                "traffic": round(traffic_bpt * tokens_per_launch) if traffic_bpt else None,
                "step_frac": round(bpt * step.tokens_per_step / (ms / args.steps / 1e3) / 1e9 / peak, 4)}
    kernels = {k: {"launches_per_step": v[0] / args.steps, "ms_per_step": round(v[2] / args.steps, 4),
                   "share": round(v[2] / sum(x[2] for x in ktimes.values()), 4)} for k, v in ktimes.items()}
    # the state pass: tensor-pipe fraction against the tf32 rate measured now, and the single-session latency
    # floor (dependent 64-token block steps of one head x the measured time per step)
    state_pass = None
    if "state_output" in ktimes and "prefill_fused" not in ktimes:   # every call of the step in two launches
        launches, timed, tot = ktimes["state_output"]
        blocks = step.block_steps_per_step * args.steps
        us_block = tot * 1e3 / blocks
        flops = 6.0 * sh.d_k * sh.d_v * sh.n_v_heads * step.tokens_per_step * args.steps
        tf32 = tf32_tflops_probe(dev)
        achieved_tf = flops / (tot / 1e3) / 1e12
        state_pass = {"bound": "latency", "us_per_block_step": round(us_block, 3),
                      "latency_floor_ms_per_step": round(step.block_steps_per_step * us_block / 1e3, 3),
                      "tensor": {"flops_per_token": 6 * sh.d_k * sh.d_v * sh.n_v_heads, "achieved_tflops":
                                 round(achieved_tf, 1), "tf32_tflops_measured_now": round(tf32, 1),
                                 "frac": round(achieved_tf / tf32, 4)}}
    gpu_launches = int(sum(v[0] for v in ktimes.values()))

    decode = None if args.no_decode else [decode_measure(w, dev, n) for n in (1, 256)]
    branches = None if args.no_decode else branches_measure(dev)
    # the other workloads of the same layer family, each timed as the headline one (a few steps each)
    others = None
    if not args.no_other_configs:
        del step
        torch.cuda.empty_cache()
        others = {}
        for name, fn, k in (("varlen8", wl.varlen8, 10), ("long_session", wl.long_session, 10),
                            ("small_fp32", wl.small_fp32, 200)):
            others[name] = other_config_measure(name, fn(), dev, k)
            torch.cuda.empty_cache()

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "precision": PRECISION, "data": "synthetic",
            "config": config, "e2e": e2e, "gpu_launches": gpu_launches, "roofline": roofline, "kernels": kernels,
            "clocks": clocks, "state_pass": state_pass, "decode": decode, "branches": branches, "configs": others}

    # --- CPU baseline (oracle), rank 0 at N=1 only ---
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = min(args.cpu_sample_tokens, w.session_lengths[0])
        run = oracle_sample(w, n)
        t0 = time.time()
        run()
        dt = time.time() - t0
        line["cpu_baseline"] = {"value": round(n / dt, 1), "unit": UNIT, "cores": cpu_threads(sh.n_v_heads),
                                "kind": "oracle", "cpu": cpu_model(),
                                "sample": f"first {n} tokens of the {w.session_lengths[0]}-token session, all "
                                          f"{sh.n_v_heads} heads, one fp64 oracle call ({dt:.1f} s)",
                                "one_thread": oracle_one_thread_child()}
    if rank == 0:
        print(json.dumps(line), flush=True)


# the reference arm's whole run (warm-up and timed steps) is sized to take about this long on the host
REFERENCE_BUDGET_S = 120.0


def reference_sample_tokens(n_max: int, steps: int, seconds_per_token: float) -> int:
    """Tokens per step of the reference arm: the first n_max at most, fewer (a multiple of 512, at least 512
    unless n_max is smaller) when steps x n_max would outlast REFERENCE_BUDGET_S at the measured rate."""
    fit = int(REFERENCE_BUDGET_S / (max(steps, 1) * max(seconds_per_token, 1e-12)))
    return min(n_max, max(fit // 512 * 512, min(512, n_max)))


def run_reference(args, w, rank, world):
    """The oracle as the reference arm: rank 0 alone, host cores. Each step runs the oracle over the first
    tokens of the session; their number is set by an untimed probe of the oracle's rate so that the whole
    run stays within a few minutes whatever --steps and --warmup are."""
    if rank != 0:
        return
    n_max = min(args.cpu_sample_tokens, w.session_lengths[0])
    n_probe = min(2048, n_max)
    probe = oracle_sample(w, n_probe)
    probe()                                  # loads the oracle and starts its threads
    t0 = time.time()
    probe()
    n = reference_sample_tokens(n_max, args.steps + args.warmup, (time.time() - t0) / n_probe)
    run = oracle_sample(w, n)
    for _ in range(args.warmup):
        run()
    t0 = time.time()
    for _ in range(args.steps):
        run()
    dt = time.time() - t0
    v = n * args.steps / dt
    sh = w.shape
    cores = cpu_threads(sh.n_v_heads)
    sample = (f"first {n} tokens of the {w.session_lengths[0]}-token session per step, all {sh.n_v_heads} heads, "
              f"fp64 oracle")
    line = {"metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample_tokens_per_step": n, "n_qk_heads": sh.n_qk_heads,
                       "n_v_heads": sh.n_v_heads, "d_k": sh.d_k, "d_v": sh.d_v, "grid_c": sh.grid_c,
                       "parallelism": "host threads over heads"},
            "impl": "reference",
            "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
