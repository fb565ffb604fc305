"""Host-side logic of bench.py (no GPU): the multi-rank reduction over gloo
(world size 2) and the reference arm's JSON line, alone and under torchrun."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=2)
    ms, units = bench.reduce_max_sum(10.0 + rank * 5.0, 100.0 * (rank + 1))
    bench.barrier()
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_reduce_max_sum_two_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 15.0, 300.0), (1, 15.0, 300.0)]


def _check_reference_line(line):
    d = json.loads(line)
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["higher_is_better"] is True and d["steps"] == 1


def test_reference_arm_json():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--cpu-sample-tokens", "64"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    _check_reference_line(lines[0])


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
                        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "0",
                        "--gpus", "2", "--cpu-sample-tokens", "64"],
                       capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    _check_reference_line(lines[0])


def test_reference_sample_fits_the_time_budget():
    """The reference arm shrinks its per-step sample (multiples of 512) so that warm-up + timed steps stay
    within its budget at the measured oracle rate, and never grows it past the requested sample."""
    sys.path.insert(0, ROOT)
    import bench
    rate = 2.4 / 41472                       # seconds per token of the whole-layer oracle on 16 cores
    n = bench.reference_sample_tokens(41472, 103, rate)
    assert n % 512 == 0 and 512 <= n < 41472
    assert 103 * n * rate <= bench.REFERENCE_BUDGET_S
    assert bench.reference_sample_tokens(41472, 6, rate) == 41472
    assert bench.reference_sample_tokens(64, 1, 1.0) == 64
    assert bench.reference_sample_tokens(41472, 10**6, rate) == 512
