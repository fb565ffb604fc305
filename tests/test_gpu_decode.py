"""The batched decode step: CUDA-graph capture and replay, and batch forms.

A decode step reads its inputs from caller buffers and the states through
the sessions' fixed device addresses, allocates nothing and never waits on
the host, so a step can be captured once in a CUDA graph and replayed with
new inputs copied into the same buffers. Replays must give bit for bit what
eager calls give. (A replay advances the device state only; the host-side
committed count moves with the calls the host makes.)
"""
import pytest
import torch

from chunked_gated_deltanet_gb300 import gdn
from chunked_gated_deltanet_gb300 import workloads as wl
from helpers import Runner, oracle_run, out_rel, rel_l2_max, TOL

pytestmark = pytest.mark.gpu

STEPS = 5


def _prefilled(shape, n_sess, cuda_device, seed):
    runs, sessA, sessB = [], [], []
    for i in range(n_sess):
        w = wl.Workload("dgraph", shape, seed=seed + i, session_lengths=[shape.grid_c + STEPS])
        run = Runner(shape, w.session_tokens(0), w.conv_weights() if i == 0 else runs[0].cw, cuda_device)
        runs.append(run)
        for lst in (sessA, sessB):
            s, o = run.session(), run.new_out()
            assert run.prefill(s, 0, shape.grid_c, o) == shape.grid_c
            lst.append(s)
    return runs, sessA, sessB


@pytest.mark.parametrize("d", [64, 128])
def test_graph_replay_matches_eager(cuda_device, d):
    shape = wl.Shape(2, 4, d, d, 64, wl.BF16)
    runs, sessA, sessB = _prefilled(shape, 3, cuda_device, seed=70 + d)
    T0 = shape.grid_c
    step_in = lambda j, t: torch.cat([r.x[j][t:t + 1] for r in runs])
    # eager steps on A
    outA = []
    for k in range(STEPS):
        o = torch.empty((3, shape.n_v_heads, d), device=cuda_device)
        gdn.gdn_decode_step(runs[0].desc, sessA, *(step_in(j, T0 + k) for j in range(5)), runs[0].cw_t, o)
        outA.append(o)
    # one captured step on B, replayed with each step's inputs copied into the static buffers
    static_in = [step_in(j, T0).clone() for j in range(5)]
    static_out = torch.empty((3, shape.n_v_heads, d), device=cuda_device)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.gdn_decode_step(runs[0].desc, sessB, *static_in, runs[0].cw_t, static_out)
    for k in range(STEPS):
        for j in range(5):
            static_in[j].copy_(step_in(j, T0 + k))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(static_out, outA[k]), f"step {k}: replay differs from the eager call"
    for a, b in zip(sessA, sessB):
        assert torch.equal(a.S, b.S) and torch.equal(a.conv, b.conv)
    # and the replayed states are the layer's (oracle, after prefill + STEPS decode steps)
    for i, r in enumerate(runs):
        o_ref, ST_ref, cs_ref = oracle_run(shape, r.tok.slice(0, T0 + STEPS), r.cw)
        tol_o, tol_s = TOL[wl.BF16]
        assert rel_l2_max(sessB[i].S.double().cpu().numpy(), ST_ref) <= tol_s
        got = torch.stack([outA[k][i] for k in range(STEPS)]).double().cpu().numpy()
        assert out_rel(got, o_ref[T0:T0 + STEPS]) <= tol_o


def test_decode_one_session_many_heads_equals_batch_of_one(cuda_device):
    """A 16-head session decoded alone equals the same session inside a batch of 4, bit for bit."""
    shape = wl.Shape(16, 16, 128, 128, 64, wl.BF16)
    runs, sessA, sessB = _prefilled(shape, 4, cuda_device, seed=90)
    T0 = shape.grid_c
    step_in = lambda j, t: torch.cat([r.x[j][t:t + 1] for r in runs])
    ob = torch.empty((4, 16, 128), device=cuda_device)
    gdn.gdn_decode_step(runs[0].desc, sessB, *(step_in(j, T0) for j in range(5)), runs[0].cw_t, ob)
    oa = torch.empty((1, 16, 128), device=cuda_device)
    gdn.gdn_decode_step(runs[0].desc, [sessA[2]], *(runs[2].x[j][T0:T0 + 1] for j in range(5)), runs[0].cw_t, oa)
    torch.cuda.synchronize()
    assert torch.equal(oa[0], ob[2])
    assert torch.equal(sessA[2].S, sessB[2].S) and torch.equal(sessA[2].conv, sessB[2].conv)


def test_decode_over_several_launches_equals_single_steps(cuda_device):
    """A decode call over 150 sessions runs as three launches of at most 64 sessions, each letting the next
    start early; over two consecutive steps (the second reads the states the first wrote) every session's
    output, state and conv state equal those of single-session calls, bit for bit."""
    dev = cuda_device
    desc = gdn.make_desc(2, 4, 64, 64, 64, gdn.GDN_BF16, gdn.GDN_FP32)
    n, nq, nv = 150, 2 * 64, 4 * 64
    gen = torch.Generator(device=dev).manual_seed(11)
    bf = lambda *shape: torch.randn(*shape, generator=gen, device=dev).to(torch.bfloat16)
    batch = [gdn.Session(desc, dev) for _ in range(n)]
    single = [gdn.Session(desc, dev) for _ in range(n)]
    for a, b in zip(batch, single):
        a.S.copy_(0.1 * torch.randn(a.S.shape, generator=gen, device=dev))
        a.conv.copy_(bf(*a.conv.shape))
        b.S.copy_(a.S)
        b.conv.copy_(a.conv)
    cw = bf(2 * nq + nv, 4)
    for _ in range(2):
        xq, xk, xv = bf(n, nq), bf(n, nq), bf(n, nv)
        g = -0.1 * torch.nn.functional.softplus(torch.randn(n, 4, generator=gen, device=dev))
        beta = torch.sigmoid(torch.randn(n, 4, generator=gen, device=dev))
        out_b = torch.zeros((n, 4, 64), device=dev)
        gdn.gdn_decode_step(desc, batch, xq, xk, xv, g, beta, cw, out_b)
        out_s = torch.zeros((n, 4, 64), device=dev)
        for i in range(n):
            gdn.gdn_decode_step(desc, [single[i]], xq[i:i + 1], xk[i:i + 1], xv[i:i + 1], g[i:i + 1], beta[i:i + 1],
                                cw, out_s[i:i + 1])
        torch.cuda.synchronize()
        assert torch.equal(out_b, out_s)
    for a, b in zip(batch, single):
        assert torch.equal(a.S, b.S) and torch.equal(a.conv, b.conv)
        assert a.committed == b.committed == 2
