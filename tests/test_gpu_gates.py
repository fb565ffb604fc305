"""The raw-gate variant on the GPU: g and beta computed from raw projections
by gdn_gates against the oracle's fp64 version, and a prefill fed with them
against the oracle layer fed with the oracle's gates."""
import numpy as np
import pytest
import torch

import oracle
from chunked_gated_deltanet_gb300 import gdn
from chunked_gated_deltanet_gb300 import workloads as wl
from helpers import Runner, oracle_run, out_rel, rel_l2_max, TOL

pytestmark = pytest.mark.gpu


def test_gates_match_oracle(cuda_device):
    a, b, A_log, dt_bias = wl.draw_raw_gates(3000, 16, seed=4)
    a[:8] = [[60.0], [-60.0], [20.0], [-20.0], [0.0], [1e-3], [-1e-3], [7.5]]   # both tails of softplus
    desc = gdn.make_desc(16, 16, 128, 128, 64)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(cuda_device)
    g, beta = torch.empty((3000, 16), device=cuda_device), torch.empty((3000, 16), device=cuda_device)
    gdn.gdn_gates(desc, t(a), t(b), t(A_log), t(dt_bias), g, beta)
    torch.cuda.synchronize()
    g_ref, beta_ref = oracle.gates(a.astype(np.float64), b.astype(np.float64), A_log.astype(np.float64),
                                   dt_bias.astype(np.float64))
    gg, bb = g.double().cpu().numpy(), beta.double().cpu().numpy()
    assert np.all(np.isfinite(gg)) and np.all(gg < 0) and np.all((bb > 0) & (bb < 1))
    # fp32 exp / log1p: a few ulp; and x = a + dt_bias rounded to fp32 (half an ulp of x), which moves
    # softplus(x) ~ e^x by a relative |x| * 2^-24 where x is very negative
    x = np.abs(a.astype(np.float64) + dt_bias.astype(np.float64)[None, :])
    assert np.all(np.abs(gg - g_ref) / np.abs(g_ref) <= 1e-6 + 1.2e-7 * x)
    assert np.max(np.abs(bb - beta_ref) / beta_ref) < 1e-6


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_with_raw_gates_matches_oracle(cuda_device, d):
    shape = wl.Shape(2, 4, d, d, 64, wl.BF16)
    T = 700
    w = wl.Workload("rawg", shape, seed=12, session_lengths=[T])
    tok = w.session_tokens(0)
    a, b, A_log, dt_bias = wl.draw_raw_gates(T, shape.n_v_heads, seed=12)
    run = Runner(shape, tok, w.conv_weights(), cuda_device)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(cuda_device)
    g, beta = run.x[3], run.x[4]          # the drawn gates are replaced by the computed ones
    gdn.gdn_gates(run.desc, t(a), t(b), t(A_log), t(dt_bias), g, beta)
    s, out = run.session(), run.new_out()
    assert run.prefill(s, 0, T, out, gdn.GDN_ALLOW_PARTIAL) == T
    torch.cuda.synchronize()
    g_ref, beta_ref = oracle.gates(a.astype(np.float64), b.astype(np.float64), A_log.astype(np.float64),
                                   dt_bias.astype(np.float64))
    tok_ref = wl.Tokens(tok.xq, tok.xk, tok.xv, g_ref, beta_ref)
    o_ref, ST_ref, _ = oracle_run(shape, tok_ref, run.cw)
    tol_o, tol_s = TOL[wl.BF16]
    assert out_rel(out.double().cpu().numpy(), o_ref) <= tol_o
    assert rel_l2_max(s.S.double().cpu().numpy(), ST_ref) <= tol_s
