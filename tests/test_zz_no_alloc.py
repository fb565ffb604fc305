"""The no-allocation prefill (gdn_prefill_chunks_noalloc) against the regular one.

This call serves callers that cannot allocate device memory: code whose memory
a host framework plans once up front, and latency-critical code that must not
call cudaMalloc / cudaFree (they can synchronise the device). Its scratch is a
fixed array inside the library. These checks call it through the C ABI several
times in a row on one session (each call reuses the scratch the one before it
left behind) and compare each call's outputs, the session state and the conv
state with gdn_prefill_chunks on a twin session. The two run the same kernels
on the same inputs, so they must agree bit for bit; the parity tolerance is
checked as well. The last call starts off the 64-token grid and is as long as
the built-in scratch allows. A call that needs more than the built-in scratch
is refused before any device work.

This file is collected last so that a stop at the first failure has already
run every other test.
"""
import numpy as np
import pytest
import torch

from chunked_gated_deltanet_gb300 import gdn
from chunked_gated_deltanet_gb300 import workloads as wl
from helpers import TOL, Runner, out_rel, rel_l2_max

pytestmark = pytest.mark.gpu


def _longest_call(desc) -> int:
    """The most tokens one partial call may process within the built-in scratch."""
    lo, hi = 0, 1 << 20
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if gdn.gdn_workspace_size(desc, mid, 1) <= gdn.GDN_NOALLOC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_noalloc_matches_workspace_prefill_bit_for_bit(cuda_device):
    shape = wl.Shape(2, 4, 128, 128, 64, wl.BF16)
    T1, T2 = 1000, 740           # first call on grid (consumes 960), second partial (ends off grid at 1,700)
    desc = gdn.make_desc(2, 4, 128, 128, 64)
    T3 = _longest_call(desc)     # third call: from 1,700 (off grid), the longest the scratch allows
    assert T3 >= 64 and gdn.gdn_workspace_size(desc, T3 + 1, 1) > gdn.GDN_NOALLOC_SCRATCH_BYTES
    w = wl.Workload("noalloc", shape, seed=31, session_lengths=[T1 + T2 + T3])
    tok, cw = w.session_tokens(0), w.conv_weights()
    run = Runner(shape, tok, cw, cuda_device)
    a, b = run.session(), run.session()
    oa, ob = run.new_out(), run.new_out()
    tol_o, tol_s = TOL[wl.BF16]

    def noalloc(sess, lo, hi, out, flags):
        xq, xk, xv, g, beta = (x[lo:hi] for x in run.x)
        return gdn.gdn_prefill_chunks_noalloc(run.desc, sess, xq, xk, xv, g, beta, run.cw_t, out[lo:hi],
                                              flags=flags)

    def agree(n):
        torch.cuda.synchronize()
        assert torch.equal(oa[:n], ob[:n])
        assert torch.equal(a.S, b.S) and torch.equal(a.conv, b.conv)
        assert np.isfinite(oa[:n].double().cpu().numpy()).all()
        assert out_rel(oa[:n].double().cpu().numpy(), ob[:n].double().cpu().numpy()) <= tol_o
        assert rel_l2_max(a.S.double().cpu().numpy(), b.S.double().cpu().numpy()) <= tol_s

    # call 1: on grid
    n1 = noalloc(a, 0, T1, oa, 0)
    m1 = run.prefill(b, 0, T1, ob, 0)
    assert n1 == m1 == 960 and a.committed == b.committed == 960
    agree(960)
    # call 2: pending tail + more, partial allowed: the session ends off grid
    n2 = noalloc(a, 960, T1 + T2, oa, gdn.GDN_ALLOW_PARTIAL)
    m2 = run.prefill(b, 960, T1 + T2, ob, gdn.GDN_ALLOW_PARTIAL)
    assert n2 == m2 == T1 + T2 - 960 and a.committed == b.committed == T1 + T2
    assert (T1 + T2) % 64 != 0
    agree(T1 + T2)
    # call 3: starts off grid, as long as the scratch allows (its blocks count from the call's first token)
    n3 = noalloc(a, T1 + T2, T1 + T2 + T3, oa, gdn.GDN_ALLOW_PARTIAL)
    m3 = run.prefill(b, T1 + T2, T1 + T2 + T3, ob, gdn.GDN_ALLOW_PARTIAL)
    assert n3 == m3 == T3 and a.committed == b.committed == T1 + T2 + T3
    agree(T1 + T2 + T3)


def test_noalloc_refuses_calls_beyond_its_scratch(cuda_device):
    shape = wl.Shape(16, 16, 128, 128, 512, wl.BF16)
    desc = gdn.make_desc(16, 16, 128, 128, 512)
    T = (_longest_call(desc) // 512 + 1) * 512   # the first whole-grid call beyond the built-in scratch
    need = gdn.gdn_workspace_size(desc, T, 1)
    assert need > gdn.GDN_NOALLOC_SCRATCH_BYTES
    sess = gdn.Session(desc, cuda_device)
    xqk = torch.zeros((T, 16 * 128), dtype=torch.bfloat16, device=cuda_device)
    xv = torch.zeros((T, 16 * 128), dtype=torch.bfloat16, device=cuda_device)
    gb = torch.zeros((T, 16), dtype=torch.float32, device=cuda_device)
    out = torch.zeros((T, 16, 128), dtype=torch.float32, device=cuda_device)
    cw = torch.zeros((shape.channels, 4), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill_chunks_noalloc(desc, sess, xqk, xqk, xv, gb, gb, cw, out)
    assert e.value.status == gdn.GDN_ERR_WORKSPACE
    assert "built-in" in str(e.value)
    assert sess.committed == 0
