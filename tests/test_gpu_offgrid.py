"""Off-grid splits, reported as a tolerance and never compared bit for bit.

A call that starts or ends off the grid ("The shadow reader", section "Exact on
a grid": results equal across calls only at the grid's positions; the page
gives grid 512 against grid 2,048 as max diff 0.44 on a K row and 0.018 on the
recurrent state) moves the 64-token compute blocks, so its rounding differs
from one unsplit call. On the 41,802-token replay session (16 heads, d = 128):

* one partial call over all tokens against the same ids fed as partial calls
  split at off-grid positions;
* a chain of one-token decode steps over the 330-token pending tail against
  one partial prefill of that tail.

Each run is checked against the oracle within the layer tolerance on every head,
and the largest relative L2 difference between the two runs (per v-head, max
over heads) is printed and recorded as a test property.
"""
import numpy as np
import pytest
import torch

from chunked_gated_deltanet_gb300 import gdn
from chunked_gated_deltanet_gb300 import workloads as wl
from helpers import TOL, Runner, oracle_run, out_rel, rel_l2_max

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

OFF_GRID_CUTS = [1000, 7777, 15000, 22222, 33333]   # none is a multiple of 64


def _rel(a: torch.Tensor, b: torch.Tensor, rows: bool) -> float:
    x, y = a.double().cpu().numpy(), b.double().cpu().numpy()
    return out_rel(x, y) if rows else rel_l2_max(x, y)


def test_off_grid_split_tolerance_report(cuda_device, record_property):
    w = wl.qwen08b_replay()
    tok, cw = w.session_tokens(0), w.conv_weights()
    T = len(tok)
    run = Runner(w.shape, tok, cw, cuda_device)
    tol_o, tol_s = TOL[w.shape.dtype]
    assert all(c % 64 for c in OFF_GRID_CUTS)

    # one partial call over every token
    one, o_one = run.session(), run.new_out()
    assert run.prefill(one, 0, T, o_one, gdn.GDN_ALLOW_PARTIAL) == T
    # the same ids as partial calls split off the grid
    split, o_split = run.session(), run.new_out()
    edges = [0] + OFF_GRID_CUTS + [T]
    for a, b in zip(edges[:-1], edges[1:]):
        assert run.prefill(split, a, b, o_split, gdn.GDN_ALLOW_PARTIAL) == b - a
    assert split.committed == one.committed == T
    torch.cuda.synchronize()
    assert torch.equal(split.conv, one.conv)   # the conv state holds raw inputs: exact however the ids are split
    d_out, d_state = _rel(o_split, o_one, True), _rel(split.S, one.S, False)

    # both against the oracle, every head
    o_ref, ST_ref, _ = oracle_run(w.shape, tok, cw)
    r_one = (out_rel(o_one.double().cpu().numpy(), o_ref), rel_l2_max(one.S.double().cpu().numpy(), ST_ref))
    r_split = (out_rel(o_split.double().cpu().numpy(), o_ref), rel_l2_max(split.S.double().cpu().numpy(), ST_ref))
    for r in (r_one, r_split):
        assert r[0] <= tol_o and r[1] <= tol_s, r

    # decode chain over the pending tail against one partial prefill of it, from the committed state
    base = run.session()
    n = run.prefill(base, 0, T, run.new_out())
    assert n == 41_472
    dec, pre = run.session(), run.session()
    gdn.gdn_state_restore(run.desc, dec, base)
    gdn.gdn_state_restore(run.desc, pre, base)
    o_pre = run.new_out()
    assert run.prefill(pre, n, T, o_pre, gdn.GDN_ALLOW_PARTIAL) == T - n
    o_dec = torch.empty_like(o_pre)
    for t in range(n, T):
        xs = [x[t:t + 1] for x in run.x]
        gdn.gdn_decode_step(run.desc, [dec], *xs, run.cw_t, o_dec[t:t + 1])
    assert dec.committed == pre.committed == T
    torch.cuda.synchronize()
    assert torch.equal(dec.conv, pre.conv)
    dd_out, dd_state = _rel(o_dec[n:], o_pre[n:], True), _rel(dec.S, pre.S, False)
    r_dec = (out_rel(o_dec[n:].double().cpu().numpy(), o_ref[n:]), rel_l2_max(dec.S.double().cpu().numpy(), ST_ref))
    assert r_dec[0] <= tol_o and r_dec[1] <= tol_s, r_dec

    report = {
        "split_vs_one_call": {"cuts": OFF_GRID_CUTS, "out_rel_l2_max": d_out, "state_rel_l2_max": d_state},
        "decode_chain_vs_partial_prefill": {"tokens": T - n, "out_rel_l2_max": dd_out, "state_rel_l2_max": dd_state},
        "vs_oracle": {"one_call": r_one, "split": r_split, "decode_chain": r_dec},
    }
    record_property("off_grid_report", report)
    print("off-grid report:", report)
    # a split moves rounding only: the two runs differ by no more than each differs from the oracle allows
    assert d_out <= 2 * tol_o and d_state <= 2 * tol_s
    assert dd_out <= 2 * tol_o and dd_state <= 2 * tol_s
