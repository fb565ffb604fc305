"""Bit-exact GPU-vs-GPU checks of the grid, fork, shared-prefix and batching rules.

* on-grid replay (turn by turn, sub-grid tail held pending) equals a fresh
  prefill on the same grid in every committed output row, the recurrent state
  and the conv state ("The shadow reader", section "Exact on a grid");
* a fork (capture, prefill tail + question with the partial flag, restore)
  leaves the committed state unchanged, and its outputs equal a full pass;
* shared prefixes cut at their last multiple of 64 and continued per branch
  equal a full-prompt pass ("qwen3_5: run prompts that share prefixes once per
  prefix", sections "Purpose" and "Test Plan");
* a session's result does not depend on the other sessions of a varlen call,
  nor on sessions time-shared through checkpoint slots ("Long context and
  sessions", section "Sessions on one engine").
"""
import numpy as np
import pytest
import torch

from chunked_gated_deltanet_gb300 import gdn
from chunked_gated_deltanet_gb300 import workloads as wl
from helpers import TOL, Runner, conv_as_f64, desc_of, oracle_run, out_rel, rel_l2_max

pytestmark = pytest.mark.gpu


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    torch.cuda.synchronize()
    return torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                       b.view(torch.uint8) if b.dtype != torch.uint8 else b)


def _replay(run: Runner, turns, out):
    """Feed turns; each call sends the pending tail plus the turn's tokens."""
    sess = run.session()
    end = 0
    for n in turns:
        end += n
        consumed = run.prefill(sess, sess.committed, end, out)
        assert consumed % run.shape.grid_c == 0
    return sess


@pytest.mark.parametrize("C", [64, 512])
def test_replay_equals_fresh(cuda_device, C):
    shape = wl.Shape(2, 4, 128, 128, C, wl.BF16)
    T = 5000
    w = wl.Workload("replay", shape, seed=1, session_lengths=[T])
    run = Runner(shape, w.session_tokens(0), w.conv_weights(), cuda_device)
    turns = wl.split_turns(T, 9, np.random.default_rng(3))
    o1, o2 = run.new_out(), run.new_out()
    s1 = _replay(run, turns, o1)
    s2 = run.session()
    n = run.prefill(s2, 0, T, o2)
    assert s1.committed == s2.committed == n == (T // C) * C
    assert _same(o1[:n], o2[:n]) and _same(s1.S, s2.S) and _same(s1.conv, s2.conv)


def test_grid64_equals_grid512_at_multiples_of_512(cuda_device):
    T = 3072
    w = wl.Workload("grids", wl.Shape(2, 2, 128, 128, 64, wl.BF16), seed=2, session_lengths=[T])
    tok, cw = w.session_tokens(0), w.conv_weights()
    r64 = Runner(wl.Shape(2, 2, 128, 128, 64, wl.BF16), tok, cw, cuda_device)
    r512 = Runner(wl.Shape(2, 2, 128, 128, 512, wl.BF16), tok, cw, cuda_device)
    o64, o512 = r64.new_out(), r512.new_out()
    s64 = _replay(r64, [700, 64, 1000, 1308], o64)
    s512 = _replay(r512, [1100, 1972], o512)
    assert s64.committed == s512.committed == T
    assert _same(o64, o512) and _same(s64.S, s512.S) and _same(s64.conv, s512.conv)


def test_fork_restores_and_matches_full_pass(cuda_device):
    shape = wl.Shape(2, 4, 128, 128, 512, wl.BF16)
    T, Q = 2700, 150
    w = wl.Workload("fork", shape, seed=4, session_lengths=[T])
    tok, cw = w.session_tokens(0), w.conv_weights()
    full = wl.Tokens.concat([tok, w.extra_tokens(0, Q)])
    run = Runner(shape, full, cw, cuda_device)
    out = run.new_out()
    sess = run.session()
    assert run.prefill(sess, 0, T, out) == 2560
    S0, conv0 = sess.S.clone(), sess.conv.clone()
    slot = run.session()
    gdn.gdn_state_capture(run.desc, sess, slot)
    # fork: pending tail (140) + question (150), partial allowed, then put the state back
    assert run.prefill(sess, 2560, T + Q, out, gdn.GDN_ALLOW_PARTIAL) == T + Q - 2560
    assert sess.committed == T + Q
    with pytest.raises(gdn.GdnError) as e:           # off grid now: on-grid calls are refused
        run.prefill(sess, T + Q, T + Q, out)
    assert e.value.status == gdn.GDN_ERR_OFF_GRID
    gdn.gdn_state_restore(run.desc, sess, slot)
    assert sess.committed == 2560
    assert _same(sess.S, S0) and _same(sess.conv, conv0)
    # full pass of (session + question)
    ref = run.session()
    oref = run.new_out()
    assert run.prefill(ref, 0, T + Q, oref, gdn.GDN_ALLOW_PARTIAL) == T + Q
    assert _same(out, oref)


def test_varlen_equals_solo(cuda_device):
    shape = wl.Shape(2, 4, 128, 128, 512, wl.BF16)
    lens = [1500, 513, 2100, 300]
    w = wl.Workload("vl", shape, seed=6, session_lengths=lens)
    cw = w.conv_weights()
    toks = [w.session_tokens(i) for i in range(len(lens))]
    packed = wl.Tokens.concat(toks)
    cu = np.concatenate([[0], np.cumsum(lens)])
    for flags in (0, gdn.GDN_ALLOW_PARTIAL):
        run = Runner(shape, packed, cw, cuda_device)
        sess = [run.session() for _ in lens]
        out = run.new_out()
        ws = gdn.workspace(run.desc, int(cu[-1]), len(lens), cuda_device)
        nc = gdn.gdn_prefill_varlen(run.desc, sess, cu, *run.x, run.cw_t, out, ws, flags=flags)
        for i, L in enumerate(lens):
            solo = Runner(shape, toks[i], cw, cuda_device)
            s, o = solo.session(), solo.new_out()
            n = solo.prefill(s, 0, L, o, flags)
            assert n == nc[i] == sess[i].committed
            assert _same(out[cu[i]:cu[i] + n], o[:n])
            assert _same(s.S, sess[i].S) and _same(s.conv, sess[i].conv)


def test_varlen_beyond_one_launch_equals_solo(cuda_device):
    """A varlen call over more sessions than one launch takes (64) runs as several launches; every session,
    empty and sub-grid ones included, still equals its own solo call bit for bit."""
    shape = wl.Shape(2, 4, 128, 128, 64, wl.BF16)
    rng = np.random.default_rng(21)
    lens = [int(x) for x in rng.integers(0, 300, size=70)]
    lens[0], lens[5], lens[69] = 0, 40, 64
    w = wl.Workload("vl70", shape, seed=22, session_lengths=[max(l, 1) for l in lens])
    cw = w.conv_weights()
    toks = [w.session_tokens(i).slice(0, L) for i, L in enumerate(lens)]
    cu = np.concatenate([[0], np.cumsum(lens)])
    run = Runner(shape, wl.Tokens.concat(toks), cw, cuda_device)
    ws = gdn.workspace(run.desc, int(cu[-1]), len(lens), cuda_device)
    for flags in (0, gdn.GDN_ALLOW_PARTIAL):
        sess, out = [run.session() for _ in lens], run.new_out()
        nc = gdn.gdn_prefill_varlen(run.desc, sess, cu, *run.x, run.cw_t, out, ws, flags=flags)
        for i, L in enumerate(lens):
            expect = L if flags else L // 64 * 64
            assert nc[i] == sess[i].committed == expect
            if L == 0:
                assert float(sess[i].S.abs().max()) == 0.0
                continue
            solo = Runner(shape, toks[i], cw, cuda_device)
            s, o = solo.session(), solo.new_out()
            assert solo.prefill(s, 0, L, o, flags) == expect
            assert _same(out[cu[i]:cu[i] + expect], o[:expect])
            assert _same(s.S, sess[i].S) and _same(s.conv, sess[i].conv)


def test_two_part_call_equals_one_part_calls(cuda_device):
    """A one-session call whose prologue would end in a partial round of SMs runs in two parts (the last
    blocks' prologue beside the first blocks' state pass). With 16 q/k heads a 48- or 50-block call takes
    that path on a 152-SM GPU; a varlen call of two sessions and 16-block calls do not. All give the same
    bits, on grid with its checkpoint and with a partial final block."""
    shape = wl.Shape(16, 16, 128, 128, 512, wl.BF16)
    T = 3172                                     # 3,072 on grid + a 100-token tail
    w = wl.Workload("twopart", shape, seed=12, session_lengths=[T])
    tok, cw = w.session_tokens(0), w.conv_weights()
    run = Runner(shape, tok, cw, cuda_device)
    pair = Runner(shape, wl.Tokens.concat([tok, tok]), cw, cuda_device)
    ws2 = gdn.workspace(pair.desc, 2 * T, 2, cuda_device)
    for flags in (0, gdn.GDN_ALLOW_PARTIAL):
        # one call (two parts where the GPU has 152 SMs), its checkpoint written by the call
        s1, slot1, o1 = run.session(), run.session(), run.new_out()
        n1 = gdn.gdn_prefill_chunks_checkpoint(run.desc, s1, slot1, *run.x, run.cw_t, o1, run.ws, flags=flags)
        assert n1 == (T if flags else 3072) == s1.committed == slot1.committed
        # the same tokens as two sessions of one varlen call (never split)
        sv, ov = [pair.session(), pair.session()], pair.new_out()
        nv = gdn.gdn_prefill_varlen(pair.desc, sv, [0, T, 2 * T], *pair.x, pair.cw_t, ov, ws2, flags=flags)
        assert nv == [n1, n1]
        for i, s in enumerate(sv):
            assert _same(ov[i * T:i * T + n1], o1[:n1]) and _same(s.S, s1.S) and _same(s.conv, s1.conv)
        assert _same(slot1.S, s1.S) and _same(slot1.conv, s1.conv)
    # on grid: three 16-block calls (one part each) reach the same state and outputs
    s3, o3 = run.session(), run.new_out()
    for a in (0, 1024, 2048):
        assert run.prefill(s3, a, a + 1024, o3) == 1024
    s4, o4 = run.session(), run.new_out()
    assert run.prefill(s4, 0, T, o4) == 3072
    assert _same(o3[:3072], o4[:3072]) and _same(s3.S, s4.S) and _same(s3.conv, s4.conv)


def test_interleaved_sessions_through_slots(cuda_device):
    """One working session time-shared by 3 conversations through slots equals uninterrupted runs."""
    shape = wl.Shape(2, 2, 128, 128, 64, wl.BF16)
    lens = [900, 700, 1000]
    w = wl.Workload("inter", shape, seed=8, session_lengths=lens)
    cw = w.conv_weights()
    runs = [Runner(shape, w.session_tokens(i), cw, cuda_device) for i in range(3)]
    turns = [wl.split_turns(L, 4, np.random.default_rng(10 + i)) for i, L in enumerate(lens)]
    work = runs[0].session()
    slots = [runs[0].session() for _ in range(3)]
    outs = [r.new_out() for r in runs]
    ends = [0, 0, 0]
    for k in range(4):
        for i in range(3):
            gdn.gdn_state_restore(runs[i].desc, work, slots[i])
            ends[i] += turns[i][k]
            runs[i].prefill(work, work.committed, ends[i], outs[i])
            gdn.gdn_state_capture(runs[i].desc, work, slots[i])
    for i in range(3):
        s, o = runs[i].session(), runs[i].new_out()
        n = runs[i].prefill(s, 0, lens[i], o)
        assert slots[i].committed == n
        assert _same(outs[i][:n], o[:n]) and _same(slots[i].S, s.S) and _same(slots[i].conv, s.conv)


def test_refused_requests_change_nothing(cuda_device):
    shape = wl.Shape(2, 2, 128, 128, 512, wl.BF16)
    w = wl.Workload("refuse", shape, seed=12, session_lengths=[2048])
    run = Runner(shape, w.session_tokens(0), w.conv_weights(), cuda_device)
    a, b = run.session(), run.session()
    oa, ob = run.new_out(), run.new_out()
    run.prefill(a, 0, 1024, oa)
    run.prefill(b, 0, 1024, ob)
    S_before = b.S.clone()
    small_ws = torch.empty(1024, dtype=torch.uint8, device=cuda_device)
    xq, xk, xv, g, beta = (t[1024:] for t in run.x)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill_chunks(run.desc, b, xq, xk, xv, g, beta, run.cw_t, ob[1024:], small_ws)
    assert e.value.status == gdn.GDN_ERR_WORKSPACE
    other = desc_of(wl.Shape(2, 2, 128, 128, 64, wl.BF16))
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill_chunks(other, b, xq, xk, xv, g, beta, run.cw_t, ob[1024:], run.ws)
    assert e.value.status == gdn.GDN_ERR_STATE_MISMATCH
    assert b.committed == 1024 and _same(b.S, S_before)
    run.prefill(a, 1024, 2048, oa)
    run.prefill(b, 1024, 2048, ob)
    assert _same(oa, ob) and _same(a.S, b.S) and _same(a.conv, b.conv)


def _shared_prefix_run(w: wl.Workload, cw, device, reverse=False):
    """Prefix runs once to its last multiple of 64; groups and branches continue from captured states."""
    shape = w.shape
    R = w.request_prefix
    req = w.session_tokens(0, R)
    groups = [w.extra_tokens(g, gp) for g, gp in enumerate(w.group_prefixes)]
    res = {}
    full_tok = wl.Tokens.concat([req] + groups + [w.extra_tokens(100 + 4 * g + b, n)
                                                  for g, br in enumerate(w.branches) for b, n in enumerate(br)])
    run = Runner(shape, full_tok, cw, device)
    desc = run.desc
    cut = wl.grid_floor(R, 64)
    prefix_sess, prefix_slot = run.session(), run.session()
    scratch = run.new_out(R)
    xs = lambda toks: wl.tokens_to_torch(toks, shape.dtype, device)

    def feed(sess, toks, a, b, out, flags):
        x = xs(toks.slice(a, b))
        return gdn.gdn_prefill_chunks(desc, sess, *x, run.cw_t, out, run.ws, flags=flags)

    assert feed(prefix_sess, req, 0, cut, scratch, 0) == cut
    gdn.gdn_state_capture(desc, prefix_sess, prefix_slot)
    slot_copy = prefix_slot.S.clone()
    g_order = list(range(len(w.group_prefixes)))
    if reverse:
        g_order.reverse()
    work = run.session()
    for g in g_order:
        gp = w.group_prefixes[g]
        prompt = wl.Tokens.concat([req, groups[g]])
        gcut = wl.grid_floor(R + gp, 64)
        gslot = run.session()
        gdn.gdn_state_restore(desc, work, prefix_slot)
        if gcut > cut:
            assert feed(work, prompt, cut, gcut, run.new_out(gcut - cut), 0) == gcut - cut
        gdn.gdn_state_capture(desc, work, gslot)
        b_order = list(range(len(w.branches[g])))
        if reverse:
            b_order.reverse()
        for b in b_order:
            n = w.branches[g][b]
            bt = wl.Tokens.concat([prompt, w.extra_tokens(100 + 4 * g + b, n)])
            gdn.gdn_state_restore(desc, work, gslot)
            ob = run.new_out(len(bt) - gcut)
            assert feed(work, bt, gcut, len(bt), ob, gdn.GDN_ALLOW_PARTIAL) == len(bt) - gcut
            res[(g, b)] = (bt, gcut, ob, work.S.clone(), work.conv.clone())
    assert _same(prefix_slot.S, slot_copy) and prefix_slot.committed == cut
    return run, res


def test_shared_prefix_branches_equal_full_pass(cuda_device):
    """Request prefix 1,000; groups 0/1/70/128; 4 branches each; grid 64."""
    w = wl.shared_prefix()
    cw = w.conv_weights()
    run, res = _shared_prefix_run(w, cw, cuda_device)
    assert len(res) == 16
    for (g, b), (bt, gcut, ob, S, conv) in res.items():
        x = wl.tokens_to_torch(bt, w.shape.dtype, cuda_device)
        sess = run.session()
        of = run.new_out(len(bt))
        assert gdn.gdn_prefill_chunks(run.desc, sess, *x, run.cw_t, of, run.ws, flags=gdn.GDN_ALLOW_PARTIAL) == len(bt)
        assert _same(ob, of[gcut:]), (g, b)
        assert _same(S, sess.S) and _same(conv, sess.conv)
    # state isolation: groups and branches reversed give the same results
    _, res2 = _shared_prefix_run(w, cw, cuda_device, reverse=True)
    for k, v in res.items():
        assert _same(v[2], res2[k][2]) and _same(v[3], res2[k][3])


def test_shared_prefix_branches_match_oracle(cuda_device):
    """The shared-prefix workload's own data (request prefix 1,000 cut to 960; groups 0/1/70/128; 4 branches
    each; grid 64; 16 heads, d = 128) against the oracle: each branch's outputs from its cut onward, its
    final state and its conv state, every head, against one oracle pass over the branch's full prompt."""
    w = wl.shared_prefix()
    cw = w.conv_weights()
    _, res = _shared_prefix_run(w, cw, cuda_device)
    tol_o, tol_s = TOL[w.shape.dtype]
    assert len(res) == 16
    for (g, b), (bt, gcut, ob, S, conv) in res.items():
        o_ref, ST_ref, cs_ref = oracle_run(w.shape, bt, cw)
        r_o = out_rel(ob.double().cpu().numpy(), o_ref[gcut:])
        r_s = rel_l2_max(S.double().cpu().numpy(), ST_ref)
        assert r_o <= tol_o and r_s <= tol_s, ((g, b), r_o, r_s)
        assert np.array_equal(conv_as_f64(conv), cs_ref), (g, b)


def test_branches_in_one_call_equal_restore_and_prefill(cuda_device):
    """All branches of a group in one gdn_prefill_branches call, reading the group's state in place, equal
    the restore-then-prefill results bit for bit; an empty branch becomes a copy of the prefix, which is
    left unchanged."""
    w = wl.shared_prefix()
    cw = w.conv_weights()
    run, res = _shared_prefix_run(w, cw, cuda_device)
    desc, shape = run.desc, w.shape
    R, cut = w.request_prefix, wl.grid_floor(w.request_prefix, 64)
    req = w.session_tokens(0, R)
    xs = lambda toks: wl.tokens_to_torch(toks, shape.dtype, cuda_device)
    for g, gp in enumerate(w.group_prefixes):
        prompt = wl.Tokens.concat([req, w.extra_tokens(g, gp)])
        gcut = wl.grid_floor(R + gp, 64)
        gstate = run.session()
        x = xs(prompt.slice(0, gcut))
        assert gdn.gdn_prefill_chunks(desc, gstate, *x, run.cw_t, run.new_out(gcut), run.ws) == gcut
        S_before, conv_before = gstate.S.clone(), gstate.conv.clone()
        tails = [res[(g, b)][0].slice(gcut, len(res[(g, b)][0])) for b in range(len(w.branches[g]))]
        tails.append(prompt.slice(gcut, gcut))   # an empty branch
        cu = [0]
        for t in tails:
            cu.append(cu[-1] + len(t))
        packed = xs(wl.Tokens.concat(tails))
        out = torch.full((cu[-1], shape.n_v_heads, shape.d_v), float("nan"), device=cuda_device)
        branches = [run.session() for _ in tails]
        ws = gdn.workspace(desc, cu[-1] + 64 * len(tails), len(tails), cuda_device)
        n = gdn.gdn_prefill_branches(desc, gstate, branches, cu, *packed, run.cw_t, out, ws,
                                     flags=gdn.GDN_ALLOW_PARTIAL)
        assert n == [len(t) for t in tails]
        torch.cuda.synchronize()
        for b in range(len(tails) - 1):
            bt, bcut, ob, S, conv = res[(g, b)]
            assert bcut == gcut
            assert _same(out[cu[b]:cu[b + 1]], ob), (g, b)
            assert _same(branches[b].S, S) and _same(branches[b].conv, conv), (g, b)
            assert branches[b].committed == len(bt)
        empty = branches[-1]
        assert empty.committed == gcut and _same(empty.S, S_before) and _same(empty.conv, conv_before)
        assert _same(gstate.S, S_before) and _same(gstate.conv, conv_before) and gstate.committed == gcut


@pytest.mark.parametrize("dtype,d", [(wl.BF16, 128), (wl.BF16, 64), (wl.FP32, 64)])
def test_checkpointing_prefill_equals_prefill_then_capture(cuda_device, dtype, d):
    """gdn_prefill_chunks_checkpoint writes into its slot exactly what a capture after the call would, and
    leaves the session as gdn_prefill_chunks does; a call with nothing to commit checkpoints the unchanged
    state; the varlen form does the same per session."""
    shape = wl.Shape(2, 4, d, d, 128, dtype)
    w = wl.Workload("ckpt", shape, seed=51, session_lengths=[700])
    run = Runner(shape, w.session_tokens(0), w.conv_weights(), cuda_device)
    a, b = run.session(), run.session()
    sa, sb = run.session(), run.session()
    oa, ob = run.new_out(), run.new_out()
    for lo, hi in ((0, 300), (256, 600), (512, 600)):      # the last call commits nothing
        x = [t[lo:hi] for t in run.x]
        na = gdn.gdn_prefill_chunks(run.desc, a, *x, run.cw_t, oa[lo:hi], run.ws)
        gdn.gdn_state_capture(run.desc, a, sa)
        nb = gdn.gdn_prefill_chunks_checkpoint(run.desc, b, sb, *x, run.cw_t, ob[lo:hi], run.ws)
        assert na == nb and a.committed == b.committed == sa.committed == sb.committed
        assert sb.tag == sa.tag == a.tag
        assert _same(oa, ob) and _same(a.S, b.S) and _same(a.conv, b.conv)
        assert _same(sa.S, sb.S) and _same(sa.conv, sb.conv)
    # varlen: three sessions, one checkpoint each
    runs = [Runner(shape, wl.Workload("ckv", shape, seed=60 + i, session_lengths=[300 + 100 * i]).session_tokens(0),
                   run.cw, cuda_device) for i in range(3)]
    toks = [r.tok for r in runs]
    cu = np.cumsum([0] + [len(t) for t in toks]).tolist()
    x = wl.tokens_to_torch(wl.Tokens.concat(toks), dtype, cuda_device)
    ws = gdn.workspace(run.desc, cu[-1] + 64 * 3, 3, cuda_device)
    ses, slots = [run.session() for _ in range(3)], [run.session() for _ in range(3)]
    out = torch.zeros((cu[-1], shape.n_v_heads, d), device=cuda_device)
    gdn.gdn_prefill_varlen_checkpoint(run.desc, ses, slots, cu, *x, run.cw_t, out, ws)
    ref = [run.session() for _ in range(3)]
    out2 = torch.zeros_like(out)
    gdn.gdn_prefill_varlen(run.desc, ref, cu, *x, run.cw_t, out2, ws)
    assert _same(out, out2)
    for s, sl, r in zip(ses, slots, ref):
        assert sl.committed == s.committed == r.committed
        assert _same(s.S, r.S) and _same(sl.S, r.S) and _same(sl.conv, r.conv)


@pytest.mark.parametrize("n_sess", [3, 5])
def test_state_kernel_slice_width_does_not_change_results(cuda_device, n_sess):
    """The state kernel takes d_v in slices of 32, 64 or 128 columns per CTA depending on how many chains a
    launch holds (16 v-heads of d = 128: one session 32; three sessions 64; five 128). Every element's
    arithmetic is the same in each width, so a varlen call of several sessions equals each session alone bit
    for bit."""
    shape = wl.Shape(16, 16, 128, 128, 64, wl.BF16)
    runs = [Runner(shape, wl.Workload("width", shape, seed=70 + i, session_lengths=[300 + 190 * i]).session_tokens(0),
                   wl.Workload("width", shape, seed=70).conv_weights(), cuda_device) for i in range(n_sess)]
    toks = [r.tok for r in runs]
    cu = np.cumsum([0] + [len(t) for t in toks]).tolist()
    x = wl.tokens_to_torch(wl.Tokens.concat(toks), shape.dtype, cuda_device)
    ws = gdn.workspace(runs[0].desc, cu[-1] + 64 * n_sess, n_sess, cuda_device)
    both = [runs[0].session() for _ in range(n_sess)]
    out = torch.zeros((cu[-1], shape.n_v_heads, shape.d_v), device=cuda_device)
    gdn.gdn_prefill_varlen(runs[0].desc, both, cu, *x, runs[0].cw_t, out, ws, flags=gdn.GDN_ALLOW_PARTIAL)
    for i, r in enumerate(runs):
        solo, o = r.session(), r.new_out()
        assert r.prefill(solo, 0, len(r.tok), o, gdn.GDN_ALLOW_PARTIAL) == len(r.tok)
        assert _same(out[cu[i]:cu[i + 1]], o), i
        assert _same(both[i].S, solo.S) and _same(both[i].conv, solo.conv), i
