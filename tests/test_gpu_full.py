"""Full-size workloads through the C ABI: bit-exact structure checks on every
row, and oracle parity on every head of every session (the oracle runs over
groups of v-heads, which is exactly what it computes for the whole layer: heads
are independent, and each group carries the q/k heads it reads).

* Qwen3.5-0.8B-shaped replay: 41,802 tokens in 30 turns, grid 512, held tail;
  replay == fresh bit for bit, then the fork of the bench step; all 16 heads
  against the oracle over every row, the fork's state and the conv state.
* varlen batch of 8 sessions (Hk 16, Hv 32, grid 512) in 6 turn rounds with a
  checkpoint slot per session and round; varlen == solo bit for bit; every
  session's committed rows, final state and conv state against the oracle.
* long session of 100,000 tokens (Hk 16, Hv 32, slow decay) in 6 turns with 6
  slots, then 64 forks of 20..200 question tokens; every fork restores the
  committed state bit for bit and equals a full pass of (session + question);
  all 32 heads against the oracle on the committed session and two forks.
"""
import numpy as np
import pytest
import torch

from chunked_gated_deltanet_gb300 import gdn
from chunked_gated_deltanet_gb300 import workloads as wl
from helpers import TOL, Runner, conv_as_f64, oracle_run, out_rel, rel_l2_max

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _same(a, b):
    torch.cuda.synchronize()
    return torch.equal(a, b)


def _head_groups(sh, size=16):
    """v-heads in groups of `size` (whole GQA groups), so that one oracle call holds a bounded slice of the
    layer while its threads still run one head each."""
    size = max(sh.n_v_heads // sh.n_qk_heads, min(size, sh.n_v_heads))
    return [list(range(a, min(a + size, sh.n_v_heads))) for a in range(0, sh.n_v_heads, size)]


def _parity(shape, tok, cw, out_rows, S_gpu, conv_gpu=None, ST0=None, cs0=None, act=0, q_scale=1.0):
    """Every v-head against the oracle: outputs over every row, the final state, and (given) the conv state,
    which holds raw inputs and must match exactly. Returns the oracle's final state [Hv, dk, dv] and conv
    state [3, ch] over all heads, the starting point of a continuation."""
    import oracle
    tol_o, tol_s = TOL[shape.dtype]
    Hk, Hv, dk, dv = shape.n_qk_heads, shape.n_v_heads, shape.d_k, shape.d_v
    ST_all = np.zeros((Hv, dk, dv))
    cs_all = np.zeros((3, shape.channels))
    nq = Hk * dk
    worst_o = worst_s = 0.0
    for vh in _head_groups(shape):
        o_ref, ST_ref, cs_ref = oracle_run(shape, tok, cw, v_heads=vh, ST0=ST0, conv_state=cs0, act=act,
                                           q_scale=q_scale)
        worst_o = max(worst_o, out_rel(out_rows[:, vh].double().cpu().numpy(), o_ref))
        worst_s = max(worst_s, rel_l2_max(S_gpu[vh].double().cpu().numpy(), ST_ref))
        _, qk_cols, v_cols = oracle.head_columns(Hk, Hv, dk, dv, vh)
        chan = np.concatenate([qk_cols, nq + qk_cols, 2 * nq + v_cols])
        ST_all[vh] = ST_ref
        cs_all[:, chan] = cs_ref
        del o_ref
    assert worst_o <= tol_o, worst_o
    assert worst_s <= tol_s, worst_s
    if conv_gpu is not None:
        assert np.array_equal(conv_as_f64(conv_gpu), cs_all)
    return ST_all, cs_all


def test_qwen08b_replay_full(cuda_device):
    w = wl.qwen08b_replay()
    tok = wl.Tokens.concat([w.session_tokens(0), w.extra_tokens(0, w.fork_questions[0])])
    T = w.session_lengths[0]
    cw = w.conv_weights()
    run = Runner(w.shape, tok, cw, cuda_device)
    o_rep, o_fresh = run.new_out(), run.new_out()
    rep = run.session()
    slots = [run.session() for _ in range(6)]
    end = 0
    for k, n in enumerate(w.turns[0]):
        end += n
        run.prefill(rep, rep.committed, end, o_rep)
        gdn.gdn_state_capture(run.desc, rep, slots[k % 6])
    fresh = run.session()
    n = run.prefill(fresh, 0, T, o_fresh)
    assert rep.committed == fresh.committed == n == 41_472 and T - n == 330
    assert _same(o_rep[:n], o_fresh[:n]) and _same(rep.S, fresh.S) and _same(rep.conv, fresh.conv)
    assert slots[(len(w.turns[0]) - 1) % 6].committed == n
    # the fork of the bench step: 330 pending + 290 question tokens, then restore
    S0, c0 = rep.S.clone(), rep.conv.clone()
    slot = run.session()
    gdn.gdn_state_capture(run.desc, rep, slot)
    assert run.prefill(rep, n, len(tok), o_rep, gdn.GDN_ALLOW_PARTIAL) == len(tok) - n
    S_fork = rep.S.clone()
    gdn.gdn_state_restore(run.desc, rep, slot)
    assert _same(rep.S, S0) and _same(rep.conv, c0) and rep.committed == n
    full = run.session()
    run.prefill(full, 0, len(tok), o_fresh, gdn.GDN_ALLOW_PARTIAL)
    assert _same(o_rep[n:], o_fresh[n:]) and _same(S_fork, full.S)
    # every head against the oracle over every row (committed rows and the fork's), the fork's final state
    # and its conv state
    _parity(w.shape, tok, cw, o_fresh, full.S, full.conv)


def test_varlen8_full(cuda_device):
    w = wl.varlen8()
    sh, cw = w.shape, w.conv_weights()
    C = sh.grid_c
    toks = [w.session_tokens(i) for i in range(8)]
    lens = w.session_lengths
    runs = [Runner(sh, t, cw, cuda_device) for t in toks]
    desc = runs[0].desc
    sess = [r.session() for r in runs]
    slots = [[r.session() for _ in range(6)] for r in runs]
    outs = [r.new_out() for r in runs]
    ends = [0] * 8
    max_round = max(sum(tt[k] for tt in w.turns) + 8 * C for k in range(6))
    ws = gdn.workspace(desc, max_round, 8, cuda_device)
    for r in range(6):
        pieces, cu = [], [0]
        for i in range(8):
            a = sess[i].committed
            ends[i] += w.turns[i][r]
            pieces.append((i, a, ends[i]))
            cu.append(cu[-1] + ends[i] - a)
        cat = lambda j: torch.cat([runs[i].x[j][a:b] for i, a, b in pieces])
        x = [cat(j) for j in range(5)]
        out = torch.empty((cu[-1], sh.n_v_heads, sh.d_v), dtype=torch.float32, device=cuda_device)
        nc = gdn.gdn_prefill_varlen(desc, sess, cu, *x, runs[0].cw_t, out, ws)
        for k, (i, a, b) in enumerate(pieces):
            outs[i][a:a + nc[k]] = out[cu[k]:cu[k] + nc[k]]
            gdn.gdn_state_capture(desc, sess[i], slots[i][r])
    for i in range(8):
        # solo replay with the same turn boundaries and a capture per turn
        s, o = runs[i].session(), runs[i].new_out()
        e = 0
        for r in range(6):
            e += w.turns[i][r]
            runs[i].prefill(s, s.committed, e, o)
            assert slots[i][r].committed == s.committed
            tmp = runs[i].session()
            gdn.gdn_state_capture(desc, s, tmp)
            assert _same(tmp.S, slots[i][r].S) and _same(tmp.conv, slots[i][r].conv)
        n = s.committed
        assert n == (lens[i] // C) * C == sess[i].committed
        assert _same(o[:n], outs[i][:n]) and _same(s.S, sess[i].S) and _same(s.conv, sess[i].conv)
    # fresh single call == replay for the longest session
    i = int(np.argmax(lens))
    f, of = runs[i].session(), runs[i].new_out()
    n = runs[i].prefill(f, 0, lens[i], of)
    assert _same(of[:n], outs[i][:n]) and _same(f.S, sess[i].S)
    # oracle parity: every session's committed rows, final state and conv state, all 32 heads
    for j in range(8):
        n = sess[j].committed
        _parity(sh, toks[j].slice(0, n), cw, outs[j][:n], sess[j].S, sess[j].conv)


def test_long_session_forks_full(cuda_device):
    w = wl.long_session()
    sh, cw = w.shape, w.conv_weights()
    T = w.session_lengths[0]
    Qmax = max(w.fork_questions)
    tok = w.session_tokens(0)
    buf = wl.Tokens.concat([tok, w.extra_tokens(0, Qmax)])      # rows past T are rewritten per fork
    run = Runner(sh, buf, cw, cuda_device)
    run.ws = gdn.workspace(run.desc, T + Qmax + 64, 1, cuda_device)
    desc = run.desc
    sess, out = run.session(), run.new_out()
    slots = [run.session() for _ in range(6)]
    end = 0
    for k, n in enumerate(w.turns[0]):
        end += n
        run.prefill(sess, sess.committed, end, out)
        gdn.gdn_state_capture(desc, sess, slots[k])
    committed = sess.committed
    assert committed == 99_840 and slots[5].committed == committed
    S0, c0 = sess.S.clone(), sess.conv.clone()
    fork_slot = run.session()
    full = run.session()
    of = run.new_out()
    checked = {}
    for j, q in enumerate(w.fork_questions):
        qt = w.extra_tokens(j, q)
        for dst, src in zip(run.x, wl.tokens_to_torch(qt, sh.dtype, cuda_device)):
            dst[T:T + q] = src
        gdn.gdn_state_capture(desc, sess, fork_slot)
        fo = run.new_out(T + q - committed)
        xs = [x[committed:T + q] for x in run.x]
        assert gdn.gdn_prefill_chunks(desc, sess, *xs, run.cw_t, fo, run.ws, flags=gdn.GDN_ALLOW_PARTIAL) == \
            T + q - committed
        S_fork = sess.S.clone()
        gdn.gdn_state_restore(desc, sess, fork_slot)
        assert sess.committed == committed and _same(sess.S, S0) and _same(sess.conv, c0)
        gdn.gdn_session_init(desc, full)
        xs = [x[:T + q] for x in run.x]
        gdn.gdn_prefill_chunks(desc, full, *xs, run.cw_t, of[:T + q], run.ws, flags=gdn.GDN_ALLOW_PARTIAL)
        assert _same(fo, of[committed:T + q]) and _same(S_fork, full.S), j
        if j in (0, 1):
            checked[j] = (qt, fo.clone(), S_fork)
    # oracle parity, all 32 heads: the committed session, then two forks continuing from it
    ST_ref, cs_ref = _parity(sh, tok.slice(0, committed), cw, out[:committed], S0, c0)
    tail = tok.slice(committed, T)
    for j, (qt, fo, S_fork) in checked.items():
        _parity(sh, wl.Tokens.concat([tail, qt]), cw, fo, S_fork, ST0=ST_ref, cs0=cs_ref)


def test_grid_2048_replay_and_grid_independence(cuda_device):
    """Grid 2,048 on the replay tokens: turn-by-turn replay equals a fresh call bit for bit, and, since the
    grid sets only the commit granularity and the 64-token block the arithmetic, both equal the grid-512
    results at the common committed length."""
    w = wl.qwen08b_replay()
    tok, cw = w.session_tokens(0), w.conv_weights()
    sh2048 = wl.Shape(w.shape.n_qk_heads, w.shape.n_v_heads, w.shape.d_k, w.shape.d_v, 2048, w.shape.dtype)
    run = Runner(sh2048, tok, cw, cuda_device)
    o_rep, o_fresh = run.new_out(), run.new_out()
    rep, fresh = run.session(), run.session()
    end = 0
    for n in w.turns[0]:
        end += n
        run.prefill(rep, rep.committed, end, o_rep)
    n = run.prefill(fresh, 0, len(tok), o_fresh)
    assert rep.committed == fresh.committed == n == 20 * 2048
    assert _same(o_rep[:n], o_fresh[:n]) and _same(rep.S, fresh.S) and _same(rep.conv, fresh.conv)
    run512 = Runner(w.shape, tok, cw, cuda_device)
    s512, o512 = run512.session(), run512.new_out()
    assert run512.prefill(s512, 0, n, o512) == n
    assert _same(o512[:n], o_fresh[:n]) and _same(s512.S, fresh.S) and _same(s512.conv, fresh.conv)


def test_silu_and_q_scale_on_the_replay(cuda_device):
    """The replay tokens with the SiLU conv and q scaled by d^-1/2: every head against the oracle."""
    w = wl.qwen08b_replay()
    tok, cw = w.session_tokens(0), w.conv_weights()
    qs = float(w.shape.d_k) ** -0.5
    run = Runner(w.shape, tok, cw, cuda_device, act=gdn.GDN_CONV_SILU, q_scale=qs)
    sess, out = run.session(), run.new_out()
    n = run.prefill(sess, 0, len(tok), out)
    _parity(w.shape, tok.slice(0, n), cw, out[:n], sess.S, sess.conv, act=1, q_scale=qs)
