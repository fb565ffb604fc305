"""GPU parity against the fp64 oracle, element by element, through the C ABI.

Tolerance (relative L2 per v-head, max over heads): outputs 2e-3 and final
fp32 state 1e-3 for bf16 inputs; 1e-5 for both with fp32 inputs. The conv
state holds raw inputs, so it is compared bit for bit.
"""
import numpy as np
import pytest
import torch

from chunked_gated_deltanet_gb300 import gdn
from chunked_gated_deltanet_gb300 import workloads as wl
from helpers import TOL, Runner, conv_as_f64, oracle_run, out_rel, rel_l2_max

pytestmark = pytest.mark.gpu


def _check(run: Runner, sess, out, n, o_ref, ST_ref, cs_ref, tol=None):
    tol_o, tol_s = tol or TOL[run.shape.dtype]
    torch.cuda.synchronize()
    o = out[:n].double().cpu().numpy()
    assert np.isfinite(o).all()
    r_o = out_rel(o, o_ref[:n]) if n else 0.0
    r_s = rel_l2_max(sess.S.double().cpu().numpy(), ST_ref)
    assert r_o <= tol_o, f"output rel L2 {r_o:.3e} > {tol_o}"
    assert r_s <= tol_s, f"state rel L2 {r_s:.3e} > {tol_s}"
    assert np.array_equal(conv_as_f64(sess.conv), cs_ref), "conv state differs"
    return r_o, r_s


def test_small_fp32_workload(cuda_device):
    """fp32 inputs, T=2048, 2 heads, d=64, C=64, one call."""
    w = wl.small_fp32()
    tok, cw = w.session_tokens(0), w.conv_weights()
    run = Runner(w.shape, tok, cw, cuda_device)
    sess, out = run.session(), run.new_out()
    assert run.prefill(sess, 0, 2048, out) == 2048
    o_ref, ST_ref, cs_ref = oracle_run(w.shape, tok, cw)
    _check(run, sess, out, 2048, o_ref, ST_ref, cs_ref)
    assert sess.committed == 2048


CASES = [
    # Hk, Hv, d, C, T, partial, act, q_scale, out_dtype
    (2, 2, 128, 64, 300, False, 0, 1.0, gdn.GDN_FP32),
    (2, 4, 128, 512, 1100, True, 0, 1.0, gdn.GDN_FP32),
    (1, 2, 64, 64, 777, True, 1, 0.5, gdn.GDN_FP32),
    (4, 4, 128, 512, 2048, False, 0, 1.0, gdn.GDN_FP32),
    (2, 4, 128, 128, 650, True, 0, 1.0, gdn.GDN_BF16),
    (3, 6, 64, 64, 1, True, 0, 1.0, gdn.GDN_FP32),
    (2, 2, 128, 64, 64, False, 0, 1.0, gdn.GDN_FP32),
    (1, 4, 128, 64, 300, True, 0, 1.0, gdn.GDN_FP32),   # four v-heads per q/k head
    (2, 4, 128, 64, 333, True, 1, 0.7, gdn.GDN_FP32),   # SiLU conv with two v-heads per q/k head
]


@pytest.mark.parametrize("Hk,Hv,d,C,T,partial,act,qs,odt", CASES)
def test_bf16_cases(cuda_device, Hk, Hv, d, C, T, partial, act, qs, odt):
    shape = wl.Shape(Hk, Hv, d, d, C, wl.BF16)
    w = wl.Workload("case", shape, seed=T, session_lengths=[T])
    tok, cw = w.session_tokens(0), w.conv_weights()
    run = Runner(shape, tok, cw, cuda_device, out_dtype=odt, act=act, q_scale=qs)
    sess, out = run.session(), run.new_out()
    n = run.prefill(sess, 0, T, out, gdn.GDN_ALLOW_PARTIAL if partial else 0)
    assert n == (T if partial else (T // C) * C)
    o_ref, ST_ref, cs_ref = oracle_run(shape, tok.slice(0, n), cw, act=act, q_scale=qs)
    _check(run, sess, out, n, o_ref, ST_ref, cs_ref)
    torch.cuda.synchronize()
    # rows of tokens that were not consumed are untouched
    assert torch.isnan(out[n:].float()).all()


def test_carried_state_over_calls(cuda_device):
    """On-grid calls of 512, 1536 and 1024 tokens carry S and the conv state."""
    shape = wl.Shape(2, 4, 128, 128, 512, wl.BF16)
    w = wl.Workload("carry", shape, seed=5, session_lengths=[3072])
    tok, cw = w.session_tokens(0), w.conv_weights()
    run = Runner(shape, tok, cw, cuda_device)
    sess, out = run.session(), run.new_out()
    a = 0
    for n in (512, 1536, 1024):
        assert run.prefill(sess, a, a + n, out) == n
        a += n
    o_ref, ST_ref, cs_ref = oracle_run(shape, tok, cw)
    _check(run, sess, out, 3072, o_ref, ST_ref, cs_ref)


def test_empty_and_sub_grid_calls(cuda_device):
    shape = wl.Shape(2, 2, 128, 128, 512, wl.BF16)
    w = wl.Workload("edge", shape, seed=9, session_lengths=[600])
    tok, cw = w.session_tokens(0), w.conv_weights()
    run = Runner(shape, tok, cw, cuda_device)
    sess, out = run.session(), run.new_out()
    assert run.prefill(sess, 0, 0, out) == 0                       # empty call
    assert run.prefill(sess, 0, 300, out) == 0                     # below one grid chunk: all pending
    torch.cuda.synchronize()
    assert sess.committed == 0 and torch.isnan(out.float()).all()
    assert float(sess.S.abs().max()) == 0.0
    assert run.prefill(sess, 0, 600, out) == 512
    o_ref, ST_ref, cs_ref = oracle_run(shape, tok.slice(0, 512), cw)
    _check(run, sess, out, 512, o_ref, ST_ref, cs_ref)


def test_decode_steps_match_oracle(cuda_device):
    """Prefill 512 tokens, then 5 decode steps; each step's output and the state against the oracle."""
    shape = wl.Shape(2, 4, 128, 128, 512, wl.BF16)
    w = wl.Workload("dec", shape, seed=11, session_lengths=[517])
    tok, cw = w.session_tokens(0), w.conv_weights()
    run = Runner(shape, tok, cw, cuda_device)
    sess, out = run.session(), run.new_out()
    assert run.prefill(sess, 0, 517, out) == 512
    for t in range(512, 517):
        xq, xk, xv, g, beta = (x[t:t + 1] for x in run.x)
        gdn.gdn_decode_step(run.desc, [sess], xq, xk, xv, g, beta, run.cw_t, out[t:t + 1])
    assert sess.committed == 517
    o_ref, ST_ref, cs_ref = oracle_run(shape, tok, cw)
    _check(run, sess, out, 517, o_ref, ST_ref, cs_ref)


@pytest.mark.parametrize("dtype,d,act,q_scale", [(wl.FP32, 64, gdn.GDN_CONV_NONE, 1.0),
                                                  (wl.BF16, 128, gdn.GDN_CONV_SILU, 128 ** -0.5),
                                                  (wl.BF16, 64, gdn.GDN_CONV_NONE, 1.0)],
                         ids=["fp32_d64", "bf16_d128_silu_qscale", "bf16_d64"])
def test_decode_variants_match_oracle(cuda_device, dtype, d, act, q_scale):
    """Decode steps after a prefill, for fp32 inputs, the SiLU conv with a q scale, and d = 64 (GQA layer,
    two v-heads per q/k head): outputs, state and conv state against the oracle."""
    shape = wl.Shape(2, 4, d, d, 64, dtype)
    w = wl.Workload("decv", shape, seed=17, session_lengths=[132])
    tok, cw = w.session_tokens(0), w.conv_weights()
    run = Runner(shape, tok, cw, cuda_device, act=act, q_scale=q_scale)
    sess, out = run.session(), run.new_out()
    assert run.prefill(sess, 0, 132, out) == 128
    for t in range(128, 132):
        gdn.gdn_decode_step(run.desc, [sess], *(x[t:t + 1] for x in run.x), run.cw_t, out[t:t + 1])
    assert sess.committed == 132
    o_ref, ST_ref, cs_ref = oracle_run(shape, tok, cw, act=act, q_scale=q_scale)
    _check(run, sess, out, 132, o_ref, ST_ref, cs_ref)


def test_decode_batch_equals_single(cuda_device):
    """A decode step over 3 sessions equals three single-session steps, bit for bit."""
    shape = wl.Shape(2, 4, 64, 64, 64, wl.BF16)
    runs, sessA, sessB = [], [], []
    for i in range(3):
        w = wl.Workload("decb", shape, seed=20 + i, session_lengths=[70 + i])
        run = Runner(shape, w.session_tokens(0), w.conv_weights() if i == 0 else runs[0].cw, cuda_device)
        runs.append(run)
        for lst in (sessA, sessB):
            s, o = run.session(), run.new_out()
            run.prefill(s, 0, 64, o)
            lst.append(s)
    outA = torch.zeros((3, 4, 64), device=cuda_device)
    cat = lambda j, t: torch.cat([r.x[j][t:t + 1] for r in runs])
    t = 64
    gdn.gdn_decode_step(runs[0].desc, sessA, *(cat(j, t) for j in range(5)), runs[0].cw_t, outA)
    for i, r in enumerate(runs):
        ob = torch.zeros((1, 4, 64), device=cuda_device)
        gdn.gdn_decode_step(r.desc, [sessB[i]], *(x[t:t + 1] for x in r.x), runs[0].cw_t, ob)
        torch.cuda.synchronize()
        assert torch.equal(ob[0], outA[i])
        assert torch.equal(sessA[i].S, sessB[i].S) and torch.equal(sessA[i].conv, sessB[i].conv)


def test_decode_close_to_one_token_partial_prefill(cuda_device):
    shape = wl.Shape(2, 2, 128, 128, 64, wl.BF16)
    w = wl.Workload("dec1", shape, seed=13, session_lengths=[129])
    tok, cw = w.session_tokens(0), w.conv_weights()
    run = Runner(shape, tok, cw, cuda_device)
    a, b = run.session(), run.session()
    oa, ob = run.new_out(), run.new_out()
    run.prefill(a, 0, 128, oa)
    run.prefill(b, 0, 128, ob)
    gdn.gdn_decode_step(run.desc, [a], *(x[128:129] for x in run.x), run.cw_t, oa[128:129])
    run.prefill(b, 128, 129, ob, gdn.GDN_ALLOW_PARTIAL)
    torch.cuda.synchronize()
    # the decode step is fp32; the bf16-input prefill runs on tf32 tensor cores: layer tolerance
    tol_o, tol_s = TOL[wl.BF16]
    ra = oa[128].double().cpu().numpy()
    rb = ob[128].double().cpu().numpy()
    assert np.linalg.norm(ra - rb) <= tol_o * np.linalg.norm(rb)
    assert rel_l2_max(a.S.double().cpu().numpy(), b.S.double().cpu().numpy()) <= tol_s
    assert torch.equal(a.conv, b.conv) and a.committed == b.committed == 129


def test_conv_state_readback(cuda_device):
    shape = wl.Shape(1, 1, 64, 64, 64, wl.BF16)
    w = wl.Workload("cs", shape, seed=3, session_lengths=[130])
    tok, cw = w.session_tokens(0), w.conv_weights()
    run = Runner(shape, tok, cw, cuda_device)
    sess, out = run.session(), run.new_out()
    run.prefill(sess, 0, 130, out)                                  # commits 128
    host = torch.empty((3, shape.channels), dtype=torch.bfloat16).pin_memory()
    gdn.gdn_conv_state(run.desc, sess, host)
    torch.cuda.synchronize()
    expect = np.concatenate([tok.xq[125:128], tok.xk[125:128], tok.xv[125:128]], axis=1)
    assert np.array_equal(host.view(torch.int16).numpy().view(np.uint16), expect)


@pytest.mark.parametrize("kind", ["strong_decay", "no_decay", "alternating"])
def test_extreme_gates_match_oracle(cuda_device, kind):
    """Gates at the edges of their range, where the block's triangular system is least benign: beta near 1
    with a log-decay of -3 per token (decays across a block underflow to zero), with none (g = 0, every
    block's A at full strength), or alternating between the two. 700 tokens (ragged last block), two v-heads
    per q/k head, d = 128 on the tensor-core prologue."""
    shape = wl.Shape(2, 4, 128, 128, 64, wl.BF16)
    T = 700
    w = wl.Workload("gates", shape, seed=31, session_lengths=[T])
    tok, cw = w.session_tokens(0), w.conv_weights()
    rng = np.random.default_rng(5)
    beta = (0.99 - 0.01 * rng.random((T, 4))).astype(np.float32)
    if kind == "strong_decay":
        g = (-3.0 - 0.5 * rng.random((T, 4))).astype(np.float32)
    elif kind == "no_decay":
        g = np.zeros((T, 4), np.float32)
    else:
        g = np.where((np.arange(T) // 7 % 2 == 0)[:, None], -3.0, 0.0).astype(np.float32) * np.ones((1, 4), np.float32)
    tok = wl.Tokens(tok.xq, tok.xk, tok.xv, g, beta)
    run = Runner(shape, tok, cw, cuda_device)
    sess, out = run.session(), run.new_out()
    n = run.prefill(sess, 0, T, out, gdn.GDN_ALLOW_PARTIAL)
    assert n == T
    o_ref, ST_ref, cs_ref = oracle_run(shape, tok, cw)
    _check(run, sess, out, n, o_ref, ST_ref, cs_ref)
