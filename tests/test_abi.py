"""C ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and refuses invalid calls on the host before any device work.
(All calls here fail validation first, so none reaches the CUDA runtime.)"""
import ctypes
import os
import re

import pytest

from chunked_gated_deltanet_gb300 import gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    txt = open(os.path.join(ROOT, "include", "gdn.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", txt)))


@pytest.fixture(scope="module")
def lib():
    from chunked_gated_deltanet_gb300 import build
    build.build()
    return gdn.load_library()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(gdn.EXPORTED)


def test_only_c_abi_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.LIB_PATH], capture_output=True, text=True).stdout
    text_syms = [l.split()[-1] for l in out.splitlines() if " T " in l]
    assert sorted(s for s in text_syms if s.startswith("gdn_")) == sorted(gdn.EXPORTED)


def _desc(**kw):
    base = dict(n_qk_heads=16, n_v_heads=16, d_k=128, d_v=128, grid_c=512)
    base.update(kw)
    return gdn.make_desc(**base)


def test_desc_validation(lib):
    assert gdn.gdn_desc_check(_desc()) == gdn.GDN_OK
    assert gdn.gdn_desc_check(_desc(n_qk_heads=16, n_v_heads=32)) == gdn.GDN_OK
    assert gdn.gdn_desc_check(_desc(d_k=64, d_v=64, grid_c=64, in_dtype=gdn.GDN_FP32)) == gdn.GDN_OK
    for bad in (dict(n_v_heads=24), dict(n_qk_heads=0), dict(d_k=96, d_v=96), dict(d_v=64),
                dict(grid_c=100), dict(grid_c=0), dict(grid_c=8192), dict(in_dtype=7), dict(out_dtype=3),
                dict(conv_act=2)):
        assert gdn.gdn_desc_check(_desc(**bad)) == gdn.GDN_ERR_SHAPE, bad
    assert gdn.gdn_desc_check(_desc(l2_eps=0.0)) == gdn.GDN_ERR_INVALID_ARG
    assert gdn.gdn_desc_check(_desc(q_scale=float("inf"))) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_desc_check(None) == gdn.GDN_ERR_INVALID_ARG


def test_tags_distinguish_layers(lib):
    tags = {gdn.gdn_desc_tag(_desc(**kw)) for kw in
            (dict(), dict(grid_c=64), dict(in_dtype=gdn.GDN_FP32), dict(n_v_heads=32), dict(conv_act=1),
             dict(q_scale=0.5), dict(out_dtype=gdn.GDN_BF16))}
    assert len(tags) == 7 and 0 not in tags
    assert gdn.gdn_desc_tag(_desc()) == gdn.gdn_desc_tag(_desc())
    assert gdn.gdn_desc_tag(_desc(grid_c=3)) == 0


def test_sizes(lib):
    d = _desc()
    assert gdn.gdn_state_bytes(d) == 16 * 128 * 128 * 4            # 1 MiB per layer for the 0.8B shape
    assert gdn.gdn_conv_state_bytes(d) == 3 * (2 * 16 * 128 + 16 * 128) * 2
    d2 = _desc(n_v_heads=32)
    assert gdn.gdn_state_bytes(d2) == 2 * 1024 * 1024
    ws1 = gdn.gdn_workspace_size(d, 1024, 1)
    assert ws1 > 0 and gdn.gdn_workspace_size(d, 4096, 1) > ws1
    assert gdn.gdn_workspace_size(d, -1, 1) == 0


def _fake_session(desc, committed=0, tag=None):
    # host-only struct with fake (never dereferenced) aligned device addresses
    return gdn.gdn_session(0x10000, 0x20000, committed, gdn.gdn_desc_tag(desc) if tag is None else tag)


def _call_prefill(lib, desc, sess, n_tokens, flags=0, ws_bytes=1 << 40, ptr=0x100000):
    nc = ctypes.c_int64(-7)
    p = ctypes.c_void_p(ptr)
    st = lib.gdn_prefill_chunks(ctypes.byref(desc), ctypes.byref(sess), p, p, p, p, p, p, n_tokens, flags, p,
                                ctypes.byref(nc), p, ws_bytes, None)
    return st, nc.value


def test_prefill_refusals_mutate_nothing(lib):
    d = _desc()
    # off grid without the partial flag
    s = _fake_session(d, committed=100)
    st, nc = _call_prefill(lib, d, s, 1024)
    assert st == gdn.GDN_ERR_OFF_GRID and s.committed == 100 and nc == -7
    assert b"off grid" in lib.gdn_last_error()
    # another layer's state
    s = _fake_session(d, tag=12345)
    st, _ = _call_prefill(lib, d, s, 1024)
    assert st == gdn.GDN_ERR_STATE_MISMATCH and s.committed == 0
    # a missing slot used as a session
    s = _fake_session(d, committed=-1)
    assert _call_prefill(lib, d, s, 1024)[0] == gdn.GDN_ERR_STATE_MISMATCH
    # workspace too small
    s = _fake_session(d)
    st, _ = _call_prefill(lib, d, s, 1024, ws_bytes=1000)
    assert st == gdn.GDN_ERR_WORKSPACE and s.committed == 0
    # misaligned input pointer
    assert _call_prefill(lib, d, s, 1024, ptr=0x100004)[0] == gdn.GDN_ERR_INVALID_ARG
    # negative token count, unknown flag
    assert _call_prefill(lib, d, s, -1)[0] == gdn.GDN_ERR_INVALID_ARG
    assert _call_prefill(lib, d, s, 1024, flags=4)[0] == gdn.GDN_ERR_INVALID_ARG
    assert s.committed == 0


def test_noalloc_refusals_before_any_device_work(lib):
    """The no-allocation prefill refuses, on the host and before touching the GPU, a call whose scratch would
    exceed the built-in array, and hands malformed arguments to the regular validation."""
    d = _desc()
    s = _fake_session(d)
    nc = ctypes.c_int64(-7)
    p = ctypes.c_void_p(0x100000)

    def call(n_tokens, flags=0):
        return lib.gdn_prefill_chunks_noalloc(ctypes.byref(d), ctypes.byref(s), p, p, p, p, p, p, n_tokens, flags,
                                              p, ctypes.byref(nc), None)

    T = 4096                      # whole grid chunks, far beyond the built-in scratch for this layer
    need = gdn.gdn_workspace_size(d, T, 1)
    assert need > gdn.GDN_NOALLOC_SCRATCH_BYTES
    assert call(T) == gdn.GDN_ERR_WORKSPACE
    assert b"built-in" in lib.gdn_last_error()
    assert call(-1) == gdn.GDN_ERR_INVALID_ARG
    assert call(T, flags=4) == gdn.GDN_ERR_INVALID_ARG
    assert s.committed == 0 and nc.value == -7


def test_varlen_refusals(lib):
    d = _desc()
    sess = (gdn.gdn_session * 2)(_fake_session(d), gdn.gdn_session(0x30000, 0x40000, 0, gdn.gdn_desc_tag(d)))
    nc = (ctypes.c_int64 * 2)()
    p = ctypes.c_void_p(0x100000)

    def call(cu, sessions=sess, n=2):
        cua = (ctypes.c_int64 * len(cu))(*cu)
        return lib.gdn_prefill_varlen(ctypes.byref(d), sessions, n, cua, p, p, p, p, p, p, 0, p, nc, p, 1 << 40, None)

    assert call([0, 600, 500]) == gdn.GDN_ERR_INVALID_ARG            # decreasing offsets
    assert call([5, 600, 1200]) == gdn.GDN_ERR_INVALID_ARG           # must start at 0
    same = (gdn.gdn_session * 2)(_fake_session(d), _fake_session(d))
    assert call([0, 512, 1024], same) == gdn.GDN_ERR_INVALID_ARG     # duplicate sessions
    assert call([0, 512], sess, 0) == gdn.GDN_ERR_INVALID_ARG        # no sessions
    assert sess[0].committed == 0 and sess[1].committed == 0


def test_state_call_refusals(lib):
    d = _desc()
    src = _fake_session(d, committed=512)
    slot = gdn.gdn_session(0x50000, 0x60000, -1, 0)
    # restoring a missing slot is refused
    assert lib.gdn_state_restore(ctypes.byref(d), ctypes.byref(src), ctypes.byref(slot), None) == \
        gdn.GDN_ERR_STATE_MISMATCH
    assert src.committed == 512
    # a slot of another grid is refused
    other = _desc(grid_c=64)
    slot2 = gdn.gdn_session(0x50000, 0x60000, 512, gdn.gdn_desc_tag(other))
    assert lib.gdn_state_restore(ctypes.byref(d), ctypes.byref(src), ctypes.byref(slot2), None) == \
        gdn.GDN_ERR_STATE_MISMATCH
    # capture into the source's own buffers is refused
    self_slot = _fake_session(d)
    assert lib.gdn_state_capture(ctypes.byref(d), ctypes.byref(src), ctypes.byref(self_slot), None) == \
        gdn.GDN_ERR_INVALID_ARG
    # decode with no sessions / duplicate sessions
    p = ctypes.c_void_p(0x100000)
    two = (gdn.gdn_session * 2)(_fake_session(d), _fake_session(d))
    assert lib.gdn_decode_step(ctypes.byref(d), two, 2, p, p, p, p, p, p, p, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_decode_step(ctypes.byref(d), two, 0, p, p, p, p, p, p, p, None) == gdn.GDN_ERR_INVALID_ARG


def test_status_strings(lib):
    assert lib.gdn_status_string(gdn.GDN_ERR_OFF_GRID) == b"GDN_ERR_OFF_GRID"
    assert lib.gdn_status_string(99) == b"unknown status"


def _fake(desc, base, committed=0):
    # device addresses that are never dereferenced: every call below is refused first
    return gdn.gdn_session(ctypes.c_void_p(base), ctypes.c_void_p(base + 0x100000), committed, gdn.gdn_desc_tag(desc))


def test_branch_and_checkpoint_refusals(lib):
    d = _desc(grid_c=64)
    vp = ctypes.c_void_p
    x = [vp(0x7000000 + 0x10000 * i) for i in range(7)]     # xq, xk, xv, g, beta, conv_w, out
    cu = (ctypes.c_int64 * 3)(0, 64, 128)
    nc = (ctypes.c_int64 * 2)()
    prefix = _fake(d, 0x1000000, committed=128)
    br = (gdn.gdn_session * 2)(_fake(d, 0x2000000), _fake(d, 0x3000000))

    def branches(pref, arr, flags=0):
        return lib.gdn_prefill_branches(ctypes.byref(d), pref, arr, 2, cu, *x[:6], flags, x[6], nc,
                                        vp(0x9000000), 1 << 30, None)

    assert branches(None, br) == gdn.GDN_ERR_INVALID_ARG
    alias = (gdn.gdn_session * 2)(_fake(d, 0x2000000), _fake(d, 0x1000000))   # a branch is the prefix
    assert branches(ctypes.byref(prefix), alias) == gdn.GDN_ERR_INVALID_ARG
    off = _fake(d, 0x1000000, committed=100)                                 # off grid, no partial flag
    assert branches(ctypes.byref(off), br) == gdn.GDN_ERR_OFF_GRID
    foreign = _fake(_desc(grid_c=128), 0x1000000, committed=128)
    assert branches(ctypes.byref(foreign), br) == gdn.GDN_ERR_STATE_MISMATCH
    assert [b.committed for b in br] == [0, 0] and prefix.committed == 128

    s = _fake(d, 0x4000000)
    slot = _fake(d, 0x5000000, committed=-1)

    def ckpt(sess, sl):
        return lib.gdn_prefill_chunks_checkpoint(ctypes.byref(d), ctypes.byref(sess), ctypes.byref(sl), *x[:6], 64,
                                                 0, x[6], ctypes.byref(ctypes.c_int64()), vp(0x9000000), 1 << 30,
                                                 None)

    assert ckpt(s, _fake(d, 0x4000000)) == gdn.GDN_ERR_INVALID_ARG           # the slot is the session
    nul = gdn.gdn_session(None, None, -1, gdn.gdn_desc_tag(d))
    assert ckpt(s, nul) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_prefill_varlen_checkpoint(ctypes.byref(d), ctypes.byref(s), None, 1, cu, *x[:6], 0, x[6], nc,
                                             vp(0x9000000), 1 << 30, None) == gdn.GDN_ERR_INVALID_ARG
    assert (slot.committed, s.committed) == (-1, 0)


def test_gate_call_refusals(lib):
    """gdn_gates checks its layer description, sizes, pointers and alignment on the host."""
    d = gdn.make_desc(2, 4, 64, 64, 64)
    P = lambda v: ctypes.c_void_p(v)
    ok = [P(0x1000), P(0x2000), P(0x3000), P(0x4000)]
    outs = [P(0x5000), P(0x6000)]
    call = lambda desc, ins, n, o: lib.gdn_gates(ctypes.byref(desc), *ins, n, *o, None)
    assert call(d, [None] + ok[1:], 8, outs) == gdn.GDN_ERR_INVALID_ARG
    assert call(d, ok, 8, [outs[0], None]) == gdn.GDN_ERR_INVALID_ARG
    assert call(d, [P(0x1002)] + ok[1:], 8, outs) == gdn.GDN_ERR_INVALID_ARG     # misaligned
    assert call(d, ok, -1, outs) == gdn.GDN_ERR_INVALID_ARG
    bad = gdn.make_desc(2, 3, 64, 64, 64)                                      # Hv not a multiple of Hk
    assert call(bad, ok, 8, outs) != gdn.GDN_OK


def test_missing_library_fails_loudly(tmp_path):
    """No fallback: without the built library the binding raises instead of computing anything."""
    with pytest.raises(ImportError):
        gdn.load_library(str(tmp_path / "libgdn.so"))


def test_product_package_never_uses_the_oracle():
    """The oracle is test infrastructure: nothing in the package imports, loads or names its module."""
    pkg = os.path.join(ROOT, "chunked_gated_deltanet_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "gdn_oracle" not in text, f
