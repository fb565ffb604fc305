"""Serialised-state refusals that need no GPU: every check runs on the host
before any device work. The blobs are packed here from the header layout the
C header documents, so these tests also pin that layout."""
import ctypes
import os
import struct

import numpy as np
import pytest

from chunked_gated_deltanet_gb300 import gdn

# "GDNSTATE", version, header bytes, tag, Hk, Hv, d_k, d_v, grid, in_dtype, committed, S bytes, conv bytes,
# checksum, completion marker, 40 bytes of padding
HDR = struct.Struct("<8sIIQ6iqQQQQ40x")


@pytest.fixture(scope="module")
def lib():
    from chunked_gated_deltanet_gb300 import build
    build.build()
    return gdn.load_library()


def _desc(**kw):
    base = dict(n_qk_heads=2, n_v_heads=4, d_k=64, d_v=64, grid_c=64)
    base.update(kw)
    return gdn.make_desc(**base)


def _blob(desc, committed=128, tag=None, magic=b"GDNSTATE", version=1, checksum=0, complete=0, payload=True):
    S, C = gdn.gdn_state_bytes(desc), gdn.gdn_conv_state_bytes(desc)
    tag = gdn.gdn_desc_tag(desc) if tag is None else tag
    h = HDR.pack(magic, version, 128, tag, desc.n_qk_heads, desc.n_v_heads, desc.d_k, desc.d_v, desc.grid_c,
                 desc.in_dtype, committed, S, C, checksum, complete)
    return np.frombuffer(h + (bytes(S + C) if payload else b""), dtype=np.uint8).copy()


def _fake_session(desc):
    # device addresses are never dereferenced: every call below is refused first
    return gdn.gdn_session(ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), 7, gdn.gdn_desc_tag(desc))


def _deserialize(lib, desc, blob, nbytes=None):
    s = _fake_session(desc)
    st = lib.gdn_state_deserialize(ctypes.byref(desc), blob.ctypes.data_as(ctypes.c_void_p),
                                   blob.nbytes if nbytes is None else nbytes, ctypes.byref(s), None)
    assert (s.committed, s.tag) == (7, gdn.gdn_desc_tag(desc)), "a refused restore changed the session"
    return st


def test_header_layout_is_128_bytes_and_sizes_add_up(lib):
    d = _desc()
    assert HDR.size == 128
    assert gdn.gdn_state_blob_bytes(d) == 128 + gdn.gdn_state_bytes(d) + gdn.gdn_conv_state_bytes(d)
    assert gdn.gdn_state_blob_bytes(_desc(grid_c=100)) == 0


def test_deserialize_refusals(lib):
    d = _desc()
    M = gdn.GDN_ERR_STATE_MISMATCH
    assert _deserialize(lib, d, _blob(d)) == M                                   # no completion marker
    assert _deserialize(lib, d, _blob(d, magic=b"NOTSTATE", complete=1)) == M    # not a state
    assert _deserialize(lib, d, _blob(d, version=2, complete=1)) == M            # another format version
    other = _desc(grid_c=128)
    assert _deserialize(lib, d, _blob(d, tag=gdn.gdn_desc_tag(other), complete=1)) == M   # another layer
    assert _deserialize(lib, other, _blob(d, complete=1)) == M                   # shapes agree, grid does not
    assert _deserialize(lib, d, _blob(d, complete=1, payload=False)) == M        # shorter than its header says
    assert _deserialize(lib, d, _blob(d), nbytes=64) == gdn.GDN_ERR_INVALID_ARG  # shorter than a header
    assert _deserialize(lib, d, _blob(d, committed=-1, complete=1)) == M


def test_load_refusals(lib, tmp_path):
    d = _desc()
    s = _fake_session(d)
    load = lambda path: lib.gdn_state_load(ctypes.byref(d), os.fsencode(str(path)), ctypes.byref(s), None)
    assert load(tmp_path / "absent") == gdn.GDN_ERR_NOT_FOUND
    (tmp_path / "short").write_bytes(b"GDNSTATE" + bytes(100))
    assert load(tmp_path / "short") == gdn.GDN_ERR_STATE_MISMATCH
    (tmp_path / "unsummed").write_bytes(_blob(d, complete=1).tobytes())
    assert load(tmp_path / "unsummed") == gdn.GDN_ERR_STATE_MISMATCH            # a file must carry its checksum
    (tmp_path / "incomplete").write_bytes(_blob(d, checksum=5).tobytes())
    assert load(tmp_path / "incomplete") == gdn.GDN_ERR_STATE_MISMATCH
    assert (s.committed, s.tag) == (7, gdn.gdn_desc_tag(d))
    assert lib.gdn_state_save(ctypes.byref(d), ctypes.byref(s), b"", None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_state_load(ctypes.byref(d), b"", ctypes.byref(s), None) == gdn.GDN_ERR_INVALID_ARG
    foreign = _fake_session(_desc(grid_c=128))
    assert lib.gdn_state_load(ctypes.byref(d), os.fsencode(str(tmp_path / "absent")), ctypes.byref(foreign),
                              None) == gdn.GDN_ERR_STATE_MISMATCH


def test_status_strings(lib):
    assert lib.gdn_status_string(gdn.GDN_ERR_NOT_FOUND) == b"GDN_ERR_NOT_FOUND"
    assert lib.gdn_status_string(gdn.GDN_ERR_IO) == b"GDN_ERR_IO"
