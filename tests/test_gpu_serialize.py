"""Serialised states on the GPU: pinned-memory round trip, file round trip,
refusals, and the write protocol (a failed save leaves the path empty)."""
import os

import pytest
import torch

from chunked_gated_deltanet_gb300 import gdn
from chunked_gated_deltanet_gb300 import workloads as wl
from helpers import Runner

pytestmark = pytest.mark.gpu


def _session_after(run, n):
    s, o = run.session(), run.new_out()
    assert run.prefill(s, 0, n, o) == n
    return s


@pytest.fixture
def run(cuda_device):
    shape = wl.Shape(2, 4, 128, 128, 64, wl.BF16)
    w = wl.Workload("ser", shape, seed=33, session_lengths=[512])
    return Runner(shape, w.session_tokens(0), w.conv_weights(), cuda_device)


def _continue_equal(run, a, b, start):
    oa, ob = run.new_out(), run.new_out()
    run.prefill(a, start, start + 128, oa)
    run.prefill(b, start, start + 128, ob)
    torch.cuda.synchronize()
    assert torch.equal(oa[start:start + 128], ob[start:start + 128])
    assert torch.equal(a.S, b.S) and torch.equal(a.conv, b.conv)


def test_pinned_round_trip_is_bitwise(run):
    src = _session_after(run, 192)
    blob = torch.empty(gdn.gdn_state_blob_bytes(run.desc), dtype=torch.uint8).pin_memory()
    gdn.gdn_state_serialize(run.desc, src, blob)
    torch.cuda.synchronize()
    dst = run.session()
    gdn.gdn_state_deserialize(run.desc, blob, dst)
    torch.cuda.synchronize()
    assert dst.committed == src.committed == 192
    assert torch.equal(dst.S, src.S) and torch.equal(dst.conv, src.conv)
    _continue_equal(run, src, dst, 192)
    # without its completion marker the same blob reads as missing, and the destination stays as it was
    blob[80:88] = 0
    fresh = run.session()
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_state_deserialize(run.desc, blob, fresh)
    assert e.value.status == gdn.GDN_ERR_STATE_MISMATCH and fresh.committed == 0


def test_file_round_trip_refusals_and_overwrite(run, tmp_path):
    path = str(tmp_path / "state.gdn")
    a = _session_after(run, 128)
    gdn.gdn_state_save(run.desc, a, path)
    assert os.path.getsize(path) == gdn.gdn_state_blob_bytes(run.desc)
    assert not os.path.exists(path + ".tmp")
    b = run.session()
    gdn.gdn_state_load(run.desc, path, b)
    assert b.committed == 128 and torch.equal(a.S, b.S) and torch.equal(a.conv, b.conv)
    # a newer save replaces the file
    c = _session_after(run, 256)
    gdn.gdn_state_save(run.desc, c, path)
    gdn.gdn_state_load(run.desc, path, b)
    assert b.committed == 256 and torch.equal(c.S, b.S)
    _continue_equal(run, c, b, 256)
    # a flipped payload byte fails the checksum; another layer description is refused
    raw = bytearray(open(path, "rb").read())
    raw[128 + 1000] ^= 0x40
    bad = str(tmp_path / "bad.gdn")
    open(bad, "wb").write(bytes(raw))
    d = run.session()
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_state_load(run.desc, bad, d)
    assert e.value.status == gdn.GDN_ERR_STATE_MISMATCH and d.committed == 0
    other = gdn.make_desc(2, 4, 128, 128, 512)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_state_load(other, path, gdn.Session(other, run.dev))
    assert e.value.status == gdn.GDN_ERR_STATE_MISMATCH


def test_failed_save_leaves_nothing_stale(run, tmp_path):
    path = str(tmp_path / "state.gdn")
    gdn.gdn_state_save(run.desc, _session_after(run, 64), path)
    os.mkdir(path + ".tmp")            # the temporary file cannot be created: the save fails midway
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_state_save(run.desc, _session_after(run, 128), path)
    assert e.value.status == gdn.GDN_ERR_IO
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_state_load(run.desc, path, run.session())
    assert e.value.status == gdn.GDN_ERR_NOT_FOUND    # missing, not the older 64-token state
