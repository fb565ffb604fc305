"""Host-side checks of the synthetic workloads and the grid arithmetic (no GPU)."""
import json
import os

import numpy as np

from chunked_gated_deltanet_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_grid_tail_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "grid_tail.json")))
    w = wl.qwen08b_replay()
    assert sum(w.turns[0]) == g["session_tokens"] == w.session_lengths[0]
    assert w.shape.grid_c == g["grid"]
    # replaying turn by turn while holding the sub-grid tail commits only whole chunks
    committed, pending = 0, 0
    for n in w.turns[0]:
        avail = pending + n
        take = wl.grid_floor(avail, w.shape.grid_c)
        committed += take
        pending = avail - take
    assert committed == g["committed"] and pending == g["pending_tail"]


def test_prefix_cut_rule_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "prefix_cuts.json")))
    for prefix, rerun in g["rows"]:
        assert prefix - wl.grid_floor(prefix, g["multiple"]) == rerun


def test_turn_recipes():
    w = wl.qwen08b_replay()
    t = w.turns[0]
    assert len(t) == 30 and min(t) >= 200 and max(t) <= 4000
    v = wl.varlen8()
    assert len(v.session_lengths) == 8
    assert all(4096 <= n <= 65536 for n in v.session_lengths)
    assert all(sum(tt) == n and len(tt) == 6 for tt, n in zip(v.turns, v.session_lengths))
    L = wl.long_session()
    assert sum(L.turns[0]) == 100_000 and len(L.fork_questions) == 64
    assert all(20 <= q <= 200 for q in L.fork_questions)
    assert wl.grid_floor(100_000, 512) == 99_840
    s = wl.shared_prefix()
    assert [wl.grid_floor(s.request_prefix + p, 64) for p in s.group_prefixes] == [960, 960, 1024, 1088]
    assert sum(len(b) for b in s.branches) == 16


def test_draws_are_split_independent():
    w = wl.small_fp32()
    full = w.session_tokens(0)
    part = w.session_tokens(0, T=100)
    assert np.array_equal(full.xq[:100], part.xq)
    # later arrays (g, beta) depend on T: sessions are drawn once at full length and sliced
    # pre-normalised q and k in the fp32 workload
    n = np.linalg.norm(full.xq.reshape(-1, 2, 64).astype(np.float64), axis=-1)
    assert np.allclose(n, 1.0, atol=1e-6)
    assert np.all(full.g < 0) and np.all((full.beta > 0) & (full.beta < 1))


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38, 1e-40], dtype=np.float32)
    b = wl.f32_to_bf16_bits(x)
    back = wl.bf16_bits_to_f32(b)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to even (1.0)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.0 + 2 ** -6)
    assert back[3] == -2.5
    import torch
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(back[:5], ref[:5])


def test_fast_bf16_path_equals_bit_formula():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-20, 20, 200_000))).astype(np.float32)
    assert np.array_equal(wl._round(x, wl.BF16), wl.f32_to_bf16_bits(x))
