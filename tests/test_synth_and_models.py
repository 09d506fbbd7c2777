"""Pins of the input generator, the byte/flop model and the dispatch formula (CPU)."""
import math

import numpy as np
import pytest

from conftest import golden
from oracle import dispatch, model
from synth import gen, workloads


def test_generator_published_vector():
    g = golden("splitmix64_vector.json")
    s = gen.SplitMix64(g["seed"])
    assert [s.next() for _ in range(5)] == [int(x) for x in g["outputs"]]
    # counter form: output n of a stream started at state s is mix64(s + n * gamma)
    assert gen.mix64(g["seed"] + 3 * gen.GAMMA) == int(g["outputs"][2])


def test_normal_table_is_a_quantile_table():
    t = gen.bf16_bits_to_f64(gen.normal_table_bits())
    assert np.all(np.diff(t) >= 0)
    np.testing.assert_array_equal(t, -t[::-1])            # symmetric quantiles
    assert abs(t.mean()) < 1e-12 and abs(t.std() - 1.0) < 2e-3
    assert abs(t[32767]) < 1e-4 and abs(t[int(0.975 * 65536)] - 1.96) < 0.01


def test_normal_bits_counter_based_and_chunk_independent():
    key = gen.stream_key(7, 1, 2, 3)
    a = gen.normal_bits(key, 0, 5000)
    b = gen.normal_bits(key, 1234, 100)
    np.testing.assert_array_equal(a[1234:1334], b)
    table = gen.normal_table_bits()
    for i in (0, 17, 4999):
        assert a[i] == table[gen.mix64(key + (i + 1) * gen.GAMMA) >> 48]


def test_pow2_scaling_is_exact():
    bits = gen.normal_bits(gen.stream_key(1, 5), 0, 1000)
    np.testing.assert_array_equal(gen.bf16_bits_to_f64(gen.scale_bf16_bits_pow2(bits, 3)),
                                  gen.bf16_bits_to_f64(bits) * 8.0)


def test_workload_shapes():
    w = workloads.config(1)
    assert (w.L, w.Hq, w.Hkv, w.d, w.B, w.prefix_lens) == (1, 4, 2, 64, 4, [64])
    assert all(1 <= r.suffix_len <= 48 for r in w.requests)
    w = workloads.config(2)
    assert (w.L, w.Hq, w.Hkv, w.d, w.B, w.prefix_lens) == (32, 32, 8, 128, 64, [16384])
    assert all(256 <= r.suffix_len <= 2048 for r in w.requests)
    w = workloads.config(4)
    assert len(w.prefix_lens) == 8 and all(2048 <= lp <= 16384 for lp in w.prefix_lens)
    counts = np.bincount([r.prefix for r in w.requests])
    assert all(16 <= c <= 64 for c in counts)
    w = workloads.config(5)
    assert w.B == 128 and w.page_size == 16 and w.steps == 32 and len(w.parents) == 32


def test_kv_bytes_per_token_printed():
    for c in golden("kv_bytes_per_token.json")["cases"]:
        assert model.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["elem_bytes"]) == c["bytes"]


def test_table23_byte_and_flop_model():
    g = golden("granikv_table23_byte_model.json")
    s, p, tol = g["shape"], g["printed"], g["tolerance_rel"]
    paged = model.paged_prefix_bytes(s["B"], s["Lp"], s["Hkv"], s["d"], s["elem_bytes"])
    shared = model.shared_prefix_bytes(s["Lp"], s["Hkv"], s["d"], s["elem_bytes"])
    flops = model.prefix_flops(s["B"], s["Hq"], s["Lp"], s["d"])
    assert abs(paged / 1e9 - p["paged_bytes_model_GB"]) / p["paged_bytes_model_GB"] < tol
    assert abs(shared / 1e6 - p["shared_bytes_model_MB"]) / p["shared_bytes_model_MB"] < tol
    assert abs(flops / 1e9 - p["useful_GFLOP"]) / p["useful_GFLOP"] < tol
    assert abs(flops / (p["paged_bytes_measured_GB"] * 1e9) - p["paged_arith_intensity_measured"]) < 0.01
    assert abs(flops / (p["hot_dram_measured_MB"] * 1e6) - p["hot_arith_intensity_measured"]) < 1.0


def test_eq2_meff_and_a100_threshold_rows():
    g = golden("granikv_table16_meff.json")
    for B, meff, route in g["rows"]:
        m = dispatch.m_eff(B, g["n_q_per_kv"])
        assert m == meff
        assert ("dense" if m >= g["m_sat_a100"] else "cascade") == route


CM = dict(c_flat_us=5.0, bw_flat_gbs=4000.0, c_cascade_us=10.0, bw_prefix_gbs=5000.0, bw_suffix_gbs=4000.0,
          c_merge_us=0.001, prefix_tile_us=2.0, prefix_item_us=3.0, gather_sm_gbs=1.0, c_gather_us=4.0,
          prefix_tile_split_us=2.5, warp_tile_us=0.25, warp_group_us=0.03125, warp_item_us=1.5, warp_split_ratio=1.5,
          prefix_cta_ramp_us=4.0, prefix_cta_gather_ratio=1.0, c_merge_state_us=0.5, prefix_item_split_us=3.0,
          warp_item_split_us=1.5, prefix_item_crowd_us=0.0, split_gather_ratio_tensor=1.0, c_gather_split_us=4.0,
          split_tensor_us=0.0)


def test_cost_model_closed_form():
    cm = CM
    # one group of 64 requests (g = 4 -> M = 256: one tensor-core row block, two warp-MMA
    # row blocks), Lp = 1000 (8 key tiles), suffixes 100 each, Hkv = 8, d = 128
    f = dispatch.features([1000] * 64, [100] * 64, [0] * 64, 32, 8, 128)
    kv = 2 * 8 * 128 * 2
    assert f["bytes_flat"] == 64 * 1100 * kv and f["bytes_suffix"] == 64 * 100 * kv
    assert f["prefix"] == [dict(M=256, bytes=1000 * kv, flops=4 * 64 * 32 * 1000 * 128, lp=1000)]
    # work decomposition: row blocks x KV heads x key splits
    assert dispatch.n_items(f, 1) == 64 and dispatch.n_items(f, 8) == 8 and dispatch.n_items(f, 3) == 24
    assert dispatch.n_items(f, 1, "warp") == 128 and dispatch.n_items(f, 8, "warp") == 16
    # a last row block of one Q tile (M = 384: 256 + 128 rows; M = 640 at g = 5: 2 x 256 + 128)
    # takes two splits per item: 8 heads x (8 + 4) at C = 1, x (3 + 2) at C = 3; at M = 420 the
    # last block (164 rows) needs both Q tiles and is a full one
    f384 = dispatch.features([1000] * 96, [100] * 96, [0] * 96, 32, 8, 128)
    assert dispatch.n_items(f384, 1) == 8 * (8 + 4) and dispatch.n_items(f384, 3) == 8 * (3 + 2)
    f640 = dispatch.features([1000] * 128, [100] * 128, [0] * 128, 40, 8, 128)
    assert f640["prefix"][0]["M"] == 640 and dispatch.n_items(f640, 1) == 8 * (2 * 8 + 4)
    # unpaired (split plans): every block takes one split per item
    assert dispatch.n_items(f384, 1, paired=False) == 8 * 2 * 8 and dispatch.n_items(f640, 3, paired=False) == 8 * 3 * 3
    f420 = dispatch.features([1000] * 84, [100] * 84, [0] * 84, 40, 8, 128)
    assert dispatch.n_items(f420, 1) == 8 * 2 * 8 and dispatch.n_items(f384, 1, "warp") == 3 * 8 * 8
    # sequential plan, tensor-core items of one tile: one wave of 64 items, each 2 + 3 us
    # (8 prefix splits and one suffix segment per request: 576 partial states, 9 a request)
    t_flat, t_cas = dispatch.predict(cm, f, dict(split=False, C=1, n_pre=64, kind="tensor", gather=False,
                                                 partials=576))
    assert math.isclose(t_flat, 5.0 + 64 * 1100 * kv / 4e6)
    t_levels = max(1000 * kv / 5e6, 1 * (1 * 2.0 + 3.0)) + 4.0 + 64 * 100 * kv / 4e6
    assert math.isclose(t_cas, 10.0 + t_levels + 0.001 * 64 * 32 + 0.5 * 9)
    assert dispatch.choose(t_flat, t_cas) == ("dense" if t_flat < t_cas else "cascade")
    assert dispatch.choose(1.0, 1.0) == "cascade"       # flat only when strictly faster
    # the same with warp items of 4 tiles: 32 items, one wave; the fullest warp item has
    # 128 rows (8 groups of 16), so a tile costs 0.25 + 8 * 0.03125 = 0.5 us: 4 * 0.5 + 1.5
    assert dispatch.warp_row_groups(f) == 8
    _, t_w = dispatch.predict(cm, f, dict(split=False, C=4, n_pre=32, kind="warp", gather=False, partials=192))
    assert math.isclose(t_w, 10.0 + max(1000 * kv / 5e6, 3.5) + 4.0 + 64 * 100 * kv / 4e6 + 0.001 * 64 * 32 + 0.5 * 3)
    # no suffix: no gather launch in the sequential plan; a negative total counts as zero
    f0 = dispatch.features([1000] * 64, [0] * 64, [0] * 64, 32, 8, 128)
    assert math.isclose(dispatch.sequential_levels(cm, f0, 1, 64, 152), max(1000 * kv / 5e6, 5.0))
    assert dispatch.predict(dict(cm, c_cascade_us=-100.0), f0, dict(split=False, C=1, n_pre=64, kind="tensor",
                                                                   gather=False, partials=512))[1] == 0.0
    # 200 items over 152 SMs: two waves
    assert math.isclose(dispatch.sequential_levels(cm, f, 2, 200, 152),
                        max(1000 * kv / 5e6, 2 * (2 * 2.0 + 3.0)) + 4.0 + 64 * 100 * kv / 4e6)
    # a request without a HOT prefix counts only toward the flat and suffix bytes
    f2 = dispatch.features([0, 1000], [300, 10], [-1, 0], 32, 8, 128)
    assert f2["bytes_flat"] == 1310 * kv and len(f2["prefix"]) == 1 and f2["prefix"][0]["M"] == 4


def test_split_formula_worked_example():
    """One group of 64 requests (g = 4 -> one 256-row block), Lp = 16384 (128 key tiles),
    Hkv = 8, 1000 suffix tokens each; tile 1 us, item 5 us, 50 GB/s per SM, 6000 GB/s over
    every SM, 4 us gather ramp for gather-only and for prefix CTAs, 152 SMs.  The gather is
    W = S / 50 GB/s = 5242.88 SM-us; with n items of C + 5 us whose CTAs gather too,
    T_gather = (W + (152 - n) 4 + n (C + 5 + 4)) / 152; the levels take
    max(C + 5, T_gather, (S + prefix bytes) / 6000 GB/s): HBM binds at 54.875 us from
    C = 49 down (C = 50: 55)."""
    cm = dict(CM, bw_suffix_gbs=6000.0, prefix_tile_us=1.0, prefix_item_us=5.0, gather_sm_gbs=50.0,
              prefix_tile_split_us=1.0, prefix_item_split_us=5.0)
    f = dispatch.features([16384] * 64, [1000] * 64, [0] * 64, 32, 8, 128)
    S = 64 * 1000 * 4096
    P = 16384 * 4096
    W = S / 50e3
    assert f["bytes_suffix"] == S
    assert math.isclose(dispatch.split_levels(cm, f, 50, 24, 152), 55.0)
    assert math.isclose(dispatch.split_levels(cm, f, 49, 24, 152), (S + P) / 6e6)
    # C = 64: 16 items of 69 us; the gather spread over every SM is shorter
    assert math.isclose(dispatch.split_levels(cm, f, 64, 16, 152), 69.0)
    assert (W + 136 * 4 + 16 * 73.0) / 152 < 69.0
    _, t_cas = dispatch.predict(cm, f, dict(split=True, C=32, n_pre=32, kind="tensor", gather=True, partials=320))
    assert math.isclose(t_cas, 10.0 + (S + P) / 6e6 + 0.001 * 64 * 32 + 0.5 * 5)
    # a slow gather binds: 10 GB/s per SM.  Prefix CTAs gathering at the full rate, at half
    # of it, or not at all (then the 136 others take it all after their 4 us ramp)
    cm3 = dict(cm, gather_sm_gbs=10.0)
    W3 = S / 10e3
    assert math.isclose(dispatch.split_levels(cm3, f, 64, 16, 152), (W3 + 136 * 4 + 16 * 73.0) / 152)
    assert math.isclose(dispatch.split_levels(dict(cm3, prefix_cta_gather_ratio=0.5), f, 64, 16, 152),
                        (W3 + 136 * 4 + 16 * 0.5 * 73.0) / (136 + 16 * 0.5))
    assert math.isclose(dispatch.split_levels(dict(cm3, prefix_cta_ramp_us=20.0), f, 64, 16, 152),
                        (W3 + 136 * 4 + 16 * 89.0) / 152)
    assert math.isclose(dispatch.split_levels(cm3, f, 64, 16, 152, gather=False), 4.0 + W3 / 136)
    # a split launch of tensor-core items gathers at split_gather_ratio_tensor of the rate;
    # one of warp items at the full rate
    assert math.isclose(dispatch.split_levels(dict(cm3, split_gather_ratio_tensor=0.5), f, 64, 16, 152, gather=False),
                        4.0 + 2 * W3 / 136)
    assert math.isclose(dispatch.split_levels(dict(cm3, split_gather_ratio_tensor=0.5, warp_item_split_us=5.0), f, 64,
                                              16, 152, "warp", R=1, gather=False), 4.0 + W3 / 136)
    # a split launch of tensor-core items pays split_tensor_us on top; one of warp items not
    assert math.isclose(dispatch.split_levels(dict(cm3, split_tensor_us=3.0), f, 64, 16, 152, gather=False),
                        4.0 + W3 / 136 + 3.0)
    assert math.isclose(dispatch.split_levels(dict(cm3, split_tensor_us=3.0, warp_item_split_us=5.0), f, 64, 16, 152,
                                              "warp", R=1, gather=False), 4.0 + W3 / 136)
    # each item of a split launch pays prefix_item_crowd_us per item of the launch
    assert math.isclose(dispatch.split_levels(dict(cm, prefix_item_crowd_us=0.5), f, 64, 16, 152), 69.0 + 8.0)
    # a split item runs beside the gather: the split formula takes the split tile time and
    # the split item's fixed cost (C = 64: 16 items of 64 * 2 + 7 = 135 us against 69), the
    # sequential one the lone tile and the lone item (7 * 1 + 5)
    cm2 = dict(cm, prefix_tile_split_us=2.0, prefix_item_split_us=7.0)
    assert math.isclose(dispatch.split_levels(cm2, f, 64, 16, 152), 135.0)
    t_seq = max(P / 5e6, 7 * 1.0 + 5.0) + 4.0 + S / 6e6
    assert math.isclose(dispatch.sequential_levels(cm2, f, 7, 152, 152), t_seq)
    # the gather as a whole is held to HBM: at 1000 GB/s over every SM the 262 MB take
    # 4 + 262.1 us even though the SMs' own rate would finish them sooner
    cm4 = dict(cm, bw_suffix_gbs=1000.0)
    assert math.isclose(dispatch.split_levels(cm4, f, 64, 16, 152), (S + P) / 1e6)
    assert math.isclose(dispatch.split_levels(cm4, f, 64, 16, 152, gather=False), (S + P) / 1e6)
    assert math.isclose(dispatch.split_levels(dict(cm4, c_gather_split_us=80.0), f, 64, 16, 152), 80.0 + S / 1e6)
    # the split launch's gather starts after its own fixed cost, not the stand-alone
    # gather launch's: c_gather_us prices only the sequential plan
    assert math.isclose(dispatch.split_levels(dict(cm3, c_gather_split_us=9.0, c_gather_us=1.0), f, 64, 16, 152,
                                              gather=False), 9.0 + W3 / 136)
    assert math.isclose(dispatch.sequential_levels(dict(cm2, c_gather_split_us=50.0), f, 7, 152, 152), t_seq)
    # warp-MMA items take their own terms: 2 row blocks x 8 heads x 4 splits of 32 tiles,
    # a tile beside the gather 1.5 * (1 + 8 * 0.125) = 3 us: item 32 * 3 + 2 = 98 us
    cmw = dict(cm, warp_tile_us=1.0, warp_group_us=0.125, warp_split_ratio=1.5, warp_item_us=9.0,
               warp_item_split_us=2.0)
    assert dispatch.n_items(f, 32, "warp") == 64
    assert math.isclose(dispatch.split_levels(cmw, f, 32, 64, 152, "warp", R=8), 98.0)
    # R rounds the fullest item's 16-row groups up to a power of two
    for B, R in ((1, 1), (4, 1), (5, 2), (8, 2), (9, 4), (16, 4), (17, 8), (100, 8)):
        assert dispatch.warp_row_groups(dispatch.features([512] * B, [1] * B, [0] * B, 32, 8, 128)) == R
