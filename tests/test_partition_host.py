"""The gather partitions of a plan (gk_plan_segments), on the host.

Every token of every request is gathered exactly once; a CTA's segments are one
contiguous piece of the concatenated token stream; the quotas follow the
planner's rule (equal quotas of at least 64 tokens, multiples of 16, over at
most one CTA per SM, the last CTA taking the rest; a split plan: one slot per
SM, its end in the stream rounded to 16, a prefix CTA's slot no larger than a
gather-only CTA's); the partial states of a request are one contiguous range
of entries, which is how the merge reads them.
"""
import random

import numpy as np
import pytest

from oracle import dispatch as odisp

SMS = 152


@pytest.fixture(scope="module")
def gk():
    from paged_kv_cache_pool_gb300 import build
    build.build()
    from paged_kv_cache_pool_gb300 import binding
    return binding


def _plan(gk, pool, bases, lps, slens):
    b = gk.Batch(bases, lps, slens, None, 8192)
    return b, gk.gk_plan_build(pool, b)


def _check_cover(begin, segs, lengths):
    """Each request's [0, n) covered once; CTA b's segments continue the stream where CTA b-1 stopped."""
    assert begin[0] == 0 and begin[-1] == len(segs) and np.all(np.diff(begin) >= 0)
    pos = 0            # position in the concatenated stream
    starts = np.concatenate([[0], np.cumsum(lengths)])
    for r, t0, t1, _ in segs.tolist():
        assert 0 <= t0 < t1 <= lengths[r]
        assert starts[r] + t0 == pos, "segments leave a gap or overlap in the stream"
        pos = starts[r] + t1
    assert pos == sum(lengths)


def _tokens(begin, segs):
    return [int(sum(segs[i, 2] - segs[i, 1] for i in range(begin[b], begin[b + 1]))) for b in range(len(begin) - 1)]


def _check_entries(segs, dense):
    by_req = {}
    for r, _, _, e in segs.tolist():
        by_req.setdefault(r, []).append(e)
    seen = set()
    for r, es in by_req.items():
        if dense and es == [-1]:
            continue       # one segment: it writes the request's output itself
        assert -1 not in es
        assert es == list(range(es[0], es[0] + len(es)))     # consecutive, in stream order
        assert not seen & set(es)
        seen |= set(es)


@pytest.mark.parametrize("seed", range(6))
def test_even_partitions(gk, seed):
    """Sequential cascade and flat partitions of random batches."""
    rnd = random.Random(seed)
    pool = gk.gk_pool_create(1, 32, 8, 128, 40000, 1 << 20, 16, 0)
    try:
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SEQUENTIAL)
        prefixes = {lp: gk.gk_prefix_alloc(pool, lp) for lp in (300, 2000)}
        bases, lps, slens = [], [], []
        for _ in range(rnd.randint(1, 90)):
            lp = rnd.choice([300, 2000, 0])
            bases.append(prefixes[lp] if lp else -1)
            lps.append(lp)
            slens.append(rnd.choice([0, rnd.randint(1, 40), rnd.randint(1, rnd.choice([200, 3000]))]))
        _, plan = _plan(gk, pool, bases, lps, slens)
        s = gk.gk_plan_info(plan)
        for dense in (False, True):
            lengths = [lp + sl for lp, sl in zip(lps, slens)] if dense else list(slens)
            total = sum(lengths)
            begin, segs = gk.gk_plan_segments(plan, dense)
            ctas = len(begin) - 1
            assert ctas == odisp.gather_ctas(total, SMS) == s["dense_ctas" if dense else "suffix_ctas"]
            _check_cover(begin, segs, lengths)
            _check_entries(segs, dense)
            if ctas:
                quota = -(-max(-(-total // SMS), 64) // 16) * 16
                t = _tokens(begin, segs)
                assert t[:-1] == [quota] * (ctas - 1) and 0 < t[-1] <= quota
        gk.gk_plan_destroy(plan)
    finally:
        gk.gk_pool_destroy(pool)


@pytest.mark.parametrize("C", [0, 16, 32])
def test_split_partition(gk, C):
    """Split plan, one group of 64 requests (Lp 16384, 1000 suffix tokens each):
    one slot per SM, slot ends on multiples of 16, prefix slots no larger than the others."""
    pool = gk.gk_pool_create(1, 32, 8, 128, 16384 + 16, 64 * 1000 + 64, 1, 0)
    try:
        base = gk.gk_prefix_alloc(pool, 16384)
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SPLIT, C)
        _, plan = _plan(gk, pool, [base] * 64, [16384] * 64, [1000] * 64)
        s = gk.gk_plan_info(plan)
        assert s["cascade_split"] == 1 and s["suffix_ctas"] == SMS
        n_pre = s["prefix_ctas"]
        begin, segs = gk.gk_plan_segments(plan, False)
        _check_cover(begin, segs, [1000] * 64)
        _check_entries(segs, False)
        t = _tokens(begin, segs)
        ends = np.cumsum(t)
        assert all(e % 16 == 0 for e in ends[:-1]) and ends[-1] == 64000
        assert max(t[:n_pre]) <= min(t[n_pre:-1])
        assert max(t[n_pre:-1]) - min(t[n_pre:-1]) <= 16
        # partial states: one per (request, key split) and one per suffix segment
        splits = -(-128 // s["prefix_tiles_per_item"])
        assert s["num_partials"] == 64 * splits + len(segs)
        gk.gk_plan_destroy(plan)
    finally:
        gk.gk_pool_destroy(pool)


def test_segments_argument_errors(gk):
    import ctypes
    with pytest.raises(gk.GkError):
        gk._check(gk.lib().gk_plan_segments(None, 0, ctypes.byref(ctypes.c_int32()), ctypes.byref(ctypes.c_int32()),
                                            None, None))


def test_aot_splits_worked_example():
    """Tangram Algorithm 1 by hand: budgets 10, 7, 3 (and an empty request) over 4 CTAs:
    Omega = 20, tau = 5, S = ceil(10/5), ceil(7/5), ceil(3/5) = 2, 2, 1."""
    assert odisp.aot_splits([10, 0, 7, 3], 4) == [2, 0, 2, 1]
    assert odisp.aot_segments([10, 0, 7, 3], 4) == [(0, 0, 5), (0, 5, 10), (2, 0, 4), (2, 4, 7), (3, 0, 3)]
    # tau never drops below one token: more CTAs than tokens gives one split per token at most
    assert odisp.aot_splits([2, 1], 100) == [2, 1]
    assert odisp.aot_splits([0, 0], 8) == [0, 0]


@pytest.mark.parametrize("seed", range(4))
def test_per_request_partition_matches_algorithm_1(gk, seed):
    """GK_PARTITION_PER_REQUEST: one segment per CTA, exactly the oracle's Algorithm-1 pieces,
    for the flat partition and a sequential plan's suffix partition."""
    rnd = random.Random(100 + seed)
    pool = gk.gk_pool_create(1, 32, 8, 128, 40000, 1 << 20, 16, 0)
    try:
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SEQUENTIAL)
        gk.gk_pool_set_gather_partition(pool, gk.GK_PARTITION_PER_REQUEST)
        prefixes = {lp: gk.gk_prefix_alloc(pool, lp) for lp in (300, 2000)}
        bases, lps, slens = [], [], []
        for _ in range(rnd.randint(1, 200)):
            lp = rnd.choice([300, 2000, 0])
            bases.append(prefixes[lp] if lp else -1)
            lps.append(lp)
            slens.append(rnd.choice([0, rnd.randint(1, 40), rnd.randint(1, 5000)]))
        _, plan = _plan(gk, pool, bases, lps, slens)
        for dense in (False, True):
            lengths = [lp + sl for lp, sl in zip(lps, slens)] if dense else list(slens)
            begin, segs = gk.gk_plan_segments(plan, dense)
            want = odisp.aot_segments(lengths, SMS)
            assert [tuple(x) for x in segs[:, :3].tolist()] == want
            assert begin.tolist() == list(range(len(want) + 1))      # one segment per CTA
            _check_cover(begin, segs, lengths)
            _check_entries(segs, dense)
        gk.gk_plan_destroy(plan)
        with pytest.raises(gk.GkError):
            gk.gk_pool_set_gather_partition(pool, 7)
    finally:
        gk.gk_pool_destroy(pool)


def test_split_slots_follow_each_item(gk):
    """Split plan over two HOT groups whose items differ in length: the gather slot of each
    prefix CTA is sized to when its own item ends (gk_plan_build, split arrangement).
    Groups: 64 requests on a 16384-token prefix (128 key tiles) and 64 on a 4096-token one
    (32 tiles), g = 4 (one 256-row block per KV head), 1000 suffix tokens each; forced split
    with 48 tiles per item, which the planner balances to 43 (the fewest tiles giving as
    many items): items of 43, 43, 42 tiles (group 1) and 32 tiles (group 2), 8 KV heads
    each, longest first.  Tile 1 us, item 5 us beside the gather, 50 GB/s per SM,
    gather-only CTAs starting at 4 us and prefix CTAs 4 us after their items, at the same
    rate.  The common end T solves
    120 (T - 4) + 16 (T - 52) + 8 (T - 51) + 8 (T - 41) = S / 50 GB/s, and a CTA's slot
    weighs (T - start) / (T - 4); slot ends are the weighted shares of the token stream
    rounded to 16 tokens."""
    cm = dict(c_flat_us=5.0, bw_flat_gbs=4000.0, c_cascade_us=10.0, bw_prefix_gbs=5000.0, bw_suffix_gbs=6000.0,
              c_merge_us=0.001, prefix_tile_us=1.0, prefix_item_us=5.0, gather_sm_gbs=50.0, c_gather_us=4.0,
              prefix_tile_split_us=1.0, warp_tile_us=1e3, warp_group_us=0.0, warp_item_us=1e3, warp_split_ratio=1.0,
              prefix_cta_ramp_us=4.0, prefix_cta_gather_ratio=1.0, c_merge_state_us=0.0, prefix_item_split_us=5.0,
              warp_item_split_us=1e3, prefix_item_crowd_us=0.0, split_gather_ratio_tensor=1.0, c_gather_split_us=4.0,
              split_tensor_us=0.0)
    import json
    pool = gk.gk_pool_create(1, 32, 8, 128, 16384 + 4096 + 32, 128 * 1000 + 64, 1, 0)
    try:
        gk.gk_cost_model_load(pool, json.dumps(cm))
        gk.gk_pool_set_prefix_kernel(pool, gk.GK_PREFIX_TENSOR)
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SPLIT, 48)
        a, b = gk.gk_prefix_alloc(pool, 16384), gk.gk_prefix_alloc(pool, 4096)
        bases = [a] * 64 + [b] * 64
        lps = [16384] * 64 + [4096] * 64
        slens = [1000] * 128
        _, plan = _plan(gk, pool, bases, lps, slens)
        s = gk.gk_plan_info(plan)
        assert (s["cascade_split"], s["prefix_ctas"], s["prefix_ctas_gather"], s["suffix_ctas"]) == (1, 32, 1, SMS)
        assert s["prefix_tiles_per_item"] == 43
        begin, segs = gk.gk_plan_segments(plan, False)
        _check_cover(begin, segs, slens)
        _check_entries(segs, False)
        got = _tokens(begin, segs)
        gk.gk_plan_destroy(plan)
    finally:
        gk.gk_pool_destroy(pool)
    S_us = 128 * 1000 * 4096 / 50e3                  # the gather in SM-us at 50 GB/s
    T = (S_us + 120 * 4 + 16 * 52 + 8 * 51 + 8 * 41) / 152
    assert abs(T - 82.4590) < 1e-3
    w = [(T - 52) / (T - 4)] * 16 + [(T - 51) / (T - 4)] * 8 + [(T - 41) / (T - 4)] * 8 + [1.0] * 120
    total, acc, ends = 128000, 0.0, []
    for x in w:
        acc += x
        e = int(total * acc / sum(w) + 0.5)
        e = (e + 8) // 16 * 16
        ends.append(min(total, max(e, ends[-1] if ends else 0)))
    ends[-1] = total
    want = np.diff([0] + ends).tolist()
    assert got == want
    # shorter items, longer gathers: about 0.39 and 0.53 of a gather-only CTA's share
    assert 0.37 < np.mean(got[:16]) / np.mean(got[32:]) < 0.41 and 0.51 < np.mean(got[24:32]) / np.mean(got[32:]) < 0.55


def test_split_slots_follow_sm_speeds(gk):
    """With per-SM speeds set (gk_pool_set_sm_speeds), a split plan's slots are planned per
    SM: the slowest SMs take the prefix items and every gather-only slot's tokens follow
    its SM's speed.  Same case as the per-item test with every item of one length (C = 32:
    32 items on the 16384-token group, 8 on the 4096-token one, 40 prefix slots); speeds
    1 + 0.05 (s mod 9) - 0.2 [s mod 7 == 0], normalised to mean 1.  Without speeds the
    plan is the one CTA b takes slot b of."""
    import json
    cm = dict(c_flat_us=5.0, bw_flat_gbs=4000.0, c_cascade_us=10.0, bw_prefix_gbs=5000.0, bw_suffix_gbs=6000.0,
              c_merge_us=0.001, prefix_tile_us=1.0, prefix_item_us=5.0, gather_sm_gbs=50.0, c_gather_us=4.0,
              prefix_tile_split_us=1.0, warp_tile_us=1e3, warp_group_us=0.0, warp_item_us=1e3, warp_split_ratio=1.0,
              prefix_cta_ramp_us=4.0, prefix_cta_gather_ratio=1.0, c_merge_state_us=0.0, prefix_item_split_us=5.0,
              warp_item_split_us=1e3, prefix_item_crowd_us=0.0, split_gather_ratio_tensor=1.0, c_gather_split_us=4.0,
              split_tensor_us=0.0)
    sp = np.array([1 + 0.05 * (s % 9) - (0.2 if s % 7 == 0 else 0.0) for s in range(SMS)], np.float32)
    pool = gk.gk_pool_create(1, 32, 8, 128, 16384 + 4096 + 32, 128 * 1000 + 64, 1, 0)
    try:
        gk.gk_cost_model_load(pool, json.dumps(cm))
        gk.gk_pool_set_prefix_kernel(pool, gk.GK_PREFIX_TENSOR)
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SPLIT, 32)
        a, b = gk.gk_prefix_alloc(pool, 16384), gk.gk_prefix_alloc(pool, 4096)
        bases, lps, slens = [a] * 64 + [b] * 64, [16384] * 64 + [4096] * 64, [1000] * 128
        with pytest.raises(gk.GkError):
            gk.gk_pool_set_sm_speeds(pool, sp[:100])
        with pytest.raises(gk.GkError):
            gk.gk_pool_set_sm_speeds(pool, np.where(np.arange(SMS) == 3, -1.0, sp))
        assert len(gk.gk_pool_get_sm_speeds(pool)) == 0
        _, plan = _plan(gk, pool, bases, lps, slens)
        s0 = gk.gk_plan_info(plan)
        t0 = _tokens(*gk.gk_plan_segments(plan, False))
        gk.gk_plan_destroy(plan)
        gk.gk_pool_set_sm_speeds(pool, sp)
        got = gk.gk_pool_get_sm_speeds(pool)
        assert np.allclose(got, sp * SMS / sp.sum(), rtol=1e-6) and abs(got.mean() - 1) < 1e-6
        _, plan = _plan(gk, pool, bases, lps, slens)
        s = gk.gk_plan_info(plan)
        begin, segs = gk.gk_plan_segments(plan, False)
        _check_cover(begin, segs, slens)
        _check_entries(segs, False)
        t = _tokens(begin, segs)
        gk.gk_plan_destroy(plan)
        gk.gk_pool_set_sm_speeds(pool, None)
        _, plan = _plan(gk, pool, bases, lps, slens)
        t2 = _tokens(*gk.gk_plan_segments(plan, False))
        assert gk.gk_plan_info(plan)["sm_slots"] == 0 and t2 == t0
        gk.gk_plan_destroy(plan)
    finally:
        gk.gk_pool_destroy(pool)
    assert s0["sm_slots"] == 0 and s["sm_slots"] == 1
    n_pre = s["prefix_ctas"]
    assert n_pre == s0["prefix_ctas"] == 40 and s["prefix_ctas_gather"] == 1
    # slots in order of SM speed: the n_pre slowest take the items, all of 37 us (start 41 us);
    # the common end T solves  sum_gather-only v (T - 4) + sum_prefix v (T - 41) = S / 50 GB/s
    v = np.sort(got.astype(np.float64))
    W = 128 * 1000 * 4096 / 50e3
    T = (W + 4 * v[n_pre:].sum() + 41 * v[:n_pre].sum()) / v.sum()
    w = np.concatenate([v[:n_pre] * (T - 41) / (T - 4), v[n_pre:]])
    total, acc, ends = 128000, 0.0, []
    for x in w:
        acc += x
        e = int(total * acc / w.sum() + 0.5)
        e = (e + 8) // 16 * 16
        ends.append(min(total, max(e, ends[-1] if ends else 0)))
    ends[-1] = total
    assert t == np.diff([0] + ends).tolist()
