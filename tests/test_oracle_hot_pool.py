"""Pins of the oracle HOT allocator: a hand-worked sequence and random properties (CPU)."""
import random

import pytest

from oracle.hot_pool import HotFull, HotPool


def test_hand_worked_sequence():
    h = HotPool(100)
    assert h.alloc(10) == 0
    assert h.alloc(20) == 10
    assert h.alloc(30) == 30
    h.release(10)
    assert h.free == [(10, 30)] and h.top == 60
    assert h.alloc(15) == 10                 # first fit reuses the freed range
    assert h.free == [(25, 30)]
    assert h.alloc(6) == 60                  # the 5-token hole is too small: bump
    h.release(30)                            # [30, 60) merges with [25, 30)
    assert h.free == [(25, 60)] and h.top == 66
    h.release(60)                            # [60, 66) merges and reaches the top
    assert h.free == [] and h.top == 25
    with pytest.raises(HotFull):
        h.alloc(80)
    assert h.alloc(75) == 25 and h.top == 100


def test_release_lowers_top_and_coalesces_both_sides():
    h = HotPool(64)
    bases = [h.alloc(8) for _ in range(8)]
    assert bases == list(range(0, 64, 8))
    h.release(8)
    h.release(24)
    h.release(16)                            # joins [8,16) and [24,32)
    assert h.free == [(8, 32)]
    h.release(56)
    assert h.top == 56
    h.release(48)
    h.release(40)
    h.release(32)                            # everything above 8 is free: top drops to 8
    assert h.free == [] and h.top == 8


@pytest.mark.parametrize("seed", range(4))
def test_random_properties(seed):
    rnd = random.Random(seed)
    cap = 5000
    h = HotPool(cap)
    live = {}
    for _ in range(2000):
        if live and rnd.random() < 0.45:
            b = rnd.choice(list(live))
            h.release(b)
            del live[b]
        else:
            n = rnd.randint(1, 400)
            try:
                b = h.alloc(n)
                live[b] = n
            except HotFull:
                # nothing fits: every free range and the bump tail are shorter than n
                assert all(y - x < n for x, y in h.free) and h.top + n > cap
        ranges = sorted((b, b + n) for b, n in live.items())
        for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
            assert a1 <= b0                   # no overlap
        assert all(0 <= a and b <= h.top for a, b in ranges)
        fr = h.free
        assert fr == sorted(fr)
        for (a0, a1), (b0, b1) in zip(fr, fr[1:]):
            assert a1 < b0                    # fully coalesced
        covered = sorted(ranges + fr)
        pos = 0
        for a, b in covered:
            assert a == pos
            pos = b
        assert pos == h.top                   # live + free tile [0, top) exactly
        assert not fr or fr[-1][1] < h.top
