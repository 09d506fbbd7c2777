"""Prefix caching on the host: COLD blocks keyed by chained token hashes ("Paged
KV cache", How it works, step 5) and HOT slabs reference counted with LRU
eviction (GraniKV Section 3.2).

Pins of the oracle against what the pages fix (a block is reused only with its
whole chain of parents, a cached block outlives its requests, eviction takes the
block or slab unused for longest, a freed HOT range merges with its
neighbours), then the library against the oracle, bit for bit, on random
request streams over pools small enough to evict and to run out."""
import random

import pytest

from oracle.block_manager import BlockPool, Seq, block_key
from oracle.hot_pool import HotFull, HotPool, HotPrefixCache


@pytest.fixture(scope="module")
def gk():
    from paged_kv_cache_pool_gb300 import build
    build.build()
    from paged_kv_cache_pool_gb300 import binding
    return binding


def _write(bp, s, n):
    for _ in range(n):
        assert bp.append(s) is not None


# ---- oracle pins --------------------------------------------------------------------
def test_oracle_reuses_whole_chains_only():
    P = 16
    bp = BlockPool(16, P)
    sys_prompt = list(range(100, 132))                     # two full blocks
    a = Seq()
    _write(bp, a, 40)
    assert bp.cache_blocks(a, sys_prompt + list(range(8))) == 2   # 40 tokens: two full blocks
    # the same 32 leading tokens: both blocks reused, nothing written
    b, n = bp.create_cached(sys_prompt + [7, 8, 9])
    assert n == 32 and b.table == a.table[:2] and bp.ref[a.table[0]] == 3   # a, the cache, b
    # first block equal, second differs in its first token: only block 0
    c, n = bp.create_cached(sys_prompt[:16] + [999] + sys_prompt[17:])
    assert n == 16 and c.table == a.table[:1]
    # second block equal but the first differs: the chain breaks at block 0
    d, n = bp.create_cached([5] + sys_prompt[1:])
    assert n == 0 and d.table == []
    # a block's key depends on its parent's
    assert block_key(0, sys_prompt[16:]) != block_key(block_key(0, sys_prompt[:16]), sys_prompt[16:])


def test_oracle_cached_blocks_outlive_requests_and_evict_lru():
    P = 4
    bp = BlockPool(4, P)
    x, y = Seq(), Seq()
    _write(bp, x, 8)                                       # blocks 0, 1
    _write(bp, y, 8)                                       # blocks 2, 3
    tx, ty = list(range(8)), list(range(50, 58))
    bp.cache_blocks(y, ty)                                 # y's blocks cached first (older)
    bp.cache_blocks(x, tx)
    bp.release(x)
    bp.release(y)
    assert bp.num_free() == 0 and bp.cache_stats() == (4, 4)   # all four survive, all evictable
    # reusing x's chain makes it the most recent; a new block must evict y's oldest block
    z, n = bp.create_cached(tx)
    assert n == 8 and z.table == [0, 1]
    w = Seq()
    assert bp.append(w) is not None and w.table == [2]     # y's first cached block (oldest) went
    assert bp.cache_stats() == (3, 1)                       # x's two blocks held by z, y's second evictable
    bp.release(z)
    assert bp.cache_stats() == (3, 3)


def test_oracle_hot_cache_reuse_and_lru_eviction_with_merging():
    hc = HotPrefixCache(HotPool(100))
    a, hit = hc.acquire(1, 30)
    assert (a, hit) == (0, False)
    assert hc.acquire(1, 30) == (0, True)
    b, _ = hc.acquire(2, 30)
    c, _ = hc.acquire(3, 30)
    assert (b, c) == (30, 60)
    hc.unref(2)                          # 2 idle (older)
    hc.unref(1)
    hc.unref(1)                          # 1 idle (newer)
    assert hc.stats() == (3, 2, 60)
    # 40 tokens fit nowhere (10 at the top): 2 is evicted first, then 1, whose range
    # merges with 2's into [0, 60)
    d, hit = hc.acquire(4, 40)
    assert (d, hit) == (0, False) and set(hc.slabs) == {3, 4}
    assert hc.pool.free == [(40, 60)]
    with pytest.raises(HotFull):
        hc.acquire(5, 50)                # only 3 and 4 left, both held


# ---- library against the oracle ------------------------------------------------------
@pytest.mark.parametrize("seed", range(6))
def test_cold_cache_bit_exact(gk, seed):
    rnd = random.Random(seed)
    P = rnd.choice([1, 4, 16])
    nb = rnd.choice([24, 60])
    pool = gk.gk_pool_create(1, 8, 2, 64, 100, nb * P, P, seed)
    ref = BlockPool(nb, P, seed)
    prompts = [[rnd.randint(0, 50000) for _ in range(rnd.randint(P, 4 * P + 3))] for _ in range(4)]
    live = []          # (oracle Seq, library id, tokens written so far)
    try:
        for step in range(400):
            op = rnd.random()
            if op < 0.3 or not live:
                toks = list(rnd.choice(prompts)) + [rnd.randint(0, 50000) for _ in range(rnd.randint(0, 2 * P))]
                s, n = ref.create_cached(toks)
                sid, n2 = gk.gk_seq_create_cached(pool, toks)
                assert n2 == n
                live.append([s, sid, toks])
                # write the rest of the prompt, then cache its full blocks
                ok = True
                for _ in range(len(toks) - n):
                    res = ref.append(s)
                    try:
                        gk.gk_seq_append_slots(pool, [sid])
                        assert res is not None
                    except gk.GkError as e:
                        assert e.status == gk.GK_ERR_OOM and res is None
                        ok = False
                        break
                if ok:
                    assert gk.gk_seq_cache_blocks(pool, sid, toks) == ref.cache_blocks(s, toks)
            elif op < 0.75:
                s, sid, _ = rnd.choice(live)
                res = ref.append(s)
                try:
                    gk.gk_seq_append_slots(pool, [sid])
                    assert res is not None
                except gk.GkError as e:
                    assert e.status == gk.GK_ERR_OOM and res is None
            else:
                s, sid, _ = live.pop(rnd.randrange(len(live)))
                ref.release(s)
                gk.gk_seq_release(pool, sid)
            for s, sid, _ in live:
                t, ln = gk.gk_seq_table(pool, sid)
                assert t.tolist() == s.table and ln == s.len, f"step {step}"
            assert gk.gk_cold_stats(pool)[0] == ref.num_free()
            assert gk.gk_cold_cache_stats(pool) == ref.cache_stats()
            assert [gk.gk_block_refcount(pool, b) for b in range(nb)] == ref.ref
    finally:
        gk.gk_pool_destroy(pool)


@pytest.mark.parametrize("seed", range(6))
def test_hot_cache_bit_exact(gk, seed):
    rnd = random.Random(seed)
    cap = rnd.choice([200, 500])
    pool = gk.gk_pool_create(1, 8, 2, 64, cap, 64, 1, 0)
    ref = HotPrefixCache(HotPool(cap))
    lens = {k: rnd.randint(10, cap // 3) for k in range(12)}
    held = []
    try:
        for _ in range(300):
            if held and rnd.random() < 0.45:
                k = held.pop(rnd.randrange(len(held)))
                ref.unref(k)
                gk.gk_prefix_unref(pool, k)
            else:
                k = rnd.randrange(12)
                try:
                    want = ref.acquire(k, lens[k])
                except HotFull:
                    want = None
                try:
                    got = gk.gk_prefix_acquire(pool, k, lens[k])
                except gk.GkError as e:
                    assert e.status == gk.GK_ERR_HOT_FULL
                    got = None
                assert got == want
                if got is not None:
                    held.append(k)
            assert gk.gk_hot_cache_stats(pool) == ref.stats()
            top, nfree, free_tok = gk.gk_hot_stats(pool)
            assert (top, nfree, free_tok) == (ref.pool.top, len(ref.pool.free), ref.pool.free_tokens())
    finally:
        gk.gk_pool_destroy(pool)


def test_cache_argument_errors(gk):
    pool = gk.gk_pool_create(1, 8, 2, 64, 100, 64, 1, 0)
    try:
        base, hit = gk.gk_prefix_acquire(pool, 7, 20)
        with pytest.raises(gk.GkError):
            gk.gk_prefix_acquire(pool, 7, 21)          # same key, another length
        with pytest.raises(gk.GkError):
            gk.gk_prefix_release(pool, base)           # held by the cache
        gk.gk_prefix_unref(pool, 7)
        with pytest.raises(gk.GkError):
            gk.gk_prefix_unref(pool, 7)                # no reference left
        with pytest.raises(gk.GkError):
            gk.gk_seq_cache_blocks(pool, 12345, [1, 2])
    finally:
        gk.gk_pool_destroy(pool)
