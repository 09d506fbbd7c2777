"""Pins of the oracle block manager: the page's worked example, its slot formula,
randomised refcount invariants, and the seeded initial order (CPU)."""
import random
from collections import Counter

import pytest

from conftest import golden
from oracle.block_manager import BlockPool, Seq, initial_order, slot_of


def test_worked_example_printed_and_derived():
    g = golden("paged_kv_worked_example.json")
    pr, dv = g["printed"], g["derived"]
    pool = BlockPool(pr["pool_blocks"], pr["block_size"])
    a = Seq()
    for _ in range(pr["prompt_tokens"]):
        assert pool.append(a) is not None
    assert (len(a.table), pool.num_free()) == (pr["after_prompt"]["table_len"], pr["after_prompt"]["num_free"])
    b = pool.fork(a)
    slot, cow = pool.append(b)
    assert (cow is not None) == pr["child_first_append_copies"]
    assert (b.table[0] == a.table[0]) == pr["child_table0_equals_parent_table0"]
    assert (b.table[1] != a.table[1]) == pr["child_table1_differs_from_parent_table1"]
    assert a.table == dv["parent_table"] and b.table == dv["child_table"]
    assert list(cow) == dv["cow_pair"] and slot == dv["child_slot"]
    pool.release(a)
    pool.release(b)
    assert pool.num_free() == pr["after_release_both"]["num_free"]


def test_slot_formula_on_illustrated_tables():
    g = golden("paged_kv_slot_formula.json")
    P = g["block_size"]
    for name, t, want in g["slots"]:
        assert slot_of(g["tables"][name], P, t) == want
    for lo, hi, blk in g["printed_ranges"]["A"]:
        for t in range(lo, hi + 1):
            assert slot_of(g["tables"]["A"], P, t) // P == blk


def test_append_slots_follow_the_formula():
    pool = BlockPool(64, 4, seed=9)
    s = Seq()
    slots = [pool.append(s)[0] for _ in range(30)]
    assert slots == [slot_of(s.table, 4, t) for t in range(30)]
    assert len(s.table) == 8


def test_out_of_blocks_changes_nothing():
    pool = BlockPool(2, 4)
    a = Seq()
    for _ in range(8):
        assert pool.append(a) is not None
    assert pool.append(a) is None
    assert a.len == 8 and len(a.table) == 2 and pool.num_free() == 0
    # a COW that cannot get a block also changes nothing
    pool2 = BlockPool(1, 4)
    p = Seq()
    pool2.append(p)
    c = pool2.fork(p)
    assert pool2.append(c) is None
    assert c.table == p.table and c.len == 1 and pool2.ref[p.table[0]] == 2


def test_shared_block_k_ways_first_k_minus_1_copy():
    pool = BlockPool(32, 16)
    parent = Seq()
    for _ in range(20):
        pool.append(parent)
    kids = [pool.fork(parent) for _ in range(4)]
    pool.release(parent)
    cows = [pool.append(k)[1] for k in kids]
    assert [c is not None for c in cows] == [True, True, True, False]
    assert kids[3].table[1] == 1 and len({k.table[1] for k in kids}) == 4


def _check_invariants(pool, seqs):
    holders = Counter(b for s in seqs for b in s.table)
    for b in range(pool.n):
        assert pool.ref[b] == holders.get(b, 0)
    assert len(pool.free) == len(set(pool.free))
    assert set(pool.free) == {b for b in range(pool.n) if pool.ref[b] == 0}
    for s in seqs:
        assert len(s.table) == -(-s.len // pool.P)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_random_fork_append_release_invariants(seed):
    rnd = random.Random(seed)
    P = rnd.choice([1, 4, 16])
    pool = BlockPool(200, P, seed=seed)
    seqs = [Seq()]
    for _ in range(3000):
        op = rnd.random()
        if op < 0.7 and seqs:
            s = rnd.choice(seqs)
            before = (list(s.table), s.len, list(pool.free))
            res = pool.append(s)
            if res is None:
                assert (s.table, s.len, pool.free) == before
        elif op < 0.8 and seqs:
            seqs.append(pool.fork(rnd.choice(seqs)))
        elif op < 0.9 and seqs:
            s = seqs.pop(rnd.randrange(len(seqs)))
            pool.release(s)
        else:
            seqs.append(Seq())
        _check_invariants(pool, seqs)
    for s in seqs:
        pool.release(s)
    assert pool.num_free() == pool.n and all(r == 0 for r in pool.ref)


def test_initial_order():
    assert initial_order(6, 0) == list(range(6))
    for seed in (1, 2, 12345):
        o = initial_order(1000, seed)
        assert sorted(o) == list(range(1000)) and o != list(range(1000))
    assert initial_order(1000, 5) == initial_order(1000, 5)
    pool = BlockPool(10, 1, seed=3)
    s = Seq()
    got = [pool.append(s)[0] for _ in range(10)]
    assert got == initial_order(10, 3)


def test_splitmix64_published_vector():
    from oracle.block_manager import _splitmix64_stream
    g = golden("splitmix64_vector.json")
    gen = _splitmix64_stream(g["seed"])
    assert [next(gen) for _ in range(5)] == [int(x) for x in g["outputs"]]
