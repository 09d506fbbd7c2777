"""The oracle's physical pool path (block manager + scatter + gather) against its
logical context, and GraniKV Appendix B.6's page-size invariance (CPU)."""
import numpy as np
import pytest

from oracle import attention, reference
from oracle.pool_model import build_pool
from synth import gen, workloads


def _gathered(w, pm, bases, seqs, layer, appended):
    out = []
    for r, req in enumerate(w.requests):
        lp = w.prefix_len(r)
        base = bases[req.prefix] if req.prefix >= 0 else 0
        out.append(pm.gather(layer, base, lp, seqs[r].table, req.suffix_len + appended))
    return out


def _logical(w, layer, appended):
    cache = reference.ContextCache(w)
    return [reference.context(w, r, layer, appended, cache) for r in range(w.B)]


@pytest.mark.parametrize("cold_seed,P", [(0, 1), (11, 1), (3, 4), (5, 16)])
def test_config1_gather_matches_logical_context(cold_seed, P):
    w = workloads.config(1)
    pm, bases, seqs, bp = build_pool(w, cold_seed=cold_seed, page_size=P)
    logical = _logical(w, 0, 0)
    for (K, V), (Kl, Vl) in zip(_gathered(w, pm, bases, seqs, 0, 0), logical):
        np.testing.assert_array_equal(gen.bf16_bits_to_f64(K), Kl)
        np.testing.assert_array_equal(gen.bf16_bits_to_f64(V), Vl)


def _small_fork_workload(P):
    return workloads.config(5, n_parent=3, children=4, Lp=32, suffix_range=(20, 40), steps=5,
                            page_size=P, L=2, Hq=4, Hkv=2, d=16)


@pytest.mark.parametrize("P", [1, 4, 16])
def test_fork_cow_steps_match_logical_context(P):
    w = _small_fork_workload(P)
    pm, bases, seqs, bp = build_pool(w, steps=w.steps)
    for layer in range(w.L):
        for (K, V), (Kl, Vl) in zip(_gathered(w, pm, bases, seqs, layer, w.steps), _logical(w, layer, w.steps)):
            np.testing.assert_array_equal(gen.bf16_bits_to_f64(K), Kl)
            np.testing.assert_array_equal(gen.bf16_bits_to_f64(V), Vl)


def test_page_size_and_permutation_invariance_bit_identical():
    outs = []
    for P, seed in [(1, 0), (1, 77), (4, 5), (16, 9)]:
        w = _small_fork_workload(P)
        pm, bases, seqs, bp = build_pool(w, cold_seed=seed, steps=w.steps)
        q = reference.q_bits(w, 1, 0)
        res = []
        for r, (K, V) in enumerate(_gathered(w, pm, bases, seqs, 1, w.steps)):
            res.append(attention.attend_heads(gen.bf16_bits_to_f64(q[r]), gen.bf16_bits_to_f64(K),
                                              gen.bf16_bits_to_f64(V)))
        outs.append(res)
    for other in outs[1:]:
        for (o1, l1), (o2, l2) in zip(outs[0], other):
            np.testing.assert_array_equal(o1, o2)
            np.testing.assert_array_equal(l1, l2)


def test_cow_copies_happen_only_on_shared_partial_blocks():
    w = _small_fork_workload(16)
    pm, bases, seqs, bp = build_pool(w, steps=1)
    # every parent had a partial last block shared 4 ways: 3 of 4 children copy
    partial = sum(1 for s in w.parents if s % 16)
    w1 = _small_fork_workload(1)
    _, _, seqs1, bp1 = build_pool(w1, steps=1)
    assert bp1.num_free() == bp1.n - sum(w1.parents) - w1.B
    used16 = bp.n - bp.num_free()
    full16 = sum(-(-s // 16) for s in w.parents)
    assert used16 == full16 + 3 * partial + sum(1 for s in w.parents if s % 16 == 0) * 4
