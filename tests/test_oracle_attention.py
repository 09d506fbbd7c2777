"""Pins of the fp64 attention oracle and the Eq. 1 merge (CPU).

Each test checks the oracle against something other than itself: brute force in
50-digit arithmetic without the max shift, closed forms, the merge identity of
GraniKV Eq. 1, and invariances a wrong index or operand would break.
"""
import math

import numpy as np
import pytest

from oracle import attention

mpmath = pytest.importorskip("mpmath")


def _brute(q, k, v, scale):
    """Direct ratio of sums, 50 digits, no max subtraction."""
    mpmath.mp.dps = 50
    rows, d = q.shape
    n = k.shape[0]
    O = np.zeros((rows, d))
    L = np.zeros(rows)
    for r in range(rows):
        e = [mpmath.exp(mpmath.fsum(mpmath.mpf(float(q[r, j])) * mpmath.mpf(float(k[i, j])) for j in range(d)) * mpmath.mpf(scale))
             for i in range(n)]
        z = mpmath.fsum(e)
        for j in range(d):
            O[r, j] = float(mpmath.fsum(e[i] * mpmath.mpf(float(v[i, j])) for i in range(n)) / z)
        L[r] = float(mpmath.log(z))
    return O, L


@pytest.mark.parametrize("n,d,g", [(1, 4, 1), (3, 8, 2), (8, 16, 3), (5, 64, 4)])
def test_brute_force_tiny(n, d, g):
    rng = np.random.default_rng(n * 100 + d)
    q = rng.standard_normal((g, d)) * 2
    k = rng.standard_normal((1, n, d))
    v = rng.standard_normal((1, n, d))
    o, lse = attention.attend_heads(q, k, v)
    ob, lb = _brute(q, k[0], v[0], 1.0 / math.sqrt(d))
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lb, rtol=1e-13, atol=1e-13)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((2, 16))
    k = rng.standard_normal((1, 1, 16))
    v = rng.standard_normal((1, 1, 16))
    o, lse = attention.attend_heads(q, k, v)
    np.testing.assert_array_equal(o, np.repeat(v[0], 2, axis=0))
    np.testing.assert_allclose(lse, q @ k[0, 0] / 4.0, rtol=1e-15)


def test_zero_query_is_mean_and_log_n():
    rng = np.random.default_rng(2)
    n, d = 37, 32
    k = rng.standard_normal((1, n, d))
    v = rng.standard_normal((1, n, d))
    o, lse = attention.attend_heads(np.zeros((1, d)), k, v)
    np.testing.assert_allclose(o[0], v[0].mean(axis=0), rtol=1e-13, atol=1e-15)
    assert abs(lse[0] - math.log(n)) < 1e-14


def test_identical_keys_give_mean_and_shifted_lse():
    rng = np.random.default_rng(3)
    n, d = 11, 8
    key = rng.standard_normal(d)
    k = np.tile(key, (1, n, 1))
    v = rng.standard_normal((1, n, d))
    q = rng.standard_normal((1, d))
    o, lse = attention.attend_heads(q, k, v)
    s = float(q[0] @ key) / math.sqrt(d)
    np.testing.assert_allclose(o[0], v[0].mean(axis=0), rtol=1e-13, atol=1e-15)
    assert abs(lse[0] - (s + math.log(n))) < 1e-13


def test_dominant_key_selects_its_value():
    d, n = 16, 9
    k = np.zeros((1, n, d))
    k[0, 4, 0] = 1000.0
    v = np.arange(n * d, dtype=np.float64).reshape(1, n, d)
    q = np.zeros((1, d))
    q[0, 0] = 4.0              # score 1000 for key 4, 0 for the rest (scale 1/4)
    o, lse = attention.attend_heads(q, k, v)
    np.testing.assert_allclose(o[0], v[0, 4], rtol=1e-15)
    assert abs(lse[0] - 1000.0) < 1e-12


def test_scale_is_inverse_sqrt_d():
    # two keys: a*e1 and 0 with values 1 and 0 -> O = sigmoid(a / sqrt(d))
    for d in (16, 64, 128):
        a = 3.0
        k = np.zeros((1, 2, d))
        k[0, 0, 0] = a
        v = np.zeros((1, 2, d))
        v[0, 0, :] = 1.0
        q = np.zeros((1, d))
        q[0, 0] = 1.0
        o, lse = attention.attend_heads(q, k, v)
        x = a / math.sqrt(d)
        assert abs(o[0, 0] - 1.0 / (1.0 + math.exp(-x))) < 1e-15
        assert abs(lse[0] - math.log(math.exp(x) + 1.0)) < 1e-15


def test_gqa_head_mapping():
    rng = np.random.default_rng(4)
    hkv, g, n, d = 3, 2, 7, 8
    q = rng.standard_normal((hkv * g, d))
    k = rng.standard_normal((hkv, n, d))
    v = rng.standard_normal((hkv, n, d))
    o, lse = attention.attend_heads(q, k, v)
    for qh in range(hkv * g):
        h = qh // g
        o1, l1 = attention.attend_heads(q[qh:qh + 1], k[h:h + 1], v[h:h + 1])
        np.testing.assert_array_equal(o[qh], o1[0])
        assert lse[qh] == l1[0]


def test_key_order_invariance():
    rng = np.random.default_rng(5)
    n, d = 50, 32
    q = rng.standard_normal((4, d))
    k = rng.standard_normal((1, n, d))
    v = rng.standard_normal((1, n, d))
    perm = rng.permutation(n)
    o1, l1 = attention.attend_heads(q, k, v)
    o2, l2 = attention.attend_heads(q, k[:, perm], v[:, perm])
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


@pytest.mark.parametrize("split", [1, 17, 63])
def test_eq1_merge_equals_flat_over_concatenation(split):
    rng = np.random.default_rng(6 + split)
    n, d, hkv, g = 64, 32, 2, 3
    q = rng.standard_normal((hkv * g, d)) * 3
    k = rng.standard_normal((hkv, n, d))
    v = rng.standard_normal((hkv, n, d))
    flat = attention.attend_heads(q, k, v)
    pre = attention.attend_heads(q, k[:, :split], v[:, :split])
    suf = attention.attend_heads(q, k[:, split:], v[:, split:])
    o, lse = attention.merge([pre, suf])
    np.testing.assert_allclose(o, flat[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, flat[1], rtol=1e-13, atol=1e-13)
    # three-way split, merged in either grouping
    a, b = split // 2, split
    s1 = attention.attend_heads(q, k[:, :a], v[:, :a]) if a else None
    s2 = attention.attend_heads(q, k[:, a:b], v[:, a:b])
    s3 = attention.attend_heads(q, k[:, b:], v[:, b:])
    parts = [s for s in (s1, s2, s3) if s is not None]
    o3, l3 = attention.merge(parts)
    np.testing.assert_allclose(o3, flat[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l3, flat[1], rtol=1e-13, atol=1e-13)


def test_empty_side_merges_to_the_other():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((2, 8))
    k = rng.standard_normal((1, 5, 8))
    v = rng.standard_normal((1, 5, 8))
    full = attention.attend_heads(q, k, v)
    empty = attention.attend_heads(q, k[:, :0], v[:, :0])
    assert np.all(empty[0] == 0) and np.all(np.isneginf(empty[1]))
    o, lse = attention.merge([empty, full])
    np.testing.assert_array_equal(o, full[0])
    np.testing.assert_array_equal(lse, full[1])
    o, lse = attention.merge([empty, empty])
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_merge_weights_by_exp_lse_difference():
    # Eq. 1 closed form with two hand-set states
    o1 = np.array([[1.0, 0.0]])
    o2 = np.array([[0.0, 1.0]])
    l1 = np.array([math.log(3.0)])
    l2 = np.array([math.log(1.0)])
    o, lse = attention.merge([(o1, l1), (o2, l2)])
    np.testing.assert_allclose(o, [[0.75, 0.25]], rtol=1e-15)
    assert abs(lse[0] - math.log(4.0)) < 1e-15
