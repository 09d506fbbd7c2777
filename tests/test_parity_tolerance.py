"""The parity bounds discriminate: mistakes planted in the oracle (on the CPU)
must fail them at the configs' context lengths, while bf16 rounding of the
probabilities (what the tensor-core path does) must pass."""
import numpy as np
import pytest

from oracle import attention
from synth import gen
from parity import attention_ok

Lp, S, HKV, G, D = 16384, 1152, 8, 4, 128


@pytest.fixture(scope="module")
def ctx():
    n = (Lp + S) * HKV * D
    k = gen.bf16_bits_to_f64(gen.normal_bits(gen.stream_key(99, 1), 0, n)).reshape(Lp + S, HKV, D).transpose(1, 0, 2)
    v = gen.bf16_bits_to_f64(gen.normal_bits(gen.stream_key(99, 2), 0, n)).reshape(Lp + S, HKV, D).transpose(1, 0, 2)
    q = gen.bf16_bits_to_f64(gen.normal_bits(gen.stream_key(99, 3), 0, HKV * G * D)).reshape(HKV * G, D)
    return q, np.ascontiguousarray(k), np.ascontiguousarray(v)


def _true(ctx, qscale=1.0):
    q, k, v = ctx
    return attention.attend_heads(q * qscale, k, v)


@pytest.mark.parametrize("qscale", [1.0, 8.0])
def test_drop_suffix_fails(ctx, qscale):
    q, k, v = ctx
    ref = _true(ctx, qscale)
    bad = attention.attend_heads(q * qscale, k[:, :Lp], v[:, :Lp])
    assert not attention_ok(*bad, *ref)[0]


@pytest.mark.parametrize("qscale", [1.0])
def test_drop_one_prefix_tile_fails(ctx, qscale):
    """Diffuse softmax: a missing 128-key tile shifts every row (the peaked
    variant hides it unless the tile holds a row's top key)."""
    q, k, v = ctx
    ref = _true(ctx, qscale)
    keep = np.r_[0:4096, 4096 + 128:Lp + S]
    bad = attention.attend_heads(q * qscale, k[:, keep], v[:, keep])
    assert not attention_ok(*bad, *ref)[0]


def test_off_by_one_slot_in_permuted_pool_fails(ctx):
    """In a shuffled COLD pool, slot + 1 holds an unrelated token: the suffix
    then reads other data."""
    q, k, v = ctx
    ref = _true(ctx)
    n = S * HKV * D
    ko = gen.bf16_bits_to_f64(gen.normal_bits(gen.stream_key(98, 1), 0, n)).reshape(S, HKV, D).transpose(1, 0, 2)
    vo = gen.bf16_bits_to_f64(gen.normal_bits(gen.stream_key(98, 2), 0, n)).reshape(S, HKV, D).transpose(1, 0, 2)
    bad = attention.attend_heads(q, np.concatenate([k[:, :Lp], ko], 1), np.concatenate([v[:, :Lp], vo], 1))
    assert not attention_ok(*bad, *ref)[0]


def test_value_paired_with_neighbour_key_fails(ctx):
    q, k, v = ctx
    ref = _true(ctx, 8.0)
    idx = np.r_[1:Lp + S, 0]
    bad = attention.attend_heads(q * 8.0, k, v[:, idx])
    assert not attention_ok(*bad, *ref)[0]


def test_wrong_scale_fails(ctx):
    q, k, v = ctx
    ref = _true(ctx)
    bad = attention.attend_heads(q, k, v, scale=1.0 / 128)
    assert not attention_ok(*bad, *ref)[0]


def test_bf16_probability_rounding_passes(ctx):
    """A plain restatement with P rounded to bf16 before PV stays inside the bounds."""
    q, k, v = ctx
    for qscale in (1.0, 8.0):
        ref = _true(ctx, qscale)
        O = np.empty_like(ref[0])
        L = np.empty_like(ref[1])
        for r in range(HKV * G):
            s = (k[r // G] @ (q[r] * qscale)) / np.sqrt(D)
            m = s.max()
            p = np.exp(s - m).astype(np.float32)
            p = gen.bf16_bits_to_f64(gen._f32_to_bf16_bits(p))
            O[r] = (p @ v[r // G]) / p.sum()
            L[r] = m + np.log(p.sum())
        ok, e = attention_ok(O, L, *ref)
        assert ok, e
