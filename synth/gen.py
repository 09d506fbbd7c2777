"""Seeded, counter-based synthetic inputs shared by the oracle, the tests and the bench.

This module draws numbers; it holds none of the attention or block-manager
arithmetic.  Every value is a pure function of (seed, stream ids, element
index), so the host (numpy, here) and the device (``synth/fill.cu``) produce the
same bits, and the oracle can regenerate any K/V/Q element without reading the
device.

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014).  Output n (n >= 1) of a splitmix64 stream
whose state starts at ``s`` is ``mix64(s + n * GAMMA)``.

Normal draws: a 65,536-entry quantile table, entry i = the standard normal
inverse CDF at (i + 1/2) / 65536 computed in fp64, rounded to fp32 and then to
bf16 (both round-to-nearest-even).  A draw takes the top 16 bits of one
splitmix64 output as the table index.
"""
from __future__ import annotations

import math
import statistics
from functools import lru_cache

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1

# Stream kinds (first id of every tensor stream).
KIND_PREFIX_K = 1
KIND_PREFIX_V = 2
KIND_SUFFIX_K = 3
KIND_SUFFIX_V = 4
KIND_Q = 5
KIND_NEW_K = 6
KIND_NEW_V = 7
KIND_LENGTHS = 8


def mix64(z: int) -> int:
    """splitmix64 output finaliser on a Python int (exact 64-bit arithmetic)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, *ids: int) -> int:
    """Key of a stream: chain one splitmix64 step per id, starting from the seed."""
    k = seed & MASK64
    for i in ids:
        k = mix64(k + ((i + 1) * GAMMA))
    return k


class SplitMix64:
    """Sequential splitmix64 stream (used for lengths and permutation-free draws)."""

    def __init__(self, state: int):
        self.state = state & MASK64

    def next(self) -> int:
        self.state = (self.state + GAMMA) & MASK64
        return mix64(self.state)

    def uniform_int(self, lo: int, hi: int) -> int:
        """Uniform integer in [lo, hi], both ends included: lo + floor(u * n / 2^64)."""
        n = hi - lo + 1
        return lo + ((self.next() * n) >> 64)

    def unit(self) -> float:
        """Uniform in [0, 1) with 53 random bits."""
        return (self.next() >> 11) * (1.0 / (1 << 53))


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


@lru_cache(maxsize=1)
def normal_table_bits() -> np.ndarray:
    """uint16 [65536]: bf16 bits of the normal quantile at (i + 1/2) / 65536."""
    nd = statistics.NormalDist()
    vals = np.array([nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)], dtype=np.float64)
    return _f32_to_bf16_bits(vals)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


_U64 = np.uint64


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> _U64(30))) * _U64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> _U64(27))) * _U64(0x94D049BB133111EB)
    return z ^ (z >> _U64(31))


def normal_bits(key: int, offset: int, count: int) -> np.ndarray:
    """bf16 bits of elements [offset, offset + count) of the stream with this key."""
    out = np.empty(count, dtype=np.uint16)
    table = normal_table_bits()
    chunk = 1 << 22
    with np.errstate(over="ignore"):
        for c0 in range(0, count, chunk):
            c1 = min(count, c0 + chunk)
            n = np.arange(offset + c0 + 1, offset + c1 + 1, dtype=_U64)
            z = _U64(key) + n * _U64(GAMMA)
            out[c0:c1] = table[(_mix64_np(z) >> _U64(48)).astype(np.int64)]
    return out


def scale_bf16_bits_pow2(bits: np.ndarray, log2_scale: int) -> np.ndarray:
    """Multiply bf16 values by 2**log2_scale exactly (exponent shift; no zero/inf/nan in the table)."""
    if log2_scale == 0:
        return bits
    b = bits.astype(np.int32)
    return (b + (log2_scale << 7)).astype(np.uint16)


def log_uniform_int(rng: SplitMix64, lo: int, hi: int) -> int:
    """round(exp(U(ln lo, ln hi)))."""
    u = rng.unit()
    return int(round(math.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))))
