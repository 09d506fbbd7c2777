"""ORACLE (test infrastructure): expected attention outputs of a synthetic workload.

The context of request r at decode step t is its group's shared prefix (Lp
tokens) followed by its suffix: the tokens cached before step 0 (read from the
suffix stream of the sequence it was forked from, or its own) and the tokens
appended at steps 0..t (GraniKV Section 2.1: decode attends to all previous
tokens; configs with appends write the step's token before attention).  The
context is materialised explicitly from the seeded generator; no slot, table or
pool layout is involved here.

Q head qh uses KV head qh // g (consecutive query heads share a KV head), and
the softmax scale is 1/sqrt(d) (standard attention; the pages' formula for the
shared-prefix matmul lost the square root in extraction).
"""
from __future__ import annotations

import numpy as np

from synth import gen
from synth.gen import (KIND_NEW_K, KIND_NEW_V, KIND_PREFIX_K, KIND_PREFIX_V, KIND_Q,
                       KIND_SUFFIX_K, KIND_SUFFIX_V, bf16_bits_to_f64, normal_bits, stream_key)

from . import attention


def prefix_kv_bits(w, p, layer):
    """[Lp][Hkv][d] bits of prefix p at a layer (token-major, the write order)."""
    lp = w.prefix_lens[p]
    n = lp * w.Hkv * w.d
    k = normal_bits(stream_key(w.seed, KIND_PREFIX_K, p, layer), 0, n).reshape(lp, w.Hkv, w.d)
    v = normal_bits(stream_key(w.seed, KIND_PREFIX_V, p, layer), 0, n).reshape(lp, w.Hkv, w.d)
    return k, v


def suffix_kv_bits(w, source, length, layer):
    """[s][Hkv][d] bits of the first `length` cached suffix tokens of a source sequence."""
    n = length * w.Hkv * w.d
    k = normal_bits(stream_key(w.seed, KIND_SUFFIX_K, source, layer), 0, n).reshape(length, w.Hkv, w.d)
    v = normal_bits(stream_key(w.seed, KIND_SUFFIX_V, source, layer), 0, n).reshape(length, w.Hkv, w.d)
    return k, v


def new_kv_bits(w, layer, step, B=None):
    """[B][Hkv][d] bits of the token every request appends at a step."""
    B = w.B if B is None else B
    n = B * w.Hkv * w.d
    k = normal_bits(stream_key(w.seed, KIND_NEW_K, layer, step), 0, n).reshape(B, w.Hkv, w.d)
    v = normal_bits(stream_key(w.seed, KIND_NEW_V, layer, step), 0, n).reshape(B, w.Hkv, w.d)
    return k, v


def q_bits(w, layer, step, B=None):
    """[B][Hq][d] bits of the step's queries (times 2**q_log2_scale, exact)."""
    B = w.B if B is None else B
    q = normal_bits(stream_key(w.seed, KIND_Q, layer, step), 0, B * w.Hq * w.d)
    return gen.scale_bf16_bits_pow2(q, w.q_log2_scale).reshape(B, w.Hq, w.d)


class ContextCache:
    """Memoises the per-layer prefix and suffix streams of one workload."""

    def __init__(self, w):
        self.w = w
        self._pre = {}
        self._suf = {}

    def prefix(self, p, layer):
        key = (p, layer)
        if key not in self._pre:
            k, v = prefix_kv_bits(self.w, p, layer)
            self._pre[key] = (bf16_bits_to_f64(k).transpose(1, 0, 2), bf16_bits_to_f64(v).transpose(1, 0, 2))
        return self._pre[key]

    def suffix(self, source, length, layer):
        key = (source, layer)
        if key not in self._suf or self._suf[key][0].shape[1] < length:
            k, v = suffix_kv_bits(self.w, source, length, layer)
            self._suf[key] = (bf16_bits_to_f64(k).transpose(1, 0, 2), bf16_bits_to_f64(v).transpose(1, 0, 2))
        k, v = self._suf[key]
        return k[:, :length], v[:, :length]


def context(w, r, layer, appended=0, cache=None):
    """Explicit K, V [Hkv][n][d] fp64 of request r after `appended` step tokens."""
    cache = cache or ContextCache(w)
    req = w.requests[r]
    parts_k, parts_v = [], []
    if req.prefix >= 0:
        k, v = cache.prefix(req.prefix, layer)
        parts_k.append(k)
        parts_v.append(v)
    if req.suffix_len:
        k, v = cache.suffix(req.source, req.suffix_len, layer)
        parts_k.append(k)
        parts_v.append(v)
    for t in range(appended):
        k, v = new_kv_bits(w, layer, t)
        parts_k.append(bf16_bits_to_f64(k[r])[:, None, :])
        parts_v.append(bf16_bits_to_f64(v[r])[:, None, :])
    if not parts_k:
        z = np.zeros((w.Hkv, 0, w.d))
        return z, z.copy()
    return np.concatenate(parts_k, axis=1), np.concatenate(parts_v, axis=1)


def expected(w, layer, requests=None, appended=0, q_step=0, cache=None, q=None):
    """Oracle outputs (O [n][Hq][d], LSE [n][Hq], natural log) for the listed requests."""
    requests = list(range(w.B)) if requests is None else list(requests)
    cache = cache or ContextCache(w)
    qb = q_bits(w, layer, q_step) if q is None else q
    O = np.empty((len(requests), w.Hq, w.d))
    LSE = np.empty((len(requests), w.Hq))
    for i, r in enumerate(requests):
        K, V = context(w, r, layer, appended, cache)
        O[i], LSE[i] = attention.attend_heads(bf16_bits_to_f64(qb[r]), K, V)
    return O, LSE
