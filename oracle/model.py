"""ORACLE (test infrastructure): the byte and flop model of one decode-attention layer.

* KV bytes per token = 2 (K and V) * layers * kv_heads * head_dim * bytes
  ("Paged KV cache", Complexity and constants; 128 KB for Llama-3-8B).
* A request that reads a shared prefix from its own pages moves
  B * Lp * 2 * Hkv * d * 2 bytes per launch (GraniKV Appendix B.11, the paged
  side of Table 23), while the contiguous HOT layout reads the prefix once.
* Useful work of the shared-prefix contraction: QK^T and PV are each
  2 * M * Lp * d flops per KV head with M = B * (Hq / Hkv) stacked rows, so
  4 * B * Hq * Lp * d in total (34.4 GFLOP at B = 256, Lp = 8K, Llama head).
"""
from __future__ import annotations


def kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes=2):
    return 2 * layers * kv_heads * head_dim * elem_bytes


def paged_prefix_bytes(B, Lp, Hkv, d, elem_bytes=2):
    return B * Lp * 2 * Hkv * d * elem_bytes


def shared_prefix_bytes(Lp, Hkv, d, elem_bytes=2):
    return Lp * 2 * Hkv * d * elem_bytes


def prefix_flops(B, Hq, Lp, d):
    return 4 * B * Hq * Lp * d


def suffix_kv_bytes(suffix_lens, Hkv, d, elem_bytes=2):
    return sum(suffix_lens) * 2 * Hkv * d * elem_bytes


def dense_kv_bytes(prefix_lens, suffix_lens, Hkv, d, elem_bytes=2):
    """Flat paged decode: every request reads its whole context."""
    return sum(p + s for p, s in zip(prefix_lens, suffix_lens)) * 2 * Hkv * d * elem_bytes
