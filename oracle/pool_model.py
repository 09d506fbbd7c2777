"""ORACLE (test infrastructure): host model of the HOT and COLD KV storage.

Values are kept as bf16 bit patterns (uint16) so that copies can be compared
bit for bit with device memory.

Layouts (readings stated where the pages leave them open):
* COLD, per layer: slot-major [cold_slots][Hkv][d] for K and for V ("Paged KV
  cache": the physical pool is per layer; slot = block * P + offset).
* HOT: GraniKV Section 3.2 places (layer l, head h) of a prefix at
  base + l*Lp*Hkv + h*Lp, while a released prefix frees the token range
  [base, base + Lp).  Both hold when the allocator counts tokens and a prefix
  at token base b owns the elements [b*L*Hkv*d, (b+Lp)*L*Hkv*d) laid out
  [L][Hkv][Lp][d]: the (l, h) slice is then a contiguous [Lp][d] block.

reshape_and_cache ("Paged KV cache", How it works, step 1) writes token i's
K/V [Hkv][d] to COLD[layer][slot_mapping[i]].  A copy-on-write pair (src, dst)
copies the P slots of block src to block dst first (step 2).
"""
from __future__ import annotations

import numpy as np


class PoolModel:
    def __init__(self, L, Hkv, d, hot_tokens, cold_slots, page_size):
        self.L, self.Hkv, self.d = L, Hkv, d
        self.P = page_size
        self.hot_k = np.zeros(hot_tokens * L * Hkv * d, dtype=np.uint16)
        self.hot_v = np.zeros_like(self.hot_k)
        self.cold_k = np.zeros((L, cold_slots, Hkv, d), dtype=np.uint16)
        self.cold_v = np.zeros_like(self.cold_k)

    def hot_slice(self, which, layer, base, lp, head):
        """View of the contiguous [Lp][d] block of (layer, head) of the prefix at token base."""
        arr = self.hot_k if which == "k" else self.hot_v
        start = (base * self.L * self.Hkv + (layer * self.Hkv + head) * lp) * self.d
        return arr[start:start + lp * self.d].reshape(lp, self.d)

    def write_prefix(self, layer, base, lp, t0, k, v):
        """Prefix tokens t0.. of one layer; k, v [n][Hkv][d] bits."""
        n = k.shape[0]
        for h in range(self.Hkv):
            self.hot_slice("k", layer, base, lp, h)[t0:t0 + n] = k[:, h, :]
            self.hot_slice("v", layer, base, lp, h)[t0:t0 + n] = v[:, h, :]

    def append(self, layer, slot_mapping, k, v, cow_pairs=()):
        """Copy-on-write block copies, then scatter token i to slot_mapping[i]."""
        P = self.P
        for src, dst in cow_pairs:
            self.cold_k[layer, dst * P:(dst + 1) * P] = self.cold_k[layer, src * P:(src + 1) * P]
            self.cold_v[layer, dst * P:(dst + 1) * P] = self.cold_v[layer, src * P:(src + 1) * P]
        for i, slot in enumerate(slot_mapping):
            self.cold_k[layer, slot] = k[i]
            self.cold_v[layer, slot] = v[i]

    def gather(self, layer, hot_base, lp, table, suffix_len):
        """Context of one request: prefix tokens then suffix tokens via the table -> K, V [Hkv][n][d] bits."""
        n = lp + suffix_len
        K = np.empty((self.Hkv, n, self.d), dtype=np.uint16)
        V = np.empty_like(K)
        if lp:
            for h in range(self.Hkv):
                K[h, :lp] = self.hot_slice("k", layer, hot_base, lp, h)
                V[h, :lp] = self.hot_slice("v", layer, hot_base, lp, h)
        if suffix_len:
            t = np.arange(suffix_len)
            slots = np.asarray(table, dtype=np.int64)[t // self.P] * self.P + t % self.P
            K[:, lp:] = self.cold_k[layer, slots].transpose(1, 0, 2)
            V[:, lp:] = self.cold_v[layer, slots].transpose(1, 0, 2)
        return K, V


def build_pool(w, layers=None, cold_seed=None, page_size=None, steps=0):
    """Run a workload's setup through the oracle block manager and pool model.

    Prefixes go to the HOT allocator in order; each sequence's cached suffix is
    appended token by token (forked workloads: the parent's suffix, then the
    forks, then the parent is released); then `steps` decode-step appends for
    every request in batch order.  Returns (model, hot_bases, seqs, block_pool).
    """
    from .block_manager import BlockPool, Seq
    from .hot_pool import HotPool
    from .reference import new_kv_bits, prefix_kv_bits, suffix_kv_bits

    layers = range(w.L) if layers is None else layers
    P = w.page_size if page_size is None else page_size
    seed = w.seed if cold_seed is None else cold_seed
    cold_slots = w.cold_slots(P)
    pm = PoolModel(w.L, w.Hkv, w.d, w.hot_tokens(), cold_slots, P)
    hot = HotPool(w.hot_tokens())
    bases = [hot.alloc(lp) for lp in w.prefix_lens]
    for layer in layers:
        for p, lp in enumerate(w.prefix_lens):
            k, v = prefix_kv_bits(w, p, layer)
            pm.write_prefix(layer, bases[p], lp, 0, k, v)
    bp = BlockPool(cold_slots // P, P, seed)

    def fill(seq, source, length):
        slots = [bp.append(seq)[0] for _ in range(length)]
        for layer in layers:
            k, v = suffix_kv_bits(w, source, length, layer)
            pm.append(layer, slots, k, v)

    if w.fork_children:
        seqs = []
        for p, length in enumerate(w.parents):
            parent = Seq()
            fill(parent, p, length)
            seqs.extend(bp.fork(parent) for _ in range(w.fork_children))
            bp.release(parent)
    else:
        seqs = []
        for r, req in enumerate(w.requests):
            s = Seq()
            fill(s, req.source, req.suffix_len)
            seqs.append(s)
    for t in range(steps):
        res = [bp.append(s) for s in seqs]
        slots = [x[0] for x in res]
        cows = [x[1] for x in res if x[1] is not None]
        for layer in layers:
            k, v = new_kv_bits(w, layer, t)
            pm.append(layer, slots, k, v, cows)
    return pm, bases, seqs, bp
