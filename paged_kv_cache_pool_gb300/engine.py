"""Convenience layer over libgk for Python callers: a pool with its storage.

It allocates the HOT and COLD K/V storage as torch CUDA tensors (PyTorch is
only the device-memory and stream provider here), creates the pool over them,
keeps the plans it builds so that close() frees them, and names the calls of a
decode step, which the caller strings together in this order:

  append_slots (gk_seq_append_slots) -> append_kv (gk_append_kv, per layer;
  or the decode's fused append) -> plan (gk_plan_build / gk_plan_update)
  -> dispatch (gk_dispatch) -> decode (gk_decode_cascade | gk_decode_dense,
  per layer).

Every method is one library call; the work is in libgk.
"""
from __future__ import annotations

import numpy as np

from . import binding as gk


class Engine:
    def __init__(self, L, Hq, Hkv, d, hot_tokens, cold_slots, page_size, seed=0, device="cuda"):
        import torch
        self.torch = torch
        self.L, self.Hq, self.Hkv, self.d = L, Hq, Hkv, d
        self.page_size = page_size
        self.cold_slots = cold_slots
        self.device = torch.device(device)
        bf = torch.bfloat16
        self.hot_k = torch.empty(max(1, hot_tokens) * L * Hkv * d, dtype=bf, device=self.device)
        self.hot_v = torch.empty_like(self.hot_k)
        self.cold_k = torch.empty((L, cold_slots, Hkv, d), dtype=bf, device=self.device)
        self.cold_v = torch.empty_like(self.cold_k)
        self.pool = gk.gk_pool_create(L, Hq, Hkv, d, hot_tokens, cold_slots, page_size, seed,
                                      self.hot_k, self.hot_v, self.cold_k, self.cold_v)
        self._plans = []

    def close(self):
        for p in self._plans:
            gk.gk_plan_destroy(p)
        self._plans = []
        if self.pool:
            gk.gk_pool_destroy(self.pool)
            self.pool = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- HOT ----------------------------------------------------------------------
    def prefix_alloc(self, lp):
        return gk.gk_prefix_alloc(self.pool, lp)

    def write_prefix(self, layer, base, lp, t0, k, v, stream=None):
        gk.gk_write_prefix_kv(self.pool, stream, layer, base, lp, t0, k, v)

    # ---- COLD ---------------------------------------------------------------------
    def seq_create(self):
        return gk.gk_seq_create(self.pool)

    def seq_fork(self, parent):
        return gk.gk_seq_fork(self.pool, parent)

    def seq_release(self, seq):
        gk.gk_seq_release(self.pool, seq)

    def append_slots(self, seqs):
        return gk.gk_seq_append_slots(self.pool, seqs)

    def to_device(self, arr):
        t = self.torch.from_numpy(np.ascontiguousarray(arr))
        return t.pin_memory().to(self.device, non_blocking=True)

    def append_kv(self, layer, d_slots, k, v, d_cow=None, stream=None):
        gk.gk_append_kv(self.pool, stream, layer, d_slots, k, v, d_cow)

    def block_tables(self, seqs, max_blocks=None, out=None, lens=None):
        if max_blocks is None:
            max_blocks = max([1] + [len(gk.gk_seq_table(self.pool, s)[0]) for s in seqs])
        return gk.gk_seq_tables(self.pool, seqs, max_blocks, out, lens)[0]

    def seq_len(self, seq):
        return gk.gk_seq_table(self.pool, seq)[1]

    # ---- step -------------------------------------------------------------------------
    def batch(self, prefix_bases, prefix_lens, suffix_lens, d_table, max_blocks):
        return gk.Batch(prefix_bases, prefix_lens, suffix_lens, d_table, max_blocks)

    def plan(self, batch, stream=None, plan=None):
        if plan is None:
            plan = gk.gk_plan_build(self.pool, batch, stream)
            self._plans.append(plan)
        else:
            gk.gk_plan_update(self.pool, plan, batch, stream)
        return plan

    def dispatch(self, plan):
        return gk.gk_dispatch(self.pool, plan)

    def decode(self, layer, batch, plan, backend, stream=None):
        if backend == gk.GK_BACKEND_DENSE:
            gk.gk_decode_dense(self.pool, stream, layer, batch, plan)
        else:
            gk.gk_decode_cascade(self.pool, stream, layer, batch, plan)

    def device_error(self, stream=None):
        return gk.gk_device_error(self.pool, stream)
