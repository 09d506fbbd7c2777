"""Sets a synthetic workload up on the GPU through the library's own calls.

Inputs come from the seeded device generator (synth/fill.cu), written with
gk_write_prefix_kv (HOT) and gk_seq_append_slots + gk_append_kv (COLD), exactly
as a serving engine would; the oracle regenerates the same values on the host.
Shared by the GPU tests and bench.py.
"""
from __future__ import annotations

import numpy as np

from paged_kv_cache_pool_gb300 import binding as gk
from paged_kv_cache_pool_gb300.engine import Engine
from synth import device as sdev
from synth.gen import (KIND_NEW_K, KIND_NEW_V, KIND_PREFIX_K, KIND_PREFIX_V, KIND_Q, KIND_SUFFIX_K,
                       KIND_SUFFIX_V, stream_key)


class GpuWorkload:
    def __init__(self, w, layers=None, cold_seed=None, page_size=None, extra_steps=0, device="cuda"):
        import torch
        self.torch = torch
        self.w = w
        self.P = page_size or w.page_size
        self.layers = list(range(w.L)) if layers is None else list(layers)
        saved = w.extra_steps
        w.extra_steps = extra_steps
        cold_slots = w.cold_slots(self.P)
        w.extra_steps = saved
        self.eng = Engine(w.L, w.Hq, w.Hkv, w.d, w.hot_tokens(), cold_slots, self.P,
                          seed=w.seed if cold_seed is None else cold_seed, device=device)
        self.dev = self.eng.device
        bf = torch.bfloat16
        kv_row = w.Hkv * w.d
        # HOT prefixes, allocated in order
        self.bases = [self.eng.prefix_alloc(lp) for lp in w.prefix_lens]
        for layer in self.layers:
            for p, lp in enumerate(w.prefix_lens):
                k = torch.empty(lp * kv_row, dtype=bf, device=self.dev)
                v = torch.empty_like(k)
                sdev.fill_normal(k, stream_key(w.seed, KIND_PREFIX_K, p, layer))
                sdev.fill_normal(v, stream_key(w.seed, KIND_PREFIX_V, p, layer))
                self.eng.write_prefix(layer, self.bases[p], lp, 0, k.view(lp, w.Hkv, w.d), v.view(lp, w.Hkv, w.d))
        # COLD suffixes: one append call covering every source sequence
        if w.fork_children:
            sources = [(p, n) for p, n in enumerate(w.parents)]
        else:
            sources = [(r.source, r.suffix_len) for r in w.requests]
        src_seq = [self.eng.seq_create() for _ in sources]
        order = np.concatenate([np.full(n, s, dtype=np.int32) for s, (_, n) in zip(src_seq, sources)]) \
            if sources else np.zeros(0, np.int32)
        slots, cow = self.eng.append_slots(order)
        assert len(cow) == 0
        d_slots = self.eng.to_device(slots)
        total = len(order)
        if total:
            for layer in self.layers:
                k = torch.empty(total * kv_row, dtype=bf, device=self.dev)
                v = torch.empty_like(k)
                off = 0
                for src, n in sources:
                    if n:
                        sdev.fill_normal(k[off * kv_row:(off + n) * kv_row], stream_key(w.seed, KIND_SUFFIX_K, src, layer))
                        sdev.fill_normal(v[off * kv_row:(off + n) * kv_row], stream_key(w.seed, KIND_SUFFIX_V, src, layer))
                    off += n
                self.eng.append_kv(layer, d_slots, k, v)
        if w.fork_children:
            self.seqs = []
            for s in src_seq:
                self.seqs.extend(self.eng.seq_fork(s) for _ in range(w.fork_children))
                self.eng.seq_release(s)
        else:
            self.seqs = src_seq
        self.appended = 0
        self.last_cow = np.zeros((0, 2), np.int32)
        torch.cuda.synchronize()

    # ---- per step --------------------------------------------------------------------
    def q(self, layer, step=0):
        w = self.w
        q = self.torch.empty(w.B * w.Hq * w.d, dtype=self.torch.bfloat16, device=self.dev)
        sdev.fill_normal(q, stream_key(w.seed, KIND_Q, layer, step), log2_scale=w.q_log2_scale)
        return q.view(w.B, w.Hq, w.d)

    def new_kv(self, layer, step):
        w = self.w
        n = w.B * w.Hkv * w.d
        k = self.torch.empty(n, dtype=self.torch.bfloat16, device=self.dev)
        v = self.torch.empty_like(k)
        sdev.fill_normal(k, stream_key(w.seed, KIND_NEW_K, layer, step))
        sdev.fill_normal(v, stream_key(w.seed, KIND_NEW_V, layer, step))
        return k, v

    def append_step(self, step, layers=None):
        """Every request appends its step token (slots, copy-on-write, then the K/V writes)."""
        slots, cow = self.eng.append_slots(np.asarray(self.seqs, dtype=np.int32))
        self.last_cow = cow
        d_slots = self.eng.to_device(slots)
        d_cow = self.eng.to_device(cow.reshape(-1)) if len(cow) else None
        for layer in (self.layers if layers is None else layers):
            k, v = self.new_kv(layer, step)
            self.eng.append_kv(layer, d_slots, k, v, d_cow)
        self.appended += 1
        return slots, cow

    def batch(self):
        w = self.w
        bases = [self.bases[r.prefix] if r.prefix >= 0 else -1 for r in w.requests]
        lps = [w.prefix_lens[r.prefix] if r.prefix >= 0 else 0 for r in w.requests]
        slen = [self.eng.seq_len(s) for s in self.seqs]
        table = self.eng.block_tables(self.seqs)
        self._d_table = self.eng.to_device(table)
        b = self.eng.batch(bases, lps, slen, self._d_table, table.shape[1])
        return b

    def outputs(self):
        w = self.w
        out = self.torch.empty((w.B, w.Hq, w.d), dtype=self.torch.float32, device=self.dev)
        lse = self.torch.empty((w.B, w.Hq), dtype=self.torch.float32, device=self.dev)
        return out, lse

    def run(self, layer, backend, step=0, batch=None, plan=None):
        """One layer of one step -> (O, LSE) numpy arrays."""
        b = batch or self.batch()
        q = self.q(layer, step)
        out, lse = self.outputs()
        b.set_device(d_q=q, d_out=out, d_lse=lse)
        pl = plan or self.eng.plan(b)
        self.eng.decode(layer, b, pl, backend)
        self.torch.cuda.synchronize()
        err = self.eng.device_error()
        assert err == gk.GK_OK, f"device error word {err}"
        return out.cpu().numpy(), lse.cpu().numpy()

    def close(self):
        self.eng.close()
