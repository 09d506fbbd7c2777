"""Tensor-core utilisation of the cascade prefix contraction alone, as the work grows
(GraniKV Section 2.3, the shared-prefix matmul: every query row that shares a prefix
stacked into one contraction against the contiguous HOT slab).

For each (Lp, B) of a grid, one layer of a synthetic pool (random bf16 data; Llama-3.1-8B
attention geometry: Hq 32, Hkv 8, d 128) with one shared prefix of Lp tokens and B
requests, a sequential cascade plan, and gk_cascade_prefix timed alone with CUDA events:
L2 written and cleaned before each launch, median of `reps` launches.  Reported per cell:
the useful work 4 * B * Hq * Lp * d flops (padded rows excluded), the plan's work items and
key tiles per item, TFLOP/s and the fraction of the measured dense bf16 peak (burst, a
kernel timed alone; MEASURED_PEAKS.json at the repository root, else 1900 TFLOP/s).

    python -m paged_kv_cache_pool_gb300.prefix_scaling [--out rows.json]
"""
from __future__ import annotations

import argparse
import json
import os

import numpy as np

from . import binding as gk

LPS = (4096, 16384, 65536)
BS = (64, 256, 512)
FALLBACK_BF16_TFLOPS = 1900.0


def _peak():
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for k in ("bf16_tflops", "bf16_dense_tflops"):
            if k in d:
                return float(d[k]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def measure(lps=LPS, bs=BS, Hq=32, Hkv=8, d=128, reps=5, suffix=16):
    """-> list of per-cell dicts (times in microseconds)."""
    import torch
    from .engine import Engine
    peak, src = _peak()
    eng = Engine(1, Hq, Hkv, d, max(lps) + 16, max(bs) * suffix + 64, 1, seed=1)
    for t in (eng.hot_k, eng.hot_v, eng.cold_k, eng.cold_v):
        t.normal_()
    pool = eng.pool
    gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SEQUENTIAL, 0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=eng.device)
    clean = torch.zeros(256 << 20, dtype=torch.uint8, device=eng.device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rows = []
    for lp in lps:
        base = eng.prefix_alloc(lp)
        for B in bs:
            seqs = [eng.seq_create() for _ in range(B)]
            eng.append_slots(np.repeat(np.asarray(seqs, np.int32), suffix))
            table = eng.block_tables(seqs)
            d_table = eng.to_device(table)
            batch = eng.batch([base] * B, [lp] * B, [suffix] * B, d_table, table.shape[1])
            q = torch.randn((B, Hq, d), device=eng.device).to(torch.bfloat16)
            out = torch.empty((B, Hq, d), device=eng.device)
            lse = torch.empty((B, Hq), device=eng.device)
            batch.set_device(d_q=q, d_out=out, d_lse=lse)
            plan = gk.gk_plan_build(pool, batch)
            info = gk.gk_plan_info(plan)
            ts = []
            for _ in range(reps + 1):
                flush.zero_()
                clean.max()
                ev0.record()
                gk.gk_cascade_prefix(pool, None, 0, batch, plan)
                ev1.record()
                torch.cuda.synchronize()
                ts.append(ev0.elapsed_time(ev1) * 1e3)
            if gk.gk_device_error(pool) != gk.GK_OK:
                raise RuntimeError(f"device error at Lp={lp} B={B}")
            t = float(np.median(ts[1:]))
            flops = 4 * B * Hq * lp * d
            rows.append(dict(Lp=lp, B=B, M_eff=B * Hq // Hkv, gflop=flops / 1e9, items=info["prefix_ctas"],
                             tiles_per_item=info["prefix_tiles_per_item"], t_us=t,
                             tflops=flops / (t * 1e-6) / 1e12, frac=flops / (t * 1e-6) / 1e12 / peak,
                             peak_tflops=peak, peak_source=src))
            gk.gk_plan_destroy(plan)
            for sq in seqs:
                eng.seq_release(sq)
        gk.gk_prefix_release(pool, base)
    eng.close()
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None)
    a = ap.parse_args()
    from . import build
    build.build()
    rows = measure()
    for r in rows:
        print(json.dumps(r))
    if a.out:
        with open(a.out, "w") as f:
            json.dump(rows, f, indent=1)


if __name__ == "__main__":
    main()
