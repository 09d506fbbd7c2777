"""Where the two backends cross on this GPU, and how often the dispatcher routes
to each (GraniKV Appendix B.4 and B.4b, re-run: the pages fit the saturation
threshold M_sat = 1024 on A100 and say it must be re-fit on other hardware).

Two parts:

  measure  On one layer of a synthetic pool (random bf16 data), for every cell
           of an (Lp, B) grid with one shared prefix and suffixes drawn from
           U{16..512} (the pages' 16..512-token user turns), time the three
           choices with CUDA events, L2 flushed before every launch: the flat
           (dense) backend, the cascade over tensor-core prefix items and the
           cascade over warp-MMA prefix items (GraniKV Section 3.5's two prefix
           kernels), each as the planner arranges it, and record the predictions
           and the pick of the default plan (GK_PREFIX_AUTO, then gk_dispatch).
           Per cell: M_eff = B * g (GraniKV Eq. 2), the fastest choice, and the
           regret of the pick (its time over the fastest one's, - 1).

  trace    Host only.  Per (Lp, B) cell, 200 decode steps whose realised batch
           is B plus a Poisson(B / 8) burst of requests whose prefill overlaps
           the step (the pages' reason the realised batch exceeds the admission
           batch), suffixes redrawn every step; the fraction of steps the
           dispatcher routes to the dense backend (the pages' Table 15).

    python -m paged_kv_cache_pool_gb300.dispatch_sweep measure [--out rows.json]
    python -m paged_kv_cache_pool_gb300.dispatch_sweep trace
"""
from __future__ import annotations

import argparse
import json
import os

import numpy as np

from . import binding as gk

LPS = (512, 2048, 8192, 16384)
BS = (8, 32, 128, 256, 512)
S_RANGE = (16, 512)
COST_MODEL = os.path.join(os.path.dirname(os.path.abspath(__file__)), "cost_model_gb300.json")


def _load_cost_model(pool, path):
    if path and os.path.exists(path):
        with open(path) as f:
            gk.gk_cost_model_load(pool, f.read())


def _suffixes(rng, n):
    return rng.integers(S_RANGE[0], S_RANGE[1] + 1, n).astype(np.int32)


def measure(lps=LPS, bs=BS, Hq=32, Hkv=8, d=128, reps=7, seed=7, cost_model=COST_MODEL):
    """-> list of per-cell dicts (times in microseconds)."""
    import torch
    from .engine import Engine
    g = Hq // Hkv
    cold = max(bs) * S_RANGE[1] + 4096
    eng = Engine(1, Hq, Hkv, d, sum(lps) + 16 * len(lps), cold, 1, seed=1)
    for t in (eng.hot_k, eng.hot_v, eng.cold_k, eng.cold_v):
        t.normal_()
    pool = eng.pool
    _load_cost_model(pool, cost_model)
    # L2 flush: write a buffer larger than L2, then read another one, so that each timed launch
    # starts from a cold L2 holding no dirty lines (their write-back would be timed)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=eng.device)
    clean = torch.zeros(256 << 20, dtype=torch.uint8, device=eng.device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        ts = []
        for _ in range(reps + 1):
            flush.zero_()
            clean.max()
            ev0.record()
            fn()
            ev1.record()
            torch.cuda.synchronize()
            ts.append(ev0.elapsed_time(ev1) * 1e3)
        return float(np.median(ts[1:]))

    rows = []
    for lp in lps:
        base = eng.prefix_alloc(lp)
        for B in bs:
            rng = np.random.default_rng([seed, lp, B])
            s = _suffixes(rng, B)
            seqs = [eng.seq_create() for _ in range(B)]
            eng.append_slots(np.repeat(np.asarray(seqs, np.int32), s))
            table = eng.block_tables(seqs)
            d_table = eng.to_device(table)
            batch = eng.batch([base] * B, [lp] * B, s.tolist(), d_table, table.shape[1])
            q = torch.randn((B, Hq, d), device=eng.device).to(torch.bfloat16)
            out = torch.empty((B, Hq, d), device=eng.device)
            lse = torch.empty((B, Hq), device=eng.device)
            batch.set_device(d_q=q, d_out=out, d_lse=lse)
            t, pred, arr, detail = {}, {}, {}, {}
            for kind, kernel in (("tensor", gk.GK_PREFIX_TENSOR), ("warp", gk.GK_PREFIX_WARP)):
                gk.gk_pool_set_prefix_kernel(pool, kernel)
                # the planner's arrangement (timed whole, and its levels and merge launches
                # alone), then the sequential arrangement for the same kind of item
                for mode, mname in ((gk.GK_CASCADE_AUTO, "auto"), (gk.GK_CASCADE_SEQUENTIAL, "sequential")):
                    gk.gk_pool_set_cascade_mode(pool, mode, 0)
                    plan = gk.gk_plan_build(pool, batch)
                    info = gk.gk_plan_info(plan)
                    _, p_dense, p_cas = gk.gk_dispatch(pool, plan)
                    t_cas = timed(lambda: gk.gk_decode_cascade(pool, None, 0, batch, plan))
                    t_lev = timed(lambda: gk.gk_cascade_levels(pool, None, 0, batch, plan))
                    t_mrg = timed(lambda: gk.gk_cascade_merge(pool, None, 0, batch, plan))
                    detail[f"{kind}_{mname}"] = dict(info, t_cascade_us=t_cas, t_levels_us=t_lev, t_merge_us=t_mrg,
                                                     pred_cascade_us=p_cas)
                    if mname == "auto":
                        pred[kind] = p_cas
                        arr[kind] = dict(split=info["cascade_split"], C=info["prefix_tiles_per_item"],
                                         n_pre=info["prefix_ctas"], suffix_ctas=info["suffix_ctas"],
                                         partials=info["num_partials"], gather=info["prefix_ctas_gather"])
                        t[kind] = t_cas
                        if kind == "tensor":
                            t["dense"] = timed(lambda: gk.gk_decode_dense(pool, None, 0, batch, plan))
                    gk.gk_plan_destroy(plan)
                gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_AUTO, 0)
            pred["dense"] = p_dense
            gk.gk_pool_set_prefix_kernel(pool, gk.GK_PREFIX_AUTO)
            plan = gk.gk_plan_build(pool, batch)
            choice, _, _ = gk.gk_dispatch(pool, plan)
            auto_kind = "warp" if gk.gk_plan_info(plan)["prefix_kernel"] == gk.GK_PREFIX_WARP else "tensor"
            gk.gk_plan_destroy(plan)
            if gk.gk_device_error(pool) != gk.GK_OK:
                raise RuntimeError(f"device error at Lp={lp} B={B}")
            pick = "dense" if choice == gk.GK_BACKEND_DENSE else auto_kind
            fastest = min(t, key=t.get)
            rows.append(dict(Lp=lp, B=B, M_eff=B * g, suffix_tokens=int(s.sum()),
                             t_dense_us=t["dense"], t_tensor_us=t["tensor"], t_warp_us=t["warp"],
                             pred_dense_us=pred["dense"], pred_tensor_us=pred["tensor"], pred_warp_us=pred["warp"],
                             plan_tensor=arr["tensor"], plan_warp=arr["warp"], plans=detail,
                             pick=pick, fastest=fastest, regret=t[pick] / t[fastest] - 1.0))
            for sq in seqs:
                eng.seq_release(sq)
        gk.gk_prefix_release(pool, base)
    eng.close()
    return rows


def crossover(rows):
    """Per Lp: the M_eff values of the grid at which each choice is measured fastest."""
    out = {}
    for lp in sorted({r["Lp"] for r in rows}):
        out[lp] = {k: [r["M_eff"] for r in rows if r["Lp"] == lp and r["fastest"] == k]
                   for k in ("dense", "tensor", "warp")}
    return out


def trace(lps=LPS, bs=BS, Hq=32, Hkv=8, d=128, steps=200, seed=11, cost_model=COST_MODEL, num_sms=None):
    """-> {(Lp, B): fraction of steps routed to dense} on a host-only pool."""
    burst_max = max(bs) * 2
    pool = gk.gk_pool_create(1, Hq, Hkv, d, sum(lps) + 16 * len(lps), burst_max * S_RANGE[1] + 4096, 1, 0)
    try:
        _load_cost_model(pool, cost_model)
        frac = {}
        for lp in lps:
            base = gk.gk_prefix_alloc(pool, lp)
            for B in bs:
                rng = np.random.default_rng([seed, lp, B])
                dense = 0
                for _ in range(steps):
                    n = B + int(rng.poisson(B / 8))
                    s = _suffixes(rng, n)
                    batch = gk.Batch([base] * n, [lp] * n, s.tolist(), None, S_RANGE[1])
                    plan = gk.gk_plan_build(pool, batch)
                    dense += gk.gk_dispatch(pool, plan)[0] == gk.GK_BACKEND_DENSE
                    gk.gk_plan_destroy(plan)
                frac[(lp, B)] = dense / steps
            gk.gk_prefix_release(pool, base)
        return frac
    finally:
        gk.gk_pool_destroy(pool)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("part", choices=["measure", "trace"])
    ap.add_argument("--out", default=None)
    a = ap.parse_args()
    from . import build
    build.build()
    if a.part == "measure":
        rows = measure()
        for r in rows:
            print(json.dumps(r))
        print(json.dumps({"fastest_by_M_eff": crossover(rows),
                          "max_regret": max(r["regret"] for r in rows)}))
        if a.out:
            with open(a.out, "w") as f:
                json.dump(rows, f, indent=1)
    else:
        frac = trace()
        print("routed to dense, Lp x B:", " ".join(f"{B:>6}" for B in BS))
        for lp in LPS:
            print(f"{lp:>26}", " ".join(f"{frac[(lp, B)]:6.0%}" for B in BS))


if __name__ == "__main__":
    main()
