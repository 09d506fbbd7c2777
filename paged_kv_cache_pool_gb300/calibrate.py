"""Measure the dispatcher's cost model on this GPU (GraniKV Section 3.6: the
routing rule stays, its numbers are re-fit per GPU; Appendix B.4b's sweep).

Times, with CUDA events, on one layer of synthetic pools (random bf16 data):
  * the flat backend over several (B, Lp, s)              -> c_flat_us, bw_flat_gbs
  * the suffix gather over every SM, several volumes        -> c_gather_us + bytes / bw_suffix_gbs
  * prefix items of C key tiles, forced split plans and the -> prefix_item_us + C * prefix_tile_us
    sequential plans of several M_eff = B * g
  * the tile of an item beside the gather                   -> prefix_tile_split_us = SPLIT_TILE_RATIO *
                                                               prefix_tile_us
  * the gather alone on the SMs long prefix items leave it  -> gather_sm_gbs
  * the merge                                               -> c_merge_us per (request, head)
  * the whole cascade, both arrangements                    -> c_cascade_us (mean residual)
and writes the JSON that gk_cost_model_load reads.

    python -m paged_kv_cache_pool_gb300.calibrate --out cost_model_gb300.json
"""
from __future__ import annotations

import argparse
import json

import numpy as np

from . import binding as gk
from .engine import Engine


def _time(fn, reps=10, warm=3):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / reps  # us


class _Case:
    """One layer of a pool with B requests sharing a prefix of Lp and suffixes of s tokens."""

    def __init__(self, eng, B, lp, s, Hq, d, mode=gk.GK_CASCADE_SEQUENTIAL, tiles=0):
        import torch
        self.eng = eng
        base = eng.prefix_alloc(lp)
        self.base = base
        seqs = [eng.seq_create() for _ in range(B)]
        order = np.repeat(np.asarray(seqs, np.int32), s)
        if len(order):
            eng.append_slots(order)
        self.seqs = seqs
        table = eng.block_tables(seqs)
        self.d_table = eng.to_device(table)
        self.batch = eng.batch([base] * B, [lp] * B, [s] * B, self.d_table, table.shape[1])
        self.q = torch.randn((B, Hq, d), device=eng.device).to(torch.bfloat16)
        self.out = torch.empty((B, Hq, d), device=eng.device)
        self.lse = torch.empty((B, Hq), device=eng.device)
        self.batch.set_device(d_q=self.q, d_out=self.out, d_lse=self.lse)
        gk.gk_pool_set_cascade_mode(eng.pool, mode, tiles)
        self.plan = gk.gk_plan_build(eng.pool, self.batch)
        gk.gk_pool_set_cascade_mode(eng.pool, gk.GK_CASCADE_AUTO)
        self.info = gk.gk_plan_info(self.plan)

    def close(self):
        gk.gk_plan_destroy(self.plan)
        for s in self.seqs:
            self.eng.seq_release(s)
        gk.gk_prefix_release(self.eng.pool, self.base)


def calibrate(Hq=32, Hkv=8, d=128, device="cuda"):
    import torch
    g = Hq // Hkv
    hot = 32768 + 16
    cold = 256 * 2048 + 64 * 4096 + 4096
    eng = Engine(1, Hq, Hkv, d, hot, cold, 1, seed=1, device=device)
    eng.hot_k.normal_()
    eng.hot_v.normal_()
    eng.cold_k.normal_()
    eng.cold_v.normal_()
    pool = eng.pool
    kv_tok = 2 * Hkv * d * 2

    flat_pts, suf_pts, cas_pts, merge_pts = [], [], [], []
    tile_pts, sm_pts = [], []
    for B, lp, s in [(8, 2048, 256), (32, 4096, 512), (64, 16384, 1024), (128, 8192, 512), (256, 4096, 1024)]:
        c = _Case(eng, B, lp, s, Hq, d)
        t_flat = _time(lambda: gk.gk_decode_dense(pool, None, 0, c.batch, c.plan))
        t_pre = _time(lambda: gk.gk_cascade_prefix(pool, None, 0, c.batch, c.plan))
        t_suf = _time(lambda: gk.gk_cascade_suffix(pool, None, 0, c.batch, c.plan))
        t_mrg = _time(lambda: gk.gk_cascade_merge(pool, None, 0, c.batch, c.plan))
        t_cas = _time(lambda: gk.gk_decode_cascade(pool, None, 0, c.batch, c.plan))
        flat_pts.append((c.info["dense_bytes"], t_flat))
        suf_pts.append((c.info["suffix_bytes"], t_suf))
        merge_pts.append((B * Hq, t_mrg))
        if c.info["prefix_ctas"] <= 152:   # one wave of items
            tile_pts.append((c.info["prefix_tiles_per_item"], t_pre))
        cas_pts.append((dict(c.info), t_cas, B))
        c.close()
    # split plans: prefix items of C tiles alone, and the whole split cascade
    for C in (16, 32, 64, 128):
        c = _Case(eng, 64, 16384, 1024, Hq, d, gk.GK_CASCADE_SPLIT, C)
        if c.info["cascade_split"]:
            t_pre = _time(lambda: gk.gk_cascade_prefix(pool, None, 0, c.batch, c.plan))
            t_cas = _time(lambda: gk.gk_decode_cascade(pool, None, 0, c.batch, c.plan))
            tile_pts.append((c.info["prefix_tiles_per_item"], t_pre))
            cas_pts.append((dict(c.info), t_cas, 64))
        c.close()
    # the gather alone on part of the SMs: long items (one key split, 64 of them at
    # M_eff 2048) leave their CTAs no suffix share, so the suffix runs on the other
    # SMs only, well below HBM saturation
    c = _Case(eng, 512, 16384, 128, Hq, d, gk.GK_CASCADE_SPLIT, 128)
    if c.info["cascade_split"]:
        t_suf = _time(lambda: gk.gk_cascade_suffix(pool, None, 0, c.batch, c.plan))
        n_sms = c.info["suffix_ctas"] - c.info["prefix_ctas"]
        sm_pts.append((n_sms, c.info["suffix_bytes"] / (t_suf * 1e3)))
    c.close()
    eng.close()
    torch.cuda.synchronize()

    keep = ("max_m_eff", "prefix_bytes", "prefix_ctas", "suffix_bytes", "suffix_ctas", "cascade_split",
            "prefix_tiles_per_item")
    return refit(dict(flat=flat_pts, suffix=suf_pts, merge=merge_pts, tile=tile_pts, gather_sm=sm_pts,
                      cascade=[t for _, t, _ in cas_pts],
                      cascade_info=[dict({k: i[k] for k in keep}, B=B, Hq=Hq) for i, _, B in cas_pts]))


# An item of a split plan shares HBM with a gather that keeps it busy, and its
# K/V tiles wait longer: on GB300 a 32-tile item beside the benchmark layer's
# gather ran 1.9-2.0 us per tile against 1.53-1.56 us alone (per-phase
# %globaltimer stamps in an instrumented build), a ratio of about 1.28.
SPLIT_TILE_RATIO = 1.28


def _linfit(pts):
    x = np.array([p[0] for p in pts], float)
    y = np.array([p[1] for p in pts], float)
    A = np.vstack([np.ones_like(x), x]).T
    (c0, slope), *_ = np.linalg.lstsq(A, y, rcond=None)
    return max(0.0, float(c0)), float(slope)


def refit(measured, num_sms=152):
    """Cost-model coefficients from the measured points (intercepts are fixed costs)."""
    c_flat, s_flat = _linfit(measured["flat"])
    c_suf, s_suf = _linfit(measured["suffix"])
    c_mrg, s_mrg = _linfit(measured["merge"])
    item, tile = _linfit(measured["tile"])
    cm = dict(c_flat_us=c_flat, bw_flat_gbs=1.0 / max(s_flat, 1e-12) / 1e3, c_cascade_us=0.0,
              bw_prefix_gbs=6000.0, bw_suffix_gbs=1.0 / max(s_suf, 1e-12) / 1e3, c_merge_us=max(s_mrg, 0.0),
              prefix_tile_us=max(tile, 1e-3), prefix_item_us=item, gather_sm_gbs=44.0, c_gather_us=c_suf,
              prefix_tile_split_us=max(tile, 1e-3) * SPLIT_TILE_RATIO)
    # per-SM gather bandwidth: the suffix alone on the SMs the long items leave it
    per_sm = [bw / n for n, bw in measured["gather_sm"] if n > 0]
    if per_sm:
        cm["gather_sm_gbs"] = float(np.median(per_sm))
    # the cascade's fixed cost: the merge launch's intercept plus the mean residual
    # of the whole cascade over the model when it is positive
    res = []
    for info, t_cas in zip(measured["cascade_info"], measured["cascade"]):
        tile_us = cm["prefix_tile_split_us"] if info["cascade_split"] else cm["prefix_tile_us"]
        item_us = info["prefix_tiles_per_item"] * tile_us + cm["prefix_item_us"]
        if info["cascade_split"]:
            bal = (info["suffix_bytes"] / (cm["gather_sm_gbs"] * 1e3) + info["prefix_ctas"] * item_us) / num_sms
            levels = max(item_us, bal, (info["suffix_bytes"] + info["prefix_bytes"]) / (cm["bw_suffix_gbs"] * 1e3))
        else:
            waves = -(-info["prefix_ctas"] // num_sms)
            levels = (max(info["prefix_bytes"] / (cm["bw_prefix_gbs"] * 1e3), waves * item_us) if info["prefix_ctas"] else 0.0)
            levels += cm["c_gather_us"] + info["suffix_bytes"] / (cm["bw_suffix_gbs"] * 1e3)
        res.append(t_cas - (c_mrg + levels + cm["c_merge_us"] * info["B"] * info["Hq"]))
    cm["c_cascade_us"] = c_mrg + max(0.0, float(np.mean(res)))
    cm["measured"] = measured
    return cm


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None)
    a = ap.parse_args()
    from . import build
    build.build()
    cm = calibrate()
    text = json.dumps(cm, indent=1)
    if a.out:
        with open(a.out, "w") as f:
            f.write(text)
    print(text)


if __name__ == "__main__":
    main()
