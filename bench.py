#!/usr/bin/env python
"""Decode-step benchmark of the shared-prefix paged attention library on GB300.

Workload (default, the largest that fits one GPU): Qwen-2.5-14B attention
geometry (Hq 40, Hkv 8, d 128, bf16, 48 layers), 8 shared prefixes with lengths
log-uniform in 2K..16K tokens in the HOT pool, 16..64 requests per prefix (368
in all, interleaved in the batch) with suffixes uniform in 128..4096 tokens in a
page-size-1 COLD pool with shuffled slots.  One step = the whole decode step of
all layers:
  host: gk_seq_append_slots (one token per request), gk_seq_tables,
  gk_plan_update, gk_dispatch
  device, per layer: copy-on-write copies if the step has any (gk_append_kv with
  n = 0), then the dispatcher's backend with the step's token appended by the
  decode itself (cascade: prefix contraction beside the suffix gather, LSE
  merge; or dense).
Metric: decode attention queries/s per layer = B * L / step time.
--config 2, 3 and 5 select the other multi-agent workloads.

--impl reference times the fp64 CPU oracle instead (there is no other
implementation to run); each of its steps is a bounded sample of one layer.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
for _p in (ROOT, os.path.join(ROOT, "tests")):
    if _p not in sys.path:
        sys.path.insert(0, _p)

METRIC = "decode attention queries/s per layer"
UNIT = "queries/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--override", action="append", default=[], metavar="KEY=INT",
                    help="workload override passed to synth.workloads.config (e.g. B=512, Lp=16384)")
    ap.add_argument("--stages-only", action="store_true",
                    help="time each kernel alone on layer 0 (the 'stages' object) and print only that")
    ap.add_argument("--backend", choices=["auto", "cascade", "dense"], default="auto")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="run only this many layers (small profiling case)")
    ap.add_argument("--append", choices=["fused", "separate"], default="fused",
                    help="the step's new tokens written by the decode itself, or by gk_append_kv first")
    ap.add_argument("--prefix-tiles", type=int, default=0,
                    help="split cascade with this many 128-key tiles per prefix item (default: the planner's choice)")
    ap.add_argument("--arrangement", choices=["auto", "sequential", "split"], default="auto",
                    help="cascade arrangement (gk_pool_set_cascade_mode)")
    ap.add_argument("--gather-partition", choices=["stream", "per-request"], default="stream",
                    help="work split of the stand-alone gathers (gk_pool_set_gather_partition)")
    ap.add_argument("--no-stages", action="store_true",
                    help="skip the stand-alone timing of each kernel (the 'stages' object)")
    ap.add_argument("--no-sm-speeds", action="store_true",
                    help="plan split launches without per-SM speeds (by default they are measured after the "
                         "warm-up with gk_sm_speeds_measure)")
    return ap.parse_args()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x):
    """The largest of the ranks' values (the job's time for N replicas timed side by
    side); x itself when the process runs alone.  Works over NCCL or gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, units_per_replica, elapsed_ms):
    """Whole-job throughput of `world` replicas that each processed `units_per_replica`
    in at most `elapsed_ms` (the max over ranks)."""
    return world * units_per_replica / (elapsed_ms / 1e3)


class Clocks:
    """nvidia-smi samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")
    PERIOD_MS = 10

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, window=None):
        """Stop sampling; summary of the samples (see summary)."""
        self.rows = []
        if not self.proc:
            return self.summary(window)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                row = (float(f[1]), float(f[2]), [n for n, v in zip(names, f[5:9]) if v.lower() == "active"])
            except ValueError:
                continue
            t = None
            if len(f) >= 10:
                try:
                    t = time.mktime(time.strptime(f[9].split(".")[0], "%Y/%m/%d %H:%M:%S")) + \
                        (float("0." + f[9].split(".")[1]) if "." in f[9] else 0.0)
                except (ValueError, IndexError):
                    t = None
            self.rows.append((t,) + row)
        return self.summary(window)

    def summary(self, window=None):
        """Median SM clock, max clock and throttle reasons of the samples; with window =
        (t0, t1) (host epoch seconds around a timed region) only the samples taken inside it
        count, when there are any."""
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = getattr(self, "rows", [])
        inside = rows
        where = "all samples"
        if window is not None:
            t0, t1 = window
            sel = [r for r in rows if r[0] is not None and t0 - 0.001 <= r[0] <= t1 + 0.001]
            if sel:
                inside, where = sel, "inside the timed region"
            else:
                where = "none inside the timed region; all samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = sorted(r[1] for r in inside)
        reasons = sorted({n for r in inside for n in r[3]})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "which": where, "period_ms": self.PERIOD_MS}


# sources of each profiled kernel: a committed ncu summary counts only while they are unchanged
LEVELS_SRC = ("cascade_split.cu", "prefix_body.cuh", "prefix_warp_body.cuh", "gather_body.cuh", "device_common.cuh")
GATHER_SRC = ("gather_attn.cu", "gather_body.cuh", "device_common.cuh")
PREFIX_SRC = ("prefix_tc.cu", "prefix_body.cuh", "device_common.cuh")


def source_sha256(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "paged_kv_cache_pool_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def profile_tag(workload_name):
    """The name an ncu summary under profiles/ carries for a workload: its geometry and
    batch without the layer count, the suffix range or a --layers cut (a summary covers
    one launch, which is the same in every layer)."""
    t = re.sub(r"_first\d+layers$", "", workload_name)
    t = re.sub(r"_s\d+-\d+$", "", t)
    return re.sub(r"_\d+L_", "_", t)


def _profile_value(kernel, src_files, workload_name, key="traffic_bytes_per_launch"):
    """A figure (`key: value` line) of the committed ncu summary profiles/<kernel>_<tag>.md, if
    there is one for this workload and the kernel sources are unchanged since it was taken:
    traffic_bytes_per_launch (DRAM read + write per launch) or l2_throughput_pct."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{profile_tag(workload_name)}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(key + r":\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not h:
        return None
    return float(m.group(1)) if source_sha256(src_files) == h.group(1) else None


def _profile_traffic(kernel, src_files, workload_name):
    return _profile_value(kernel, src_files, workload_name)


# ----------------------------------------------------------------------------------------------
# oracle (CPU) timing: the --impl reference arm and the cpu_baseline field
# ----------------------------------------------------------------------------------------------
def _oracle_sample(w, n_req, start=0):
    """Time the oracle on n_req requests of layer 0 -> (seconds, requests, threads)."""
    from oracle import attention, reference
    from synth.gen import bf16_bits_to_f64
    cache = reference.ContextCache(w)
    q = reference.q_bits(w, 0, 0)
    reqs = [(start + i) % w.B for i in range(n_req)]
    ctx = [reference.context(w, r, 0, 0, cache) for r in reqs]     # gather (untimed)
    t0 = time.perf_counter()
    for r, (K, V) in zip(reqs, ctx):
        attention.attend_heads(bf16_bits_to_f64(q[r]), K, V)
    dt = time.perf_counter() - t0
    return dt, len(reqs), attention.threads()


def cpu_baseline(w, budget_s=12.0):
    from oracle import attention
    attention.build()
    dt, n, thr = _oracle_sample(w, 1)
    per = max(dt, 1e-3)
    n_req = max(1, min(w.B, int(budget_s / per)))
    dt, n, thr = _oracle_sample(w, n_req, start=1)
    return {"value": n / dt, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"fp64 C oracle, layer 0 of the workload, {n} of {w.B} requests "
                      f"(all {w.Hq} query heads, contexts gathered beforehand), {dt:.1f} s"}


def run_reference(a, w):
    rank, world, _ = _dist()
    if rank != 0:
        return
    from oracle import attention
    attention.build()
    dt1, _, thr = _oracle_sample(w, 1)
    # each timed step a sample of about 4 s, less when many steps are asked for, so that the
    # whole run stays near two and a half minutes
    per_step_s = max(0.5, min(4.0, 150.0 / max(1, a.steps)))
    n_req = max(1, min(w.B, int(per_step_s / max(dt1, 1e-3))))
    for i in range(a.warmup):
        _oracle_sample(w, 1, start=i)
    total_t, total_q = 0.0, 0
    for i in range(a.steps):
        dt, n, thr = _oracle_sample(w, n_req, start=i * n_req)
        total_t += dt
        total_q += n
    value = total_q / total_t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * total_t / a.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config_dict(w, "oracle"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                             "sample": f"each step: {n_req} requests of layer 0 (all query heads), fp64 C oracle"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def _config_dict(w, backend):
    s = [r.suffix_len for r in w.requests]
    return {"workload": w.name, "B": w.B, "layers": w.L, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.d,
            "prefix_lens": w.prefix_lens, "suffix_min": min(s), "suffix_max": max(s), "suffix_sum": sum(s),
            "cold_page_size": w.page_size, "backend": backend, "parallelism": "replicas",
            "l2": f"inputs larger than L2 (each layer reads a distinct {_layer_kv_mib(w)} MiB of K/V; "
                  f"{_layer_kv_mib(w) * w.L / 1024:.1f} GiB per step)"}


def _layer_kv_mib(w):
    """K/V bytes one layer of the cascade reads: each prefix once, every suffix."""
    tok = sum(w.prefix_lens) + sum(r.suffix_len for r in w.requests)
    return int(tok * 2 * w.Hkv * w.d * 2 / 2**20)


# ----------------------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------------------
def _set_arrangement(gk, pool, a):
    if a.prefix_tiles > 0:
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SPLIT, a.prefix_tiles)
    elif a.arrangement != "auto":
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SEQUENTIAL if a.arrangement == "sequential"
                                    else gk.GK_CASCADE_SPLIT, 0)
    else:
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_AUTO, 0)


def stage_rooflines(gk, torch, pool, batch, w, P, hbm, tc_burst, reps=7):
    """Each kernel of the path timed alone on layer 0 of the batch as it stands: a sequential
    cascade plan's prefix contraction (gk_cascade_prefix), suffix gather (gk_cascade_suffix) and
    merge (gk_cascade_merge), then the dense backend (gk_decode_dense).  L2 is flushed before
    every launch (leaving it clean); the median of `reps` CUDA-event timings on the launching
    stream is kept.  The prefix contraction and the suffix gather are also timed as a decode
    step runs them: one launch per layer, back to back (each overlaps its set-up with the end
    of the one before), time per launch.
    A kernel timed alone is compared with the burst peaks.  The flat backend's prefix
    re-reads mostly hit L2, so only its DRAM bytes (from its ncu summary) are held to HBM;
    its algorithmic bytes per second are reported as they are, next to the L2 throughput
    ncu measured against the L2's own peak."""
    import numpy as np
    B, Hq, d = w.B, w.Hq, w.d
    stream = torch.cuda.current_stream()
    # L2 flush: write a buffer larger than L2, then read another one, so that the timed
    # kernel starts from a cold L2 holding no dirty lines (their write-back would be timed)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    clean = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        ts = []
        for _ in range(reps + 1):
            flush.zero_()
            clean.max()
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts[1:]))          # ms; the first launch is a warm-up

    # no fused append in these timings: the batch's new-token arrays belong to one layer
    batch.c.d_new_k = None
    batch.c.d_new_v = None
    gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SEQUENTIAL, 0)
    plan = gk.gk_plan_build(pool, batch)
    try:
        info = gk.gk_plan_info(plan)
        s_tot = int(batch.suffix_len.sum())
        q_bytes = B * Hq * d * 2
        state = Hq * (d + 1) * 4                 # one partial state: O row and LSE of every query head
        _, segs = gk.gk_plan_segments(plan, False)
        n_suf_part = len(segs)                    # one partial state per suffix segment
        n_pre_part = info["num_partials"] - n_suf_part
        t_pre = timed(lambda: gk.gk_cascade_prefix(pool, stream, 0, batch, plan))
        t_suf = timed(lambda: gk.gk_cascade_suffix(pool, stream, 0, batch, plan))
        t_mrg = timed(lambda: gk.gk_cascade_merge(pool, stream, 0, batch, plan))
        t_den = timed(lambda: gk.gk_decode_dense(pool, stream, 0, batch, plan))

        # the same kernels back to back over every layer, as they run in a decode step's
        # stream (each layer reads its own pool rows: together far more than L2); per launch
        def chained(fn):
            flush.zero_()
            clean.max()
            e0.record(stream)
            for layer in range(w.L):
                fn(layer)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / w.L
        chained(lambda l: gk.gk_cascade_prefix(pool, stream, l, batch, plan))   # warm-up
        c_pre = chained(lambda l: gk.gk_cascade_prefix(pool, stream, l, batch, plan))
        c_suf = chained(lambda l: gk.gk_cascade_suffix(pool, stream, l, batch, plan))
        if gk.gk_device_error(pool, stream):
            raise RuntimeError("device error word set in the stage timings")
        flops = info["prefix_flops"]
        pre_bytes = info["prefix_bytes"] + q_bytes + n_pre_part * state
        suf_bytes = info["suffix_bytes"] + s_tot * 4 // P + q_bytes + n_suf_part * state
        den_bytes = info["dense_bytes"] + s_tot * 4 // P + q_bytes + B * Hq * (d + 1) * 4
        out = {
            "prefix": {"kernel": "prefix_kernel", "ms": t_pre, "flops": flops, "bytes": pre_bytes,
                       "items": info["prefix_ctas"], "tiles_per_item": info["prefix_tiles_per_item"],
                       "tflops": flops / (t_pre * 1e-3) / 1e12, "gbs": pre_bytes / (t_pre * 1e-3) / 1e9},
            "suffix": {"kernel": "gather_kernel", "ms": t_suf, "bytes": suf_bytes, "ctas": info["suffix_ctas"],
                       "gbs": suf_bytes / (t_suf * 1e-3) / 1e9},
            "merge": {"kernel": "merge_kernel", "ms": t_mrg, "partials": info["num_partials"],
                      "bytes": info["num_partials"] * state + B * state},
            "dense": {"kernel": "gather_kernel (+ merge_kernel when a request is split)", "ms": t_den,
                      "bytes": den_bytes, "ctas": info["dense_ctas"], "merge": info["dense_merge"],
                      "gbs": den_bytes / (t_den * 1e-3) / 1e9},
        }
        out["prefix"]["tensor_frac"] = out["prefix"]["tflops"] / tc_burst
        out["prefix_chained"] = {"ms": c_pre, "launches": w.L, "tflops": flops / (c_pre * 1e-3) / 1e12,
                                 "tensor_frac": flops / (c_pre * 1e-3) / 1e12 / tc_burst,
                                 "gbs": pre_bytes / (c_pre * 1e-3) / 1e9}
        out["suffix_chained"] = {"ms": c_suf, "launches": w.L, "gbs": suf_bytes / (c_suf * 1e-3) / 1e9,
                                 "hbm_frac": suf_bytes / (c_suf * 1e-3) / 1e9 / hbm}
        out["prefix"]["hbm_frac"] = out["prefix"]["gbs"] / hbm
        out["prefix"]["bound"] = "tensor" if flops / pre_bytes > tc_burst * 1e3 / hbm else "hbm"
        out["suffix"]["hbm_frac"] = out["suffix"]["gbs"] / hbm
        m = out["merge"]
        m["gbs"] = m["bytes"] / (t_mrg * 1e-3) / 1e9
        # DRAM bytes per launch from the committed ncu summaries (null unless one covers this
        # workload and the kernel's sources are unchanged)
        out["prefix"]["traffic"] = _profile_traffic("prefix_kernel", PREFIX_SRC, w.name)
        out["suffix"]["traffic"] = _profile_traffic("suffix_gather", GATHER_SRC, w.name)
        dn = out["dense"]
        dn["traffic"] = _profile_traffic("dense_gather", GATHER_SRC, w.name)
        # the flat backend: DRAM bytes against HBM; its algorithmic rate counts L2 hits, so it
        # is no fraction of HBM; ncu's L2 throughput (of the L2's peak) says how close L2 runs
        dn["algorithmic_gbs"] = dn.pop("gbs")
        dn["dram_gbs"] = dn["traffic"] / (t_den * 1e-3) / 1e9 if dn["traffic"] else None
        dn["hbm_frac"] = dn["dram_gbs"] / hbm if dn["dram_gbs"] else None
        dn["l2_throughput_pct"] = _profile_value("dense_gather", GATHER_SRC, w.name, "l2_throughput_pct")
        out["peaks"] = {"hbm_gbs": hbm, "bf16_tflops": tc_burst, "which": "burst (kernels timed alone)"}
        out["timing"] = (f"layer 0, sequential plan, L2 flushed before each launch, median of {reps}; "
                         f"*_chained: one launch per layer back to back over the {w.L} layers, L2 flushed "
                         f"before the chain, time per launch")
        return out
    finally:
        gk.gk_plan_destroy(plan)


def chained_kernels(gk, torch, pool, batch, plan, w, backend, q_all, out_all, lse_all, chains=5):
    """Per-launch time of each kernel of the step's backend: the kernel launched for every
    layer back to back on one stream (each launch overlaps its set-up with the end of the one
    before, as in a decode step), L2 flushed before each chain, median of `chains` chains.
    The step's new tokens are in the pool by now, so the chains read them from there."""
    import numpy as np
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    clean = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    batch.c.d_new_k = None
    batch.c.d_new_v = None

    def chain(fn):
        ts = []
        for _ in range(chains + 1):
            flush.zero_()
            clean.max()
            e0.record(stream)
            for l in range(w.L):
                batch.set_device(d_q=q_all[l], d_out=out_all[l], d_lse=lse_all[l])
                fn(l)
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / w.L)
        return {"ms": float(np.median(ts[1:])), "launches": w.L, "chains": chains}

    out = {}
    if backend == "cascade":
        out["cascade_levels"] = chain(lambda l: gk.gk_cascade_levels(pool, stream, l, batch, plan))
        out["lse_merge"] = chain(lambda l: gk.gk_cascade_merge(pool, stream, l, batch, plan))
        out["layer"] = chain(lambda l: gk.gk_decode_cascade(pool, stream, l, batch, plan))
        # a chain of merges alone is bound by their launches; inside the step each merge's
        # launch and set-up overlap the split launch before it, so its cost there is what it
        # adds to a layer
        out["lse_merge"]["in_step_ms"] = out["layer"]["ms"] - out["cascade_levels"]["ms"]
    else:
        out["dense_gather"] = chain(lambda l: gk.gk_decode_dense(pool, stream, l, batch, plan))
    if gk.gk_device_error(pool, stream):
        raise RuntimeError("device error word set in the kernel chains")
    return out


def run_stages_only(a, w):
    """The 'stages' object alone: each kernel timed by itself on layer 0 of the workload as
    it is set up (no decode steps before it).  Used to profile one kernel launch."""
    import torch
    from gpu_workload import GpuWorkload
    from paged_kv_cache_pool_gb300 import binding as gk
    torch.cuda.set_device(0)
    gw = GpuWorkload(w)
    try:
        cm_path = os.path.join(ROOT, "paged_kv_cache_pool_gb300", "cost_model_gb300.json")
        if os.path.exists(cm_path):
            gk.gk_cost_model_load(gw.eng.pool, open(cm_path).read())
        b = gw.batch()
        q = gw.q(0)
        out, lse = gw.outputs()
        b.set_device(d_q=q, d_out=out, d_lse=lse)
        peaks, _ = _peaks()
        st = stage_rooflines(gk, torch, gw.eng.pool, b, w, gw.P, float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                             float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])))
        print(json.dumps({"workload": w.name, "stages": st}))
    finally:
        gw.close()


def run_ours(a, w):
    import numpy as np
    import torch
    from gpu_workload import GpuWorkload
    from paged_kv_cache_pool_gb300 import binding as gk
    from synth import device as sdev
    from synth.gen import KIND_NEW_K, KIND_NEW_V, KIND_Q, stream_key

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    total_steps = a.warmup + a.steps + (a.warmup + a.steps if not a.no_e2e else 0) + 2
    gw = GpuWorkload(w, extra_steps=total_steps)
    eng = gw.eng
    pool = eng.pool
    cm_path = os.path.join(ROOT, "paged_kv_cache_pool_gb300", "cost_model_gb300.json")
    if os.path.exists(cm_path):
        gk.gk_cost_model_load(pool, open(cm_path).read())
    _set_arrangement(gk, pool, a)
    if a.gather_partition == "per-request":
        gk.gk_pool_set_gather_partition(pool, gk.GK_PARTITION_PER_REQUEST)
    L, B, Hq, Hkv, d = w.L, w.B, w.Hq, w.Hkv, w.d
    stream = torch.cuda.current_stream()
    bf = torch.bfloat16

    # step inputs, resident on the device (one set reused every step)
    q_all = torch.empty((L, B, Hq, d), dtype=bf, device="cuda")
    newk = torch.empty((L, B, Hkv, d), dtype=bf, device="cuda")
    newv = torch.empty_like(newk)
    for l in range(L):
        sdev.fill_normal(q_all[l].view(-1), stream_key(w.seed, KIND_Q, l, 0))
        sdev.fill_normal(newk[l].view(-1), stream_key(w.seed, KIND_NEW_K, l, 0))
        sdev.fill_normal(newv[l].view(-1), stream_key(w.seed, KIND_NEW_V, l, 0))
    out_all = torch.empty((L, B, Hq, d), dtype=torch.float32, device="cuda")
    lse_all = torch.empty((L, B, Hq), dtype=torch.float32, device="cuda")

    seqs = np.asarray(gw.seqs, dtype=np.int32)
    P = gw.P
    max_len = max(r.suffix_len for r in w.requests) + total_steps + 1
    max_blocks = -(-max_len // P)
    h_table = torch.empty((B, max_blocks), dtype=torch.int32).pin_memory()
    h_slots = torch.empty(B, dtype=torch.int64).pin_memory()
    d_slots = torch.empty(B, dtype=torch.int64, device="cuda")
    h_lens = np.empty(B, dtype=np.int32)
    h_cow = torch.empty(2 * B, dtype=torch.int32).pin_memory()
    d_table = torch.empty((B, max_blocks), dtype=torch.int32, device="cuda")
    d_cow = torch.empty(2 * B, dtype=torch.int32, device="cuda")
    staged = torch.cuda.Event()
    bases = np.array([gw.bases[r.prefix] if r.prefix >= 0 else -1 for r in w.requests], dtype=np.int64)
    lps = np.array([w.prefix_lens[r.prefix] if r.prefix >= 0 else 0 for r in w.requests], dtype=np.int32)
    batch = gk.Batch(bases, lps, np.zeros(B, np.int32), d_table, max_blocks)
    plan = [None]
    forced = {"cascade": gk.GK_BACKEND_CASCADE, "dense": gk.GK_BACKEND_DENSE}.get(a.backend)
    launches = [0]
    dense_merge = [0]
    split = [0]
    choices = []
    predicted = []

    def step(q=q_all, k=newk, v=newv, out=out_all, lse=lse_all):
        # a0: host plan (append one token per request, tables, plan, dispatch)
        slots, cow = gk.gk_seq_append_slots(pool, seqs)
        staged.synchronize()                    # the previous step's staging copies have left
        h_slots.numpy()[:] = slots
        ncow = len(cow)
        if ncow:
            h_cow.numpy()[:2 * ncow] = cow.reshape(-1)
        gk.gk_seq_tables(pool, seqs, max_blocks, h_table.numpy(), h_lens)
        batch.suffix_len[:] = h_lens
        d_table.copy_(h_table, non_blocking=True)
        if a.append != "fused":
            d_slots.copy_(h_slots, non_blocking=True)
        if ncow:
            d_cow[:2 * ncow].copy_(h_cow[:2 * ncow], non_blocking=True)
        staged.record(stream)
        if plan[0] is None:
            plan[0] = gk.gk_plan_build(pool, batch, stream)
        else:
            gk.gk_plan_update(pool, plan[0], batch, stream)
        pinfo = gk.gk_plan_info(plan[0])
        dense_merge[0] = pinfo["dense_merge"]
        split[0] = pinfo["cascade_split"]
        choice, t_d, t_c = gk.gk_dispatch(pool, plan[0])
        predicted.append((t_d, t_c))
        if forced is not None:
            choice = forced
        choices.append(choice)
        for l in range(L):
            if a.append == "fused":
                # the step's new tokens are appended by the decode itself; copy-on-write
                # copies, when the step has any, come first
                if ncow:
                    gk.gk_append_kv(pool, stream, l, None, None, None, d_cow, n=0, n_cow=ncow)
                    launches[0] += 1
                batch.set_device(d_q=q[l], d_out=out[l], d_lse=lse[l], d_new_k=k[l], d_new_v=v[l])
            else:
                gk.gk_append_kv(pool, stream, l, d_slots, k[l], v[l], d_cow if ncow else None, n=B, n_cow=ncow)
                launches[0] += 1 + (1 if ncow else 0)
                batch.set_device(d_q=q[l], d_out=out[l], d_lse=lse[l])
            if choice == gk.GK_BACKEND_CASCADE:
                gk.gk_decode_cascade(pool, stream, l, batch, plan[0])
                launches[0] += (1 if split[0] else 2) + 1
            else:
                gk.gk_decode_dense(pool, stream, l, batch, plan[0])
                launches[0] += 1 + dense_merge[0]

    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    err = gk.gk_device_error(pool, stream)
    if err:
        raise RuntimeError(f"device error word {err} during warm-up")
    # per-SM gather speeds from the step plan's own suffix gather (layer 0, the step's new
    # tokens left out so that the pool is not written), then one more warm-up step planned
    # with them
    sm_speeds = "off"
    if not a.no_sm_speeds and int(batch.suffix_len.sum()) > 0:
        batch.set_device(d_q=q_all[0], d_out=out_all[0], d_lse=lse_all[0])
        batch.c.d_new_k = None
        batch.c.d_new_v = None
        sp = gk.gk_sm_speeds_measure(pool, stream, 0, batch, plan[0], reps=5)
        sm_speeds = f"measured (gk_sm_speeds_measure, 5 launches; slowest {sp.min():.3f}, fastest {sp.max():.3f})"
        step()
        torch.cuda.synchronize()
        err = gk.gk_device_error(pool, stream)
        if err:
            raise RuntimeError(f"device error word {err} after measuring SM speeds")
    if world > 1:
        torch.distributed.barrier()

    # ---- timed region: device-resident inputs, nothing but the steps in the stream ----
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    vis_list = [x for x in vis.split(",") if x.strip()]
    gpu_index = vis_list[local].strip() if local < len(vis_list) else str(local)
    clocks = Clocks(gpu_index)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    launches[0] = 0
    n_choice0 = len(choices)
    # Python's cyclic garbage collector stays off inside the timed regions, as timeit keeps
    # it: a full collection of this process's objects takes tens of ms of host time, which
    # would otherwise land inside some step's host work
    gc.collect()
    gc.disable()
    w0 = time.time()
    t_start.record(stream)
    for i in range(a.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    gc.enable()
    gpu_launches = launches[0]
    elapsed_ms = t_start.elapsed_time(t_end)
    err = gk.gk_device_error(pool, stream)
    if err:
        raise RuntimeError(f"device error word {err} in the timed region")
    step_choices = choices[n_choice0:]
    elapsed_ms = max_over_ranks(elapsed_ms)
    ms_per_step = elapsed_ms / a.steps
    value = replica_throughput(world, B * L * a.steps, elapsed_ms)

    # ---- e2e: host buffers, copies inside the timed region ----
    e2e = None
    if not a.no_e2e:
        hq = torch.empty_like(q_all, device="cpu").pin_memory()
        hk = torch.empty_like(newk, device="cpu").pin_memory()
        hv = torch.empty_like(newv, device="cpu").pin_memory()
        hq.copy_(q_all)
        hk.copy_(newk)
        hv.copy_(newv)
        ho = torch.empty_like(out_all, device="cpu").pin_memory()
        hl = torch.empty_like(lse_all, device="cpu").pin_memory()
        # Triple-buffered device inputs and outputs, each direction on a copy stream of its
        # own: step t+1's inputs come in and step t's outputs go out while the compute
        # stream runs, and a step waits for the outputs of the step three before it to have
        # left its buffer.  (One copy of a step's inputs or outputs now and then takes tens
        # of ms longer than its 1.2-1.9 ms; with two buffers and one copy stream those held
        # up the compute stream.  Copies in chunks of a few layers, each layer waiting for its
        # own, were slower: the waits and event records between a layer's kernels cost more
        # than the first and last copies of the region that they shorten.)
        NB = 3
        dev_in = [(torch.empty_like(q_all), torch.empty_like(newk), torch.empty_like(newv)) for _ in range(NB)]
        dev_out = [(torch.empty_like(out_all), torch.empty_like(lse_all)) for _ in range(NB)]
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(NB)]      # inputs of buffer i have landed
        ev_used = [torch.cuda.Event() for _ in range(NB)]    # the compute that read/wrote buffer i is done
        ev_out = [torch.cuda.Event() for _ in range(NB)]     # outputs of buffer i have left
        for e in ev_used + ev_out:
            e.record(stream)

        def h2d(i):
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(ev_used[i])
                for dst, src in zip(dev_in[i], (hq, hk, hv)):
                    dst.copy_(src, non_blocking=True)
                ev_in[i].record(h2d_s)

        def run_steps(n):
            h2d(0)
            for t in range(n):
                i = t % NB
                stream.wait_event(ev_in[i])
                stream.wait_event(ev_out[i])   # step t - NB has left this output buffer
                step(*dev_in[i], *dev_out[i])
                ev_used[i].record(stream)
                if t + 1 < n:
                    h2d((t + 1) % NB)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(ev_used[i])
                    ho.copy_(dev_out[i][0], non_blocking=True)
                    hl.copy_(dev_out[i][1], non_blocking=True)
                    ev_out[i].record(d2h_s)
            stream.wait_stream(h2d_s)
            stream.wait_stream(d2h_s)

        run_steps(a.warmup)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gc.collect()
        gc.disable()
        v0 = time.time()
        e0.record(stream)
        h2d_s.wait_event(e0)
        d2h_s.wait_event(e0)
        run_steps(a.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_window = (v0, time.time())
        gc.enable()
        ems = max_over_ranks(e0.elapsed_time(e1))
        h2d_bytes = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2 + B * max_blocks * 4
        d2h_bytes = ho.numel() * 4 + hl.numel() * 4
        e2e = {"value": replica_throughput(world, B * L * a.steps, ems), "unit": UNIT,
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "ms_per_step": ems / a.steps,
               "copies": "triple-buffered, one copy stream each way, overlapping the neighbouring steps' compute"}

    time.sleep(0.1)   # let the sampler report the samples of the regions' ends
    clk = clocks.stop((w0, w1))
    if e2e is not None:
        e2e["clocks"] = clocks.summary(e2e_window)

    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        gw.close()
        return

    # ---- per-kernel times: each kernel of the step's backend launched for every layer back
    # to back, as the step runs them (no event between two kernels of a layer, which would
    # stop the next one from starting early); time per launch, after the timed region ----
    info = gk.gk_plan_info(plan[0])
    backend_name = "cascade" if step_choices and step_choices[0] == gk.GK_BACKEND_CASCADE else "dense"
    kernels = chained_kernels(gk, torch, pool, batch, plan[0], w, backend_name, q_all, out_all, lse_all)
    peaks, peak_src = _peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tc_peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    s_tot = int(batch.suffix_len.sum())
    # algorithmic bytes per launch (prefix K/V once per group, suffix K/V, slots, queries, partial states)
    partial_bytes = info["num_partials"] * Hq * (d + 1) * 4
    levels_bytes = (info["prefix_bytes"] + info["suffix_bytes"] + s_tot * 4 // P + B * Hq * d * 2 + partial_bytes)
    dense_bytes = info["dense_bytes"] + s_tot * 4 // P + B * Hq * d * 2 + B * Hq * (d + 1) * 4
    if "cascade_levels" in kernels:
        kl = kernels["cascade_levels"]
        kl.update(bytes=levels_bytes, flops=info["prefix_flops"], gbs=levels_bytes / (kl["ms"] * 1e-3) / 1e9,
                  tflops=info["prefix_flops"] / (kl["ms"] * 1e-3) / 1e12,
                  arrangement="split" if info["cascade_split"] else "sequential")
    if "dense_gather" in kernels:
        kd_ = kernels["dense_gather"]
        kd_.update(bytes=dense_bytes, gbs=dense_bytes / (kd_["ms"] * 1e-3) / 1e9)
    # dominant kernel -> roofline (the cascade's two levels are one launch in a split plan)
    dom = max(((k, v["ms"]) for k, v in kernels.items() if "bytes" in v), key=lambda x: x[1])[0]
    kd = kernels[dom]
    if dom == "cascade_levels" and kd["flops"] / kd["bytes"] > tc_peak * 1e3 / hbm:
        roof = {"kernel": dom, "bound": "tensor", "achieved": kd["tflops"], "peak": tc_peak, "unit": "TFLOP/s",
                "frac": kd["tflops"] / tc_peak, "traffic": _profile_traffic("cascade_levels", LEVELS_SRC, w.name)}
    elif dom == "cascade_levels":
        roof = {"kernel": dom, "bound": "hbm", "achieved": kd["gbs"], "peak": hbm, "unit": "GB/s",
                "frac": kd["gbs"] / hbm, "traffic": _profile_traffic("cascade_levels", LEVELS_SRC, w.name)}
    else:
        # the flat backend re-reads each prefix from L2: its DRAM bytes (ncu) against HBM
        tr = _profile_traffic("dense_gather", GATHER_SRC, w.name)
        roof = {"kernel": dom, "bound": "hbm", "achieved": tr / (kd["ms"] * 1e-3) / 1e9 if tr else None,
                "peak": hbm, "unit": "GB/s", "frac": tr / (kd["ms"] * 1e-3) / 1e9 / hbm if tr else None,
                "traffic": tr, "algorithmic_gbs": kd["gbs"],
                "l2_throughput_pct": _profile_value("dense_gather", GATHER_SRC, w.name, "l2_throughput_pct")}
    roof["peak_source"] = f"{peak_src} ({'bf16_tflops_sustained' if roof['bound'] == 'tensor' else 'hbm_gbs'})"
    roof["timing"] = (f"{kd['launches']} launches back to back (one per layer, L2 flushed before the chain), "
                      f"median of {kd['chains']} chains; times {L} layers = {kd['ms'] * L:.3f} ms "
                      f"of the {ms_per_step:.3f} ms step")
    stages = None
    if not a.no_stages:
        stages = stage_rooflines(gk, torch, pool, batch, w, P, hbm,
                                 float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])))
        _set_arrangement(gk, pool, a)
    cpu = None
    if not a.no_cpu:
        cpu = cpu_baseline(w)
    pd, pc = predicted[-1]
    layer_us = ms_per_step * 1e3 / L
    dispatch = {"choice": backend_name, "predicted_dense_us": pd, "predicted_cascade_us": pc,
                "measured_layer_us": layer_us,
                "prediction_error": ((pc if backend_name == "cascade" else pd) - layer_us) / layer_us,
                "cost_model": "paged_kv_cache_pool_gb300/cost_model_gb300.json" if os.path.exists(cm_path) else "library defaults"}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": dict(_config_dict(w, backend_name), sm_speeds=sm_speeds),
            "clocks": clk, "e2e": e2e, "gpu_launches": gpu_launches, "roofline": roof,
            "cpu_baseline": cpu, "kernels": kernels, "stages": stages, "dispatch": dispatch,
            "query_rows_per_s": value * Hq,
            "plan": info}
    print(json.dumps(line))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    gw.close()


def main():
    a = _args()
    from synth import workloads
    ov = {}
    for kv in a.override:
        k, v = kv.split("=", 1)
        ov[k] = int(v)
    w = workloads.config(a.config, **ov)
    if a.layers:
        w.L = a.layers
        w.name += f"_first{a.layers}layers"
    if a.impl == "reference":
        run_reference(a, w)
    else:
        from paged_kv_cache_pool_gb300 import build
        from synth import device
        build.build()
        device.build()
        if a.stages_only:
            run_stages_only(a, w)
        else:
            run_ours(a, w)


if __name__ == "__main__":
    main()
