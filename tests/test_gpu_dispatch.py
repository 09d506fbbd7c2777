"""The dispatcher against measured GB300 times, not against a restatement of itself.

GraniKV Section 3.6 routes each step between its prefix kernels on M_eff and
says the threshold must be re-fit per GPU (Appendix B.4b); here the re-fit is
gk_calibrate and the rule is gk_dispatch over the plan the planner arranged
(flat backend, cascade over tensor-core items, cascade over warp-MMA items).
  * gk_calibrate runs through the C ABI, installs a model, and writes JSON that
    gk_cost_model_load reads back and that routes shared-prefix workloads to
    the cascade and unshared ones to the flat backend;
  * on a grid of (Lp, B) cells the three choices are timed through the ABI
    (one layer, L2 emptied before each launch, median of 11 launches, as
    gk_calibrate times the cases it fits), and the
    default plan's pick (GK_PREFIX_AUTO, then gk_dispatch, with the committed
    GB300 model) must be within 10 % of the fastest choice's time, and the
    predicted time of each choice the dispatcher weighs within 25 % of its
    measured time.  (A step whose groups stack at most 64 rows per KV head never
    takes tensor-core items, gk.h GK_PREFIX_AUTO, so that prediction is not one
    the dispatcher uses there; it is timed and reported all the same.)  CUDA
    events on this GPU resolve about 1 us, so differences under 2.5 us pass
    either bound.
"""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timing]

from paged_kv_cache_pool_gb300 import binding as gk  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CM_PATH = os.path.join(ROOT, "paged_kv_cache_pool_gb300", "cost_model_gb300.json")
SLACK_US = 2.5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_pool_gb300 import build
    build.build()


def test_calibrate_through_the_abi(tmp_path):
    from paged_kv_cache_pool_gb300.calibrate import calibrate
    out = str(tmp_path / "cm.json")
    cm = calibrate(out=out)
    for k in gk.COST_MODEL_KEYS:
        assert k in cm and np.isfinite(cm[k]), k
    assert 1000 < cm["bw_flat_gbs"] < 100000 and 1000 < cm["bw_suffix_gbs"] < 12000
    assert 0.2 < cm["prefix_tile_us"] < 10 and cm["prefix_tile_split_us"] >= cm["prefix_tile_us"]
    assert cm["warp_tile_us"] > 0 and cm["warp_group_us"] >= 0 and 5 < cm["gather_sm_gbs"] < 500
    assert len(cm["measured"]["warp items (tiles per item, tiles x row groups, us)"]) >= 3
    # the file loads as it is, and routes: five shared-prefix workloads to the cascade,
    # 64 requests with 64 distinct 4096-token prefixes to the flat backend
    from synth import workloads
    text = open(out).read()
    for n in (2, 3, 4, 5):
        w = workloads.config(n)
        pool = gk.gk_pool_create(w.L, w.Hq, w.Hkv, w.d, w.hot_tokens(), w.cold_slots(), w.page_size, 0)
        try:
            gk.gk_cost_model_load(pool, text)
            bases = [gk.gk_prefix_alloc(pool, lp) for lp in w.prefix_lens]
            b = gk.Batch([bases[r.prefix] for r in w.requests], [w.prefix_lens[r.prefix] for r in w.requests],
                         [r.suffix_len for r in w.requests], None, 8192)
            plan = gk.gk_plan_build(pool, b)
            choice, td, tc = gk.gk_dispatch(pool, plan)
            assert choice == gk.GK_BACKEND_CASCADE and tc < td, (n, td, tc)
            gk.gk_plan_destroy(plan)
        finally:
            gk.gk_pool_destroy(pool)
    pool = gk.gk_pool_create(1, 32, 8, 128, 64 * 4096, 64 * 256, 1, 0)
    try:
        gk.gk_cost_model_load(pool, text)
        bases = [gk.gk_prefix_alloc(pool, 4096) for _ in range(64)]
        plan = gk.gk_plan_build(pool, gk.Batch(bases, [4096] * 64, [100] * 64, None, 256))
        choice, td, tc = gk.gk_dispatch(pool, plan)
        assert choice == gk.GK_BACKEND_DENSE and td < tc
        gk.gk_plan_destroy(plan)
    finally:
        gk.gk_pool_destroy(pool)


@pytest.mark.parametrize("lp,B", [(512, 8), (512, 128), (4096, 8), (4096, 128)])
def test_dispatcher_against_measured_times(lp, B):
    from paged_kv_cache_pool_gb300.engine import Engine
    Hq, Hkv, d = 32, 8, 128
    rng = np.random.default_rng([lp, B])
    s = rng.integers(16, 513, B).astype(np.int32)
    eng = Engine(1, Hq, Hkv, d, lp + 16, int(s.sum()) + 4096, 1, seed=3)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    clean = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        for t in (eng.hot_k, eng.hot_v, eng.cold_k, eng.cold_v):
            t.normal_()
        pool = eng.pool
        gk.gk_cost_model_load(pool, open(CM_PATH).read())
        base = eng.prefix_alloc(lp)
        seqs = [eng.seq_create() for _ in range(B)]
        eng.append_slots(np.repeat(np.asarray(seqs, np.int32), s))
        table = eng.block_tables(seqs)
        d_table = eng.to_device(table)
        batch = eng.batch([base] * B, [lp] * B, s.tolist(), d_table, table.shape[1])
        q = torch.randn((B, Hq, d), device="cuda").to(torch.bfloat16)
        out = torch.empty((B, Hq, d), device="cuda")
        lse = torch.empty((B, Hq), device="cuda")
        batch.set_device(d_q=q, d_out=out, d_lse=lse)

        def timed(fn, reps=11):
            ts = []
            for _ in range(reps + 1):
                flush.zero_()
                clean.max()
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
            return float(np.median(ts[1:]))

        meas, pred = {}, {}
        for kind, kernel in (("tensor", gk.GK_PREFIX_TENSOR), ("warp", gk.GK_PREFIX_WARP)):
            gk.gk_pool_set_prefix_kernel(pool, kernel)
            plan = gk.gk_plan_build(pool, batch)
            _, pred["dense"], pred[kind] = gk.gk_dispatch(pool, plan)
            meas[kind] = timed(lambda: gk.gk_decode_cascade(pool, None, 0, batch, plan))
            if kind == "tensor":
                meas["dense"] = timed(lambda: gk.gk_decode_dense(pool, None, 0, batch, plan))
            gk.gk_plan_destroy(plan)
        gk.gk_pool_set_prefix_kernel(pool, gk.GK_PREFIX_AUTO)
        plan = gk.gk_plan_build(pool, batch)
        choice, _, _ = gk.gk_dispatch(pool, plan)
        kind = "warp" if gk.gk_plan_info(plan)["prefix_kernel"] == gk.GK_PREFIX_WARP else "tensor"
        gk.gk_plan_destroy(plan)
        assert gk.gk_device_error(pool) == gk.GK_OK
        pick = "dense" if choice == gk.GK_BACKEND_DENSE else kind
        best = min(meas.values())
        report = json.dumps(dict(Lp=lp, B=B, pick=pick, measured=meas, predicted=pred))
        assert meas[pick] <= best * 1.10 or meas[pick] - best <= SLACK_US, report
        weighed = [k for k in meas if not (k == "tensor" and B * (Hq // Hkv) <= 64)]
        for k in weighed:
            assert abs(pred[k] - meas[k]) <= 0.25 * meas[k] or abs(pred[k] - meas[k]) <= SLACK_US, (k, report)
        print(report)
    finally:
        eng.close()
