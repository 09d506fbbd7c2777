"""gk_decode_dense_static: the allocation-free dense decode (fixed 8 MiB scratch
compiled into the library) must give the plan path's result, call after call.

For callers that cannot allocate device memory while serving (all free HBM
already handed to the KV pool, or a framework-owned allocator).  Collected after
every other parity test (only the tests that assert on measured times follow),
so that a failure here comes after them.
"""
import numpy as np
import pytest

from parity import attention_ok
from synth import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from paged_kv_cache_pool_gb300 import binding as gk  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_pool_gb300 import build
    from synth import device
    build.build()
    device.build()


def test_static_scratch_dense_matches_plan_path_two_calls():
    from gpu_workload import GpuWorkload
    w = workloads.config(2, B=12, Lp=1500, suffix_range=(100, 700), L=2)
    gw = GpuWorkload(w)
    try:
        b = gw.batch()
        plan = gw.eng.plan(b)
        for layer in (0, 1):                      # two calls in a row; the second reuses the scratch
            q = gw.q(layer)
            ref_o, ref_l = gw.outputs()
            b.set_device(d_q=q, d_out=ref_o, d_lse=ref_l)
            gk.gk_decode_dense(gw.eng.pool, None, layer, b, plan)
            st_o, st_l = gw.outputs()
            st_o.fill_(float("nan"))
            b.set_device(d_q=q, d_out=st_o, d_lse=st_l)
            gk.gk_decode_dense_static(gw.eng.pool, None, layer, b)
            torch.cuda.synchronize()
            assert gw.eng.device_error() == gk.GK_OK
            ok, err = attention_ok(st_o.cpu().numpy(), st_l.cpu().numpy(), ref_o.cpu().numpy(), ref_l.cpu().numpy())
            assert ok, err
            assert err["max_abs"] < 1e-5, err      # same kernels, same split: equal up to merge order
    finally:
        gw.close()


def test_static_scratch_refuses_oversized_batch():
    from paged_kv_cache_pool_gb300.engine import Engine
    # 64 query heads per request; requests of 2047 tokens.  How many partial states
    # the dense split needs depends on the SM count, so the batch grows until the
    # plan's own partition needs more than the 8 MiB the scratch holds.
    Hq, d, lim = 64, 128, 8 << 20
    eng = Engine(1, Hq, 8, d, 1, 1280 * 2048, 1)
    try:
        z = torch.zeros((1, 8, d), dtype=torch.bfloat16, device="cuda")
        eng.append_kv(0, torch.zeros(1, dtype=torch.int64, device="cuda"), z, z)   # first device work
        torch.cuda.synchronize()
        for B in (320, 640, 1280):
            table = torch.zeros((B, 2048), dtype=torch.int32, device="cuda")
            q = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device="cuda")
            out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
            b = gk.Batch(np.full(B, -1), np.zeros(B), np.full(B, 2047), table, 2048, q, out, None)
            plan = gk.gk_plan_build(eng.pool, b)
            try:
                _, segs = gk.gk_plan_segments(plan, dense=True)
            finally:
                gk.gk_plan_destroy(plan)
            need = int((segs[:, 3] >= 0).sum()) * Hq * (d + 1) * 4
            if need > lim:
                break
        assert need > lim, f"no batch tried needs more than {lim} bytes of partial states ({need})"
        with pytest.raises(gk.GkError) as e:
            gk.gk_decode_dense_static(eng.pool, None, 0, b)
        assert e.value.status == gk.GK_ERR_INVALID and "scratch" in str(e.value)
    finally:
        eng.close()


def test_static_scratch_refuses_a_capturing_stream():
    """The call copies its tables from host memory it frees on return, so a
    capturing stream gets GK_ERR_UNSUPPORTED and the capture itself stays valid."""
    from gpu_workload import GpuWorkload
    w = workloads.config(2, B=4, Lp=300, suffix_range=(20, 60), L=1)
    gw = GpuWorkload(w)
    try:
        b = gw.batch()
        q = gw.q(0)
        out, lse = gw.outputs()
        b.set_device(d_q=q, d_out=out, d_lse=lse)
        gk.gk_decode_dense_static(gw.eng.pool, None, 0, b)      # first call: address look-up
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            g.capture_begin()
            try:
                with pytest.raises(gk.GkError) as e:
                    gk.gk_decode_dense_static(gw.eng.pool, s, 0, b)
            finally:
                g.capture_end()
        assert e.value.status == gk.GK_ERR_UNSUPPORTED
    finally:
        gw.close()
