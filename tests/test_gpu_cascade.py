"""gk_decode_cascade under both arrangements against the staged launches of the
same plan (gk_cascade_prefix, gk_cascade_suffix, gk_cascade_merge) and the
fp64 oracle.

A sequential plan runs the prefix items over every SM and then the suffix
gather; a split plan runs long prefix items on some SMs beside the suffix
gather on the rest, in one launch.  For one plan both entry points compute
the same partial states and merge them in the same order, so their outputs
agree bit for bit; the two arrangements split the keys differently, so each is
held to the oracle on its own.
"""
import numpy as np
import pytest

from oracle import reference
from parity import assert_attention_close
from synth import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from paged_kv_cache_pool_gb300 import binding as gk  # noqa: E402

MODES = [("sequential", gk.GK_CASCADE_SEQUENTIAL, 0), ("split", gk.GK_CASCADE_SPLIT, 0),
         ("split-short-items", gk.GK_CASCADE_SPLIT, 3)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_pool_gb300 import build
    from synth import device
    build.build()
    device.build()


def _decode(gw, layer, b, pl, q, staged):
    out, lse = gw.outputs()
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    b.set_device(d_q=q, d_out=out, d_lse=lse)
    pool = gw.eng.pool
    if staged:
        gk.gk_cascade_prefix(pool, None, layer, b, pl)
        gk.gk_cascade_suffix(pool, None, layer, b, pl)
        gk.gk_cascade_merge(pool, None, layer, b, pl)
    else:
        gk.gk_decode_cascade(pool, None, layer, b, pl)
    torch.cuda.synchronize()
    assert gw.eng.device_error() == gk.GK_OK
    return out.cpu().numpy(), lse.cpu().numpy()


def _check(gw, layers, what, requests=None, modes=MODES):
    w = gw.w
    reqs = list(range(w.B)) if requests is None else requests
    refs = {layer: reference.expected(w, layer, requests=reqs) for layer in set(layers)}
    seen = set()
    for name, mode, tiles in modes:
        gk.gk_pool_set_cascade_mode(gw.eng.pool, mode, tiles)
        b = gw.batch()
        pl = gw.eng.plan(b)
        seen.add(gk.gk_plan_info(pl)["cascade_split"])
        for layer in layers:
            q = gw.q(layer)
            O1, L1 = _decode(gw, layer, b, pl, q, staged=False)
            O0, L0 = _decode(gw, layer, b, pl, q, staged=True)
            assert np.array_equal(O1, O0) and np.array_equal(L1, L0), f"{what} {name}: cascade != stages (layer {layer})"
            O_ref, L_ref = refs[layer]
            assert_attention_close(O1[reqs], L1[reqs], O_ref, L_ref, f"{what} {name} layer {layer}")
    gk.gk_pool_set_cascade_mode(gw.eng.pool, gk.GK_CASCADE_AUTO)
    return seen


def _wl(**kw):
    from gpu_workload import GpuWorkload
    return GpuWorkload(**kw)


def test_cascade_tiny_config():
    gw = _wl(w=workloads.config(1))
    try:
        assert _check(gw, [0], "config 1") == {0, 1}
    finally:
        gw.close()


@pytest.mark.parametrize("lp,B,srange,g", [(1000, 8, (50, 300), 4), (777, 20, (0, 40), 5), (300, 33, (10, 200), 8),
                                           (4096 + 77, 70, (1, 600), 1)])
def test_cascade_shared_prefix(lp, B, srange, g):
    Hkv = 8 if g != 8 else 4
    w = workloads.config(2, B=B, Lp=lp, suffix_range=srange, L=2, Hq=Hkv * g, Hkv=Hkv)
    gw = _wl(w=w)
    try:
        assert _check(gw, [0, 1, 0], f"lp={lp} B={B} g={g}") == {0, 1}
    finally:
        gw.close()


def test_cascade_multi_prefix_cold_prefix_and_empty_context():
    """Several HOT groups, requests without a HOT prefix, and one with no context at all."""
    w = workloads.config(4, n_prefix=3, lp_range=(100, 2000), bg_range=(2, 9), suffix_range=(0, 300), L=2)
    w.requests[1].prefix = -1
    w.requests[4].prefix = -1
    w.requests[2].prefix = -1
    w.requests[2].suffix_len = 0
    gw = _wl(w=w)
    try:
        _check(gw, [0, 1], "multi-prefix")
        b = gw.batch()
        O, L = _decode(gw, 1, b, gw.eng.plan(b), gw.q(1), staged=False)
        assert np.all(O[2] == 0) and np.all(np.isneginf(L[2]))
    finally:
        gw.close()


@pytest.mark.slow
def test_cascade_full_size_llama8b_lp16384_b64():
    """The benchmarked workload at full size under both arrangements."""
    w = workloads.config(2)
    gw = _wl(w=w, layers=[0])
    try:
        assert _check(gw, [0], w.name, requests=[0, 1, w.B // 2, w.B - 1], modes=MODES[:2]) == {0, 1}
    finally:
        gw.close()


@pytest.mark.parametrize("lp,B,srange,g", [(4096 + 77, 70, (1, 600), 4), (1000, 8, (50, 300), 5)])
def test_cascade_sm_speed_slots(lp, B, srange, g):
    """Split plans planned per SM (gk_pool_set_sm_speeds, or the speeds gk_sm_speeds_measure
    takes from the plan's own suffix gather): the CTA on each SM claims the slot planned for
    it, every slot runs exactly once wherever the CTAs land, so the split launch still gives
    the staged launches' bits, and the outputs hold to the fp64 oracle."""
    Hkv = 8 if g != 8 else 4
    w = workloads.config(2, B=B, Lp=lp, suffix_range=srange, L=2, Hq=Hkv * g, Hkv=Hkv)
    gw = _wl(w=w)
    try:
        pool = gw.eng.pool
        n_sm = torch.cuda.get_device_properties(0).multi_processor_count
        rng = np.random.default_rng([lp, B])
        gk.gk_pool_set_sm_speeds(pool, rng.uniform(0.7, 1.3, n_sm))
        modes = [("split", gk.GK_CASCADE_SPLIT, 0), ("split-short-items", gk.GK_CASCADE_SPLIT, 3)]
        b = gw.batch()
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SPLIT, 0)
        pl = gw.eng.plan(b)
        assert gk.gk_plan_info(pl)["sm_slots"] == 1
        # three launches in a row: each launch's claims carry a tag of their own
        assert 1 in _check(gw, [0, 1, 0], f"sm slots lp={lp} B={B} g={g}", modes=modes)
        # speeds measured from the plan's suffix gather: one per SM, mean 1, all plausible
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SEQUENTIAL, 0)
        b = gw.batch()
        pl = gw.eng.plan(b)
        q = gw.q(0)
        out, lse = gw.outputs()
        b.set_device(d_q=q, d_out=out, d_lse=lse)
        sp = gk.gk_sm_speeds_measure(pool, None, 0, b, pl, reps=3)
        assert len(sp) == n_sm and abs(float(sp.mean()) - 1.0) < 1e-4 and sp.min() > 0.3 and sp.max() < 3.0
        assert gw.eng.device_error() == gk.GK_OK
        assert _check(gw, [1], f"measured sm slots lp={lp} B={B} g={g}", modes=modes[:1]) == {1}
        # measured again from a split plan that already runs per SM (its launches claim slots)
        gk.gk_pool_set_cascade_mode(pool, gk.GK_CASCADE_SPLIT, 0)
        b = gw.batch()
        pl = gw.eng.plan(b)
        assert gk.gk_plan_info(pl)["sm_slots"] == 1
        b.set_device(d_q=q, d_out=out, d_lse=lse)
        sp2 = gk.gk_sm_speeds_measure(pool, None, 0, b, pl, reps=3)
        assert len(sp2) == n_sm and abs(float(sp2.mean()) - 1.0) < 1e-4 and sp2.min() > 0.3 and sp2.max() < 3.0
        assert gw.eng.device_error() == gk.GK_OK
        assert _check(gw, [0], f"re-measured sm slots lp={lp} B={B} g={g}", modes=modes[:1]) == {1}
        gk.gk_pool_set_sm_speeds(pool, None)
    finally:
        gw.close()
