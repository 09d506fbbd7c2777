"""GPU parity over every kernel geometry the ABI accepts (gk_pool_config:
head_dim 64 with Hq/Hkv in {1, 2, 4}; head_dim 128 with Hq/Hkv in {1, 2, 4, 5, 8}).

Each case is shaped so that every branch of the tensor-core prefix item runs:
  * Lp = 3 full 128-key tiles plus a ragged tail of 77 keys (masked scores);
  * M_eff = B * g of about 300 stacked rows, so the first 256-row block has both
    128-row Q tiles live and the second block only its first (two = false);
  * forced split plans with 2 key tiles per item (two key splits per KV head,
    two prefix partial states per request) and with 4 (one item walks every
    key tile, the ragged one last), and a sequential plan (prefix items over
    every SM, then the suffix gather);
  * queries as drawn and scaled by 8 (a peaked softmax, whose running maximum
    grows across tiles and takes the lazy-rescale branch).
Each plan runs with both prefix kernels: tensor-core items (256 rows: the first
row block has both Q tiles live, the second only its first, so its items run S
double-buffered, take two key splits each where there are two and leave the
second's entry empty; at g = 5 a request straddles the two blocks) and warp-MMA items
(128 rows: the third row block has 44 rows, so its last live warp is partly
empty and five warps sit out).  Suffixes run from 0 tokens up (an empty side
merges to the other).  Both backends are held to the fp64 oracle at
tests/parity.py's bounds, and the cascade's one-call entry point must give the
stage-by-stage launches' bits.
"""
import numpy as np
import pytest

from oracle import reference
from parity import assert_attention_close
from synth import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from paged_kv_cache_pool_gb300 import binding as gk  # noqa: E402

GEOMETRIES = [(64, 1), (64, 2), (64, 4), (128, 1), (128, 2), (128, 4), (128, 5), (128, 8)]
LP = 3 * 128 + 77
ROWS = 300
MODES = [("split-2-tiles", gk.GK_CASCADE_SPLIT, 2), ("split-4-tiles", gk.GK_CASCADE_SPLIT, 4),
         ("sequential", gk.GK_CASCADE_SEQUENTIAL, 0)]
KINDS = [("tensor", gk.GK_PREFIX_TENSOR, 256), ("warp", gk.GK_PREFIX_WARP, 128)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_pool_gb300 import build
    from synth import device
    build.build()
    device.build()


def _workload(d, g, peaked):
    Hkv = 4
    B = -(-ROWS // g)
    return workloads.config(2, B=B, Lp=LP, suffix_range=(0, 200), L=1, Hq=Hkv * g, Hkv=Hkv, d=d,
                            q_log2_scale=3 if peaked else 0)


def _decode(gw, b, pl, q, staged):
    out, lse = gw.outputs()
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    b.set_device(d_q=q, d_out=out, d_lse=lse)
    pool = gw.eng.pool
    if staged:
        gk.gk_cascade_prefix(pool, None, 0, b, pl)
        gk.gk_cascade_suffix(pool, None, 0, b, pl)
        gk.gk_cascade_merge(pool, None, 0, b, pl)
    else:
        gk.gk_decode_cascade(pool, None, 0, b, pl)
    torch.cuda.synchronize()
    assert gw.eng.device_error() == gk.GK_OK
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("peaked", [False, True], ids=["normal", "peaked"])
@pytest.mark.parametrize("d,g", GEOMETRIES, ids=[f"d{d}-g{g}" for d, g in GEOMETRIES])
def test_every_geometry_both_backends(d, g, peaked):
    from gpu_workload import GpuWorkload
    w = _workload(d, g, peaked)
    assert w.B * g > 256 and LP % 128 != 0 and LP > 3 * 128
    gw = GpuWorkload(w)
    try:
        O_ref, L_ref = reference.expected(w, 0)
        what = f"d={d} g={g}{' peaked' if peaked else ''}"
        seen_splits = set()
        for kname, kernel, rows in KINDS:
            gk.gk_pool_set_prefix_kernel(gw.eng.pool, kernel)
            for name, mode, tiles in MODES:
                gk.gk_pool_set_cascade_mode(gw.eng.pool, mode, tiles)
                b = gw.batch()
                pl = gw.eng.plan(b)
                info = gk.gk_plan_info(pl)
                assert info["prefix_kernel"] == kernel and info["prefix_rows_per_item"] == rows
                if name.startswith("split-"):
                    # the forced plans: row blocks x KV heads x key splits of `tiles` tiles (in a
                    # split plan the last tensor-core block, 44-48 rows: one Q tile, takes one
                    # split per item like the others; sequential plans pair its splits)
                    assert info["cascade_split"] == 1 and info["prefix_tiles_per_item"] == tiles
                    full = w.B * g // rows
                    last = 0 if w.B * g % rows == 0 else 4 // tiles
                    assert info["prefix_ctas"] == (full * (4 // tiles) + last) * w.Hkv
                seen_splits.add(info["cascade_split"])
                q = gw.q(0)
                O1, L1 = _decode(gw, b, pl, q, staged=False)
                O0, L0 = _decode(gw, b, pl, q, staged=True)
                tag = f"{what} {kname} {name}"
                assert np.array_equal(O1, O0) and np.array_equal(L1, L0), f"{tag}: cascade != stages"
                assert_attention_close(O1, L1, O_ref, L_ref, f"{tag} cascade")
        assert seen_splits == {0, 1}
        gk.gk_pool_set_cascade_mode(gw.eng.pool, gk.GK_CASCADE_AUTO, 0)
        gk.gk_pool_set_prefix_kernel(gw.eng.pool, gk.GK_PREFIX_AUTO)
        O, L = gw.run(0, gk.GK_BACKEND_DENSE)
        assert_attention_close(O, L, O_ref, L_ref, f"{what} dense")
    finally:
        gw.close()


@pytest.mark.parametrize("lp,B,g,srange", [(1000, 2, 4, (10, 300)), (130, 8, 4, (0, 5)), (2048 + 5, 8, 4, (16, 512)),
                                           (512, 32, 4, (16, 512)), (777, 3, 1, (0, 50)), (300, 5, 8, (1, 40))])
def test_small_m_eff_both_prefix_kernels(lp, B, g, srange):
    """The regime the warp-MMA items are for (M_eff = B * g of 2 to 128 stacked rows), as
    the planner arranges it and forced split, with either prefix kernel, against the oracle."""
    from gpu_workload import GpuWorkload
    Hkv = 8 if g != 8 else 4
    w = workloads.config(2, B=B, Lp=lp, suffix_range=srange, L=1, Hq=Hkv * g, Hkv=Hkv)
    gw = GpuWorkload(w)
    try:
        O_ref, L_ref = reference.expected(w, 0)
        for kname, kernel, _ in KINDS:
            gk.gk_pool_set_prefix_kernel(gw.eng.pool, kernel)
            for name, mode, tiles in (("auto", gk.GK_CASCADE_AUTO, 0), ("split-1-tile", gk.GK_CASCADE_SPLIT, 1),
                                      ("sequential", gk.GK_CASCADE_SEQUENTIAL, 0)):
                gk.gk_pool_set_cascade_mode(gw.eng.pool, mode, tiles)
                b = gw.batch()
                pl = gw.eng.plan(b)
                assert gk.gk_plan_info(pl)["prefix_kernel"] == kernel
                O, L = _decode(gw, b, pl, gw.q(0), staged=False)
                assert_attention_close(O, L, O_ref, L_ref, f"lp={lp} B={B} g={g} {kname} {name}")
    finally:
        gw.close()
