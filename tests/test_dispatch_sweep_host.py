"""The backend-crossover tools (paged_kv_cache_pool_gb300.dispatch_sweep) on the host.

The routing trace follows the dispatcher: with a cost model in which the flat
backend is nearly free every step routes to it, with one in which it is very
slow none does, the fractions are deterministic for a seed; and the crossover
summary lists, per prefix length, the M_eff at which each choice was measured fastest.
"""
import json

import pytest


@pytest.fixture(scope="module")
def sweep():
    from paged_kv_cache_pool_gb300 import build
    build.build()
    from paged_kv_cache_pool_gb300 import dispatch_sweep
    return dispatch_sweep


BASE = dict(c_flat_us=14.0, bw_flat_gbs=9000.0, c_cascade_us=10.0, bw_prefix_gbs=6000.0, bw_suffix_gbs=6000.0,
            c_merge_us=0.001, prefix_tile_us=1.5, prefix_item_us=9.7, gather_sm_gbs=38.0, c_gather_us=7.0,
            prefix_tile_split_us=1.9)


def _model(tmp_path, **kw):
    p = tmp_path / "cm.json"
    p.write_text(json.dumps(dict(BASE, **kw)))
    return str(p)


def test_trace_follows_the_cost_model(sweep, tmp_path):
    grid = dict(lps=(512, 4096), bs=(8, 64), steps=20)
    free_flat = sweep.trace(cost_model=_model(tmp_path, c_flat_us=0.0, bw_flat_gbs=1e9), **grid)
    assert set(free_flat.values()) == {1.0}
    slow_flat = sweep.trace(cost_model=_model(tmp_path, c_flat_us=1e6), **grid)
    assert set(slow_flat.values()) == {0.0}
    a = sweep.trace(cost_model=_model(tmp_path), **grid)
    b = sweep.trace(cost_model=_model(tmp_path), **grid)
    assert a == b and all(0.0 <= v <= 1.0 for v in a.values())
    # the flat backend's bytes grow with Lp * B, the cascade reads the prefix once:
    # its share of the routing can only fall as the prefix grows
    for B in grid["bs"]:
        assert a[(4096, B)] <= a[(512, B)]


def test_crossover_summary(sweep):
    rows = [dict(Lp=512, M_eff=32, fastest="warp"), dict(Lp=512, M_eff=128, fastest="dense"),
            dict(Lp=512, M_eff=512, fastest="dense"), dict(Lp=2048, M_eff=32, fastest="tensor")]
    assert sweep.crossover(rows) == {512: {"dense": [128, 512], "tensor": [], "warp": [32]},
                                     2048: {"dense": [], "tensor": [32], "warp": []}}
