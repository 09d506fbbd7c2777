"""Measure the dispatcher's cost model on this GPU (GraniKV Section 3.6: the
routing rule stays, its numbers are re-fit per GPU; Appendix B.4b's sweep).

The sweep, the timing and the least-squares fit are the library's
(gk_calibrate); this module only sets up a pool of the wanted geometry with
random bf16 K/V and writes the JSON that gk_cost_model_load reads.

    python -m paged_kv_cache_pool_gb300.calibrate --out cost_model_gb300.json
"""
from __future__ import annotations

import argparse
import json
import os
import tempfile

from . import binding as gk
from .engine import Engine

# room for every case of gk_calibrate (one layer)
HOT_TOKENS = 16384 + 64
COLD_SLOTS = 262144 + 4096


def calibrate(Hq=32, Hkv=8, d=128, out=None, device="cuda"):
    """-> the fitted cost model (dict, with the measured points under "measured")."""
    import torch
    eng = Engine(1, Hq, Hkv, d, HOT_TOKENS, COLD_SLOTS, 1, seed=1, device=device)
    try:
        for t in (eng.hot_k, eng.hot_v, eng.cold_k, eng.cold_v):
            t.normal_()
        torch.cuda.synchronize()
        path = out
        if path is None:
            fd, path = tempfile.mkstemp(suffix=".json")
            os.close(fd)
        try:
            gk.gk_calibrate(eng.pool, None, path)
            with open(path) as f:
                return json.load(f)
        finally:
            if out is None:
                os.unlink(path)
    finally:
        eng.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None)
    a = ap.parse_args()
    from . import build
    build.build()
    print(json.dumps(calibrate(out=a.out), indent=1))


if __name__ == "__main__":
    main()
