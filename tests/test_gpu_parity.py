"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases are compared in full (several tiles, ragged tails, multiple splits,
several prefix groups, requests without a HOT prefix); the five workloads run at
full size on sampled layers.  Block tables, slot mappings and copy-on-write
pairs are compared bit for bit; attention within tests/parity.py's bounds.
"""
import numpy as np
import pytest

from oracle import reference
from oracle.block_manager import BlockPool, Seq
from parity import assert_attention_close, attention_ok
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


def _wl(**kw):
    from gpu_workload import GpuWorkload
    return GpuWorkload(**kw)


def _check_both(gw, layer, step=0, appended=0, what=""):
    w = gw.w
    O_ref, L_ref = reference.expected(w, layer, appended=appended, q_step=step)
    res = {}
    b = gw.batch()
    for name, be in (("cascade", gk.GK_BACKEND_CASCADE), ("dense", gk.GK_BACKEND_DENSE)):
        O, L = gw.run(layer, be, step=step, batch=b)
        res[name] = assert_attention_close(O, L, O_ref, L_ref, f"{what} {name} layer {layer}")
    return res, (O_ref, L_ref)


def test_config1_full():
    w = workloads.config(1)
    gw = _wl(w=w)
    try:
        res, _ = _check_both(gw, 0, what="config 1")
        # tables through the ABI equal the oracle block manager's (same seed, same order)
        bp = BlockPool(w.cold_slots() // w.page_size, w.page_size, w.seed)
        for r, req in enumerate(w.requests):
            s = Seq()
            for _ in range(req.suffix_len):
                bp.append(s)
            t, ln = gk.gk_seq_table(gw.eng.pool, gw.seqs[r])
            assert t.tolist() == s.table and ln == s.len
    finally:
        gw.close()


def test_config1_peaked_queries():
    w = workloads.config(1, q_log2_scale=3)
    gw = _wl(w=w)
    try:
        _check_both(gw, 0, what="config 1 peaked")
    finally:
        gw.close()


@pytest.mark.parametrize("lp,B,srange,g", [(1000, 8, (50, 300), 4), (130, 3, (1, 5), 4), (4096 + 77, 40, (200, 900), 4),
                                           (777, 20, (0, 40), 5), (300, 33, (10, 200), 8),
                                           # tiny suffixes: a gather CTA's quota spans dozens of requests,
                                           # more segments than the shared-memory segment cache holds
                                           (130, 300, (0, 3), 4)])
def test_small_shared_prefix(lp, B, srange, g):
    Hkv = 8 if g != 8 else 4
    w = workloads.config(2, B=B, Lp=lp, suffix_range=srange, L=2, Hq=Hkv * g, Hkv=Hkv)
    gw = _wl(w=w)
    try:
        for layer in (0, 1):
            _check_both(gw, layer, what=f"lp={lp} B={B} g={g}")
    finally:
        gw.close()


def test_per_request_partition_multi_prefix():
    """Tangram's per-request splits (GK_PARTITION_PER_REQUEST) for the flat backend and a
    sequential cascade: more CTAs than SMs' worth of segments, same attention."""
    w = workloads.config(4, n_prefix=3, lp_range=(100, 2000), bg_range=(2, 9), suffix_range=(0, 3000), L=1)
    gw = _wl(w=w)
    try:
        gk.gk_pool_set_gather_partition(gw.eng.pool, gk.GK_PARTITION_PER_REQUEST)
        gk.gk_pool_set_cascade_mode(gw.eng.pool, gk.GK_CASCADE_SEQUENTIAL)
        _check_both(gw, 0, what="per-request partition")
    finally:
        gw.close()


def test_multi_prefix_groups_and_cold_prefix():
    """Several HOT groups interleaved in the batch, plus requests whose prefix is in COLD."""
    w = workloads.config(4, n_prefix=3, lp_range=(100, 2000), bg_range=(2, 9), suffix_range=(0, 300), L=2)
    # two requests without a HOT prefix (their whole context in COLD, B.10 fallback)
    w.requests[1].prefix = -1
    w.requests[4].prefix = -1
    gw = _wl(w=w)
    try:
        for layer in (0, 1):
            _check_both(gw, layer, what="multi-prefix")
    finally:
        gw.close()


def test_forks_cow_steps_small_bit_exact_pool():
    """Fork + copy-on-write + appends: pool contents bit-exact against the oracle pool model,
    outputs at every step within bounds, P = 16 and P = 1 agree."""
    from oracle.pool_model import build_pool
    w = workloads.config(5, n_parent=3, children=4, Lp=200, suffix_range=(20, 60), steps=6, L=2)
    gw = _wl(w=w)
    try:
        pm, bases, seqs, bp = build_pool(w, steps=0)
        for t in range(w.steps):
            slots, cow = gw.append_step(t)
            res = [bp.append(s) for s in seqs]
            assert slots.tolist() == [x[0] for x in res]
            assert cow.tolist() == [list(x[1]) for x in res if x[1] is not None]
            for layer in range(w.L):
                from oracle.reference import new_kv_bits
                k, v = new_kv_bits(w, layer, t)
                pm.append(layer, slots, k, v, [tuple(c) for c in cow])
            if t in (0, w.steps - 1):
                for layer in range(w.L):
                    _check_both(gw, layer, step=t, appended=t + 1, what=f"fork step {t}")
        torch.cuda.synchronize()
        ck = gw.eng.cold_k.view(torch.int16).cpu().numpy().view(np.uint16)
        cv = gw.eng.cold_v.view(torch.int16).cpu().numpy().view(np.uint16)
        used = sorted({s for seq in seqs for b in seq.table for s in range(b * w.page_size, (b + 1) * w.page_size)})
        # every slot a live sequence can read holds exactly the oracle's bits
        for seq in seqs:
            for tkn in range(seq.len):
                slot = seq.table[tkn // w.page_size] * w.page_size + tkn % w.page_size
                np.testing.assert_array_equal(ck[:, slot], pm.cold_k[:, slot])
                np.testing.assert_array_equal(cv[:, slot], pm.cold_v[:, slot])
        assert used
        hk = gw.eng.hot_k.view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(hk[:pm.hot_k.size], pm.hot_k)
    finally:
        gw.close()


def test_page_size_invariance_on_gpu():
    """The same forked steps at page sizes 16, 1, 4 and two that are not powers of two
    (3, 6: the gather's slot arithmetic then divides instead of shifting), both backends."""
    outs = {gk.GK_BACKEND_CASCADE: [], gk.GK_BACKEND_DENSE: []}
    for P, seed in ((16, 5), (1, 5), (4, 11), (3, 7), (6, 5)):
        w = workloads.config(5, n_parent=2, children=3, Lp=300, suffix_range=(30, 90), steps=3, L=1)
        gw = _wl(w=w, page_size=P, cold_seed=seed)
        try:
            for t in range(w.steps):
                gw.append_step(t)
            for be in outs:
                outs[be].append(gw.run(0, be, step=w.steps - 1))
        finally:
            gw.close()
    for be, runs in outs.items():
        for O, L in runs[1:]:
            ok, e = attention_ok(O, L, *runs[0])
            assert ok and e["max_abs"] < 1e-4, (be, e)


def test_mutated_oracle_is_rejected():
    """A mistake planted in the oracle (suffix dropped) must fail against the GPU output."""
    w = workloads.config(2, B=4, Lp=2000, suffix_range=(400, 600), L=1)
    gw = _wl(w=w)
    try:
        O, L = gw.run(0, gk.GK_BACKEND_CASCADE)
        import copy
        w2 = copy.deepcopy(w)
        for r in w2.requests:
            r.suffix_len = 0
        O_bad, L_bad = reference.expected(w2, 0)
        assert not attention_ok(O, L, O_bad, L_bad)[0]
    finally:
        gw.close()


def test_dispatch_choice_is_a_backend_and_both_agree():
    w = workloads.config(3, B=16, Lp=512, suffix_range=(64, 256), L=1)
    gw = _wl(w=w)
    try:
        b = gw.batch()
        plan = gw.eng.plan(b)
        choice, td, tc = gw.eng.dispatch(plan)
        assert choice in (gk.GK_BACKEND_DENSE, gk.GK_BACKEND_CASCADE) and td > 0 and tc > 0
        O1, L1 = gw.run(0, gk.GK_BACKEND_DENSE, batch=b, plan=plan)
        O2, L2 = gw.run(0, gk.GK_BACKEND_CASCADE, batch=b, plan=plan)
        ok, e = attention_ok(O1, L1, O2, L2)
        assert ok, e
    finally:
        gw.close()


def test_device_bounds_error_is_reported_not_faulted():
    """A block id past the pool in the table is skipped by the kernel and reported."""
    w = workloads.config(2, B=2, Lp=256, suffix_range=(20, 30), L=1)
    gw = _wl(w=w)
    try:
        b = gw.batch()
        bad = gw._d_table.clone()
        bad[0, 0] = gw.eng.cold_slots // gw.P + 5       # out of range, in-bounds of the table itself
        b.set_device(d_block_table=bad)
        q = gw.q(0)
        out, lse = gw.outputs()
        b.set_device(d_q=q, d_out=out, d_lse=lse)
        plan = gw.eng.plan(b)
        gw.eng.decode(0, b, plan, gk.GK_BACKEND_CASCADE)
        torch.cuda.synchronize()
        assert gw.eng.device_error() == gk.GK_ERR_DEVICE_BOUNDS
        assert gw.eng.device_error() == gk.GK_OK          # read clears it
    finally:
        gw.close()
