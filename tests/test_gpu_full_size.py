"""Full-size parity: the five workloads at their real shapes and pool sizes,
through the same plan/launch configuration bench.py times.

The pool is allocated for every layer; the layers checked (first and last) are
filled and decoded, and the oracle computes requests one by one (all query
heads): every request of both layers for workloads 2, 3 and 4; for workload 5,
every request of both layers after the first and the last of its 32 steps, and
four requests after every step.
Block tables are compared bit for bit with the oracle block manager for every
sequence.
"""
import numpy as np
import pytest

from oracle import reference
from oracle.block_manager import BlockPool, Seq
from parity import assert_attention_close
from synth import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

from paged_kv_cache_pool_gb300 import binding as gk  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_pool_gb300 import build
    from synth import device
    build.build()
    device.build()


def _oracle_tables(w, gw):
    """Replay the workload's COLD setup in the oracle block manager; compare every table."""
    P = gw.P
    bp = BlockPool(gw.eng.cold_slots // P, P, w.seed)
    if w.fork_children:
        seqs = []
        for n in w.parents:
            s = Seq()
            for _ in range(n):
                bp.append(s)
            seqs.extend(bp.fork(s) for _ in range(w.fork_children))
            bp.release(s)
    else:
        seqs = []
        for r in w.requests:
            s = Seq()
            for _ in range(r.suffix_len):
                bp.append(s)
            seqs.append(s)
    return bp, seqs


def _compare_tables(gw, seqs):
    for sid, s in zip(gw.seqs, seqs):
        t, ln = gk.gk_seq_table(gw.eng.pool, sid)
        assert ln == s.len and t.tolist() == s.table


def _check_layer(gw, layer, reqs, step=0, appended=0, what=""):
    w = gw.w
    O_ref, L_ref = reference.expected(w, layer, requests=reqs, appended=appended, q_step=step)
    b = gw.batch()
    for name, be in (("cascade", gk.GK_BACKEND_CASCADE), ("dense", gk.GK_BACKEND_DENSE)):
        O, L = gw.run(layer, be, step=step, batch=b)
        assert_attention_close(O[reqs], L[reqs], O_ref, L_ref, f"{what} {name} layer {layer} step {step}")


@pytest.mark.parametrize("n", [2, 3, 4])
def test_full_size_single_step(n):
    from gpu_workload import GpuWorkload
    w = workloads.config(n)
    gw = GpuWorkload(w, layers=[0, w.L - 1])
    try:
        _, seqs = _oracle_tables(w, gw)
        _compare_tables(gw, seqs)
        for layer in (0, w.L - 1):
            _check_layer(gw, layer, list(range(w.B)), what=w.name)
        info = gk.gk_plan_info(gw.eng.plan(gw.batch()))
        assert info["num_groups"] == len(w.prefix_lens)
    finally:
        gw.close()


def test_full_size_peaked_queries():
    """Q x 8 concentrates each softmax on a few keys, so single-token gather errors show."""
    from gpu_workload import GpuWorkload
    w = workloads.config(2, q_log2_scale=3)
    gw = GpuWorkload(w, layers=[0])
    try:
        _check_layer(gw, 0, list(range(w.B)), what="peaked " + w.name)
    finally:
        gw.close()


def test_full_size_fork_cow_32_steps():
    from gpu_workload import GpuWorkload
    w = workloads.config(5)
    layers = [0, w.L - 1]
    gw = GpuWorkload(w, layers=layers)
    try:
        bp, seqs = _oracle_tables(w, gw)
        _compare_tables(gw, seqs)
        few = [0, 1, 2, 3]
        n_cow = 0
        for t in range(w.steps):
            slots, cow = gw.append_step(t)
            res = [bp.append(s) for s in seqs]
            assert slots.tolist() == [x[0] for x in res]
            assert cow.tolist() == [list(x[1]) for x in res if x[1] is not None]
            n_cow += len(cow)
            if t in (0, w.steps - 1):
                for layer in layers:
                    _check_layer(gw, layer, list(range(w.B)), step=t, appended=t + 1, what=w.name)
            else:
                _check_layer(gw, layers[0], few, step=t, appended=t + 1, what=w.name)
        # every parent with a partial last block was shared 4 ways: 3 copies each
        assert n_cow == 3 * sum(1 for n in w.parents if n % w.page_size)
        _compare_tables(gw, seqs)
    finally:
        gw.close()
