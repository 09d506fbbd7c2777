"""Fused append: the decode entry points take the step's new tokens (gk_batch
d_new_k / d_new_v) and write them into the pool themselves, instead of a
separate gk_append_kv scatter.

Two pools with the same seeds run the same steps of a forked workload (P 16,
copy-on-write): one appends then decodes, the other copies its COW pairs
(gk_append_kv with n = 0) and decodes with the new tokens fused.  Outputs of
both backends and the whole COLD pool must agree bit for bit, step after step;
the fused pool is also decoded once more without the fused tokens, reading
what it wrote.
"""
import numpy as np
import pytest

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


def _used_slots(gw):
    """Every pool slot a sequence's block table reaches (the rest of the pool is never written)."""
    P = gw.P
    slots = []
    for sid in gw.seqs:
        table, length = gk.gk_seq_table(gw.eng.pool, sid)
        for t in range(length):
            slots.append(int(table[t // P]) * P + t % P)
    return torch.tensor(sorted(set(slots)), dtype=torch.int64, device=gw.eng.cold_k.device)


def _pools_equal(a, b):
    sa, sb = _used_slots(a), _used_slots(b)
    assert torch.equal(sa, sb)
    return (torch.equal(a.eng.cold_k[:, sa], b.eng.cold_k[:, sb])
            and torch.equal(a.eng.cold_v[:, sa], b.eng.cold_v[:, sb]))


def _decode(gw, layer, backend, step, new_kv=None):
    b = gw.batch()
    q = gw.q(layer, step)
    out, lse = gw.outputs()
    k, v = new_kv if new_kv is not None else (None, None)
    b.set_device(d_q=q, d_out=out, d_lse=lse, d_new_k=k, d_new_v=v)
    pl = gw.eng.plan(b)
    gw.eng.decode(layer, b, pl, backend)
    torch.cuda.synchronize()
    assert gw.eng.device_error() == gk.GK_OK
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("mode", [gk.GK_CASCADE_AUTO, gk.GK_CASCADE_SEQUENTIAL, gk.GK_CASCADE_SPLIT])
def test_fused_append_equals_append_then_decode(mode):
    from gpu_workload import GpuWorkload
    w = workloads.config(5, n_parent=6, children=4, Lp=1000, suffix_range=(20, 70), steps=5, L=2)
    ref, fused = GpuWorkload(w), GpuWorkload(w)
    try:
        for gw in (ref, fused):
            gk.gk_pool_set_cascade_mode(gw.eng.pool, mode)
        n_cow = 0
        for step in range(w.steps):
            slots_ref, cow_ref = ref.append_step(step)
            slots, cow = fused.eng.append_slots(np.asarray(fused.seqs, dtype=np.int32))
            assert slots.tolist() == slots_ref.tolist() and cow.tolist() == cow_ref.tolist()
            fused.appended += 1
            n_cow += len(cow)
            d_cow = fused.eng.to_device(cow.reshape(-1)) if len(cow) else None
            for layer in range(w.L):
                if len(cow):
                    gk.gk_append_kv(fused.eng.pool, None, layer, None, None, None, d_cow, n=0, n_cow=len(cow))
                new_kv = fused.new_kv(layer, step)
                for backend in (gk.GK_BACKEND_CASCADE, gk.GK_BACKEND_DENSE):
                    O0, L0 = _decode(ref, layer, backend, step)
                    O1, L1 = _decode(fused, layer, backend, step, new_kv)
                    assert np.array_equal(O0, O1) and np.array_equal(L0, L1), f"step {step} layer {layer} backend {backend}"
            assert _pools_equal(ref, fused), f"pools differ after step {step}"
        assert n_cow > 0   # the workload exercised copy-on-write
        # the fused pool decodes from its own writes afterwards
        O0, L0 = _decode(ref, 1, gk.GK_BACKEND_CASCADE, w.steps - 1)
        O1, L1 = _decode(fused, 1, gk.GK_BACKEND_CASCADE, w.steps - 1)
        assert np.array_equal(O0, O1) and np.array_equal(L0, L1)
    finally:
        ref.close()
        fused.close()


def test_fused_append_needs_both_pointers():
    from gpu_workload import GpuWorkload
    gw = GpuWorkload(workloads.config(1))
    try:
        b = gw.batch()
        q = gw.q(0)
        out, lse = gw.outputs()
        k, _ = gw.new_kv(0, 0)
        b.set_device(d_q=q, d_out=out, d_lse=lse, d_new_k=k)
        pl = gw.eng.plan(b)
        with pytest.raises(gk.GkError):
            gw.eng.decode(0, b, pl, gk.GK_BACKEND_CASCADE)
    finally:
        gw.close()
