"""The N > 1 path of bench.py on CPU: N independent replicas (the path shards without
any exchange, so there is no collective on the data path), a barrier and the max of
the ranks' times, rank 0 printing the one JSON line.  gloo, world size 2."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank])
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    import torch.multiprocessing as mp
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    values = [3.25, 7.5]
    mp.start_processes(_worker, args=(2, _free_port(), values, out), nprocs=2, start_method="spawn")
    assert dict(out) == {0: 7.5, 1: 7.5}


def test_replica_throughput_is_the_job_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas of 64 requests x 32 layers x 10 steps in 100 ms (the slower rank's time)
    assert bench.replica_throughput(2, 64 * 32 * 10, 100.0) == 2 * 64 * 32 * 10 / 0.1
    assert bench.max_over_ranks(4.0) == 4.0   # alone: no process group


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--config", "1", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["n_gpus"] == 1
