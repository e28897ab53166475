"""The N > 1 path of bench.py on CPU: two processes over gloo.

The workloads are independent problems (replicas, no data-path collective):
the only cross-rank steps are the barrier around the timed region, the MAX
of the per-rank times, and rank 0 printing the one JSON line.  These run here
with torch.distributed's gloo backend, world size 2, on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    dist, r, w, _ = bench.init_dist()
    assert (r, w) == (rank, world) and dist is not None and dist.get_backend() == "gloo"
    dist.barrier()
    out[rank] = bench.max_over_ranks(dist, times[rank])
    dist.destroy_process_group()


def test_max_over_ranks_two_processes():
    times = [3.25, 7.5]
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, times, out), nprocs=2, join=True)
        assert dict(out) == {0: 7.5, 1: 7.5}


def test_weak_scaling_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # two replicas, each 1e9 units in 0.5 s (the slowest rank's time): 4e9 units/s
    assert bench.weak_scaling_value(2, 1e9, 0.5) == pytest.approx(4e9)
    assert bench.weak_scaling_value(1, 1e9, 0.5) == pytest.approx(2e9)


def test_reference_arm_under_torchrun_two_ranks():
    """bench.py --impl reference launched by torchrun with N > 1 ranks:
    rank 0 times the oracle and prints one JSON line, rank 1 exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
