"""The multi-rank host logic of the benchmark on CPU: world_size 2 over gloo.

Each rank is an independent replica (no collective on the data path); the
only cross-rank traffic is the barrier and the max over ranks of the timings.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank 1 is the slow one on the first value, rank 0 on the second
    mine = [10.0 + 5.0 * rank, 7.0 - 3.0 * rank]
    res = bench.max_over_ranks(mine, "cpu", world)
    dist.barrier()
    out[rank] = res
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == [15.0, 7.0]


def test_whole_job_rate():
    import bench
    assert bench.whole_job_rate(25_000_000, 2, 500.0) == pytest.approx(1e8)
    assert bench.whole_job_rate(10, 1, 1000.0) == pytest.approx(10.0)


def test_reference_arm_runs_on_host():
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--workload", "tiny_adam"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
