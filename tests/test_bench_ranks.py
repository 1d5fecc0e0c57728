"""The N > 1 path of bench.py on the CPU: two gloo ranks (the decode shards with no exchange, so N GPUs run
N replicas; the only cross-rank steps are the barrier and the max of the timings)."""

import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) ms per step over 10 steps and decoded in 5 - r ms
        total, dec = bench.max_over_ranks([10.0 * (rank + 1), 5.0 - rank], world, "cpu")
        dist.barrier()
        out[rank] = (total, dec, bench.replica_gbps(world, 1e6, total / 10))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    for r in range(world):
        total, dec, gbps = res[r]
        assert total == 20.0 and dec == 5.0  # both ranks see the maximum
        assert gbps == pytest.approx(2 * 1e6 / 2e-3 / 1e9)  # 2 replicas x 1 MB per 2 ms = 1 GB/s


def test_one_rank_keeps_its_values():
    assert bench.max_over_ranks([3.5, 1.25], 1, "cpu") == [3.5, 1.25]
    assert bench.replica_gbps(1, 5e8, 100.0) == pytest.approx(5.0)


def test_reference_arm_rank_other_than_zero_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
