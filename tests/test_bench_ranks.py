"""The multi-rank path of bench.py on CPU: two gloo ranks, max-over-ranks timing,
whole-job aggregation (weak scaling), and the reference arm printing on rank 0 only."""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local = [1.0 + rank, 10.0 - rank, 3.0]          # per-rank step times (ms)
        got = bench.max_over_ranks(local, dist, "cpu")
        rate = bench.whole_job_rate(5e9, world, got[0], 1e12)
        q.put((rank, got, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    world = 2
    port = 29500 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    mp.start_processes(_rank_main, args=(world, port, q), nprocs=world, start_method="spawn", join=True)
    res = sorted(q.get() for _ in range(world))
    for rank, got, rate in res:
        assert got == [2.0, 10.0, 3.0]                 # elementwise max over ranks
        assert rate == pytest.approx(2 * 5e9 / 2e-3 / 1e12)


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.whole_job_rate(1e9, 1, 1.0, 1e9) == pytest.approx(1000.0)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
