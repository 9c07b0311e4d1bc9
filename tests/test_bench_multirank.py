"""bench.py's multi-rank host logic on CPU: two gloo ranks, each with its own
(fake) timing; the job is as slow as its slowest rank and the whole-job
throughput counts every rank's work."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms_local = 100.0 if rank == 0 else 250.0
        tflops, ms_max = bench.job_throughput(1e12, 10, ms_local, world)
        # without --steps each rank sizes its run from its own warm-up; all
        # ranks then time the largest of those step counts
        steps = int(bench.max_over_ranks(float(2900 if rank == 0 else 3100), world))
        out[rank] = (tflops, ms_max, bench.dist_env(), steps)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_aggregation():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        tflops, ms_max, env, steps = res[rank]
        assert steps == 3100                        # every rank times the same K
        assert ms_max == 250.0                      # slowest rank
        assert tflops == pytest.approx(2 * 1e12 * 10 / 0.25 / 1e12)  # 80 TFLOPS
        assert env == (rank, world, rank)


def test_single_rank_is_local_time():
    tflops, ms = bench.job_throughput(2e12, 5, 10.0, 1)
    assert ms == 10.0 and tflops == pytest.approx(1000.0)
