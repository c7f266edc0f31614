"""The benchmark's multi-rank host logic on CPU: two gloo ranks (replicas
only -- requests are independent and no collective touches the data path).
Each rank times different work; the job's duration is the maximum over
ranks, its throughput counts every rank's rows, and ranks draw distinct
inputs."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import qsa_workloads as qw


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        dist.barrier()
        ms = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
        rows = bench.job_rows_per_second(world, 8, 100, ms)
        seeds = [bench.replica_seed(qw.WORKLOADS[1], i, rank) for i in range(4)]
        out[rank] = (ms, rows, seeds)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       join=True, start_method="spawn")
    (ms0, rows0, seeds0), (ms1, rows1, seeds1) = out[0], out[1]
    assert ms0 == ms1 == 2.5                       # the slower rank's time
    assert rows0 == rows1 == pytest.approx(2 * 8 * 100 / 0.0025)
    assert seeds0[0] == qw.WORKLOADS[1].seed         # rank 0, replica 0: the workload
    assert not set(seeds0) & set(seeds1)           # ranks draw distinct inputs


def test_single_rank_is_untouched():
    assert bench.max_over_ranks(3.25, 1, None) == 3.25
    assert bench.job_rows_per_second(1, 8, 10, 1.0) == pytest.approx(80000.0)
