"""bench.py's multi-rank logic with two gloo ranks on CPU: the job time is the
slowest rank's, and the throughput counts the work of every rank (weak
scaling: each rank runs the whole workload on its own GPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        elapsed = [12.0, 15.0][rank]              # rank 1 is the slower one
        m = bench.max_over_ranks(elapsed, world, device="cpu")
        value = bench.job_throughput(30e9, 100, m, world)
        out[rank] = (m, value)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_job_throughput():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
    assert out[0][0] == 15.0 and out[1][0] == 15.0
    expect = 30e9 * 100 * 2 / 15e-3 / 1e12
    assert out[0][1] == pytest.approx(expect) and out[1][1] == pytest.approx(expect)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1e12, 10, 1000.0, 1) == pytest.approx(10.0)   # 1e13 FLOP in 1 s
