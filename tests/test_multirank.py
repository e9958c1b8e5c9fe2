"""The multi-GPU path of bench.py, on CPU: world_size-2 gloo ranks, each with
its own problem, agree on the slowest rank's time and report the whole-job
throughput (weak scaling, no collective on the data path)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "took" 10 + r ms for its steps, and (3 - r) s end to end
        got = bench.max_over_ranks([10.0 + rank, 3.0 - rank, 1.0], torch.device("cpu"), world)
        dist.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    port = _free_port()
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
        results = dict(out)
    assert results[0] == results[1] == [11.0, 3.0, 1.0]


def test_job_throughput_is_weak_scaling():
    flops = 2 * 4096 ** 3
    one = bench.job_throughput(1, 100, flops, 10.0)
    two = bench.job_throughput(2, 100, flops, 10.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(100 * flops / 0.01 / 1e12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([1.5, 2.5], torch.device("cpu"), 1) == [1.5, 2.5]
