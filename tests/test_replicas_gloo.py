"""The multi-rank bookkeeping of bench.py (replicas: one independent view per rank) on two CPU
ranks with the gloo backend: the step time is the slowest rank's, the throughput counts every
rank's pixels."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.reduce_max(10.0 + 5.0 * rank, world)  # rank 1 is slower
        out[rank] = (ms, bench.throughput_mpix(world, 1_000_000, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_whole_job_throughput():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this (possibly threaded) process
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    assert res[0][0] == pytest.approx(15.0) and res[1][0] == pytest.approx(15.0)
    # 2 ranks x 1 Mpix per 15 ms step
    assert res[0][1] == pytest.approx(2 * 1.0 / 0.015)


def test_single_rank_is_identity():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.throughput_mpix(1, 2_000_000, 10.0) == pytest.approx(200.0)
