"""The N > 1 path of the bench on CPU: replicas under torch.distributed (gloo,
world size 2). Each rank times its own steps; the job's time is the slowest
rank's, and the reported throughput counts every rank's bytes."""
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
        dist.barrier()
        own = 10.0 + 5.0 * rank  # rank 1 is the slower replica
        ms = bench.reduce_step_time(torch, dist, torch.device("cpu"), own)
        out[rank] = ms
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 15.0


def test_job_value_counts_every_rank():
    one = bench.job_value(1e9, 1, 1.0)
    assert one == pytest.approx(1000.0)
    assert bench.job_value(1e9, 2, 1.0) == pytest.approx(2 * one)


def test_single_process_time_is_unchanged():
    assert bench.reduce_step_time(torch, None, torch.device("cpu"), 3.25) == 3.25
