"""The multi-rank bench plumbing on CPU with gloo, world size 2: replicas
exchange nothing but the max-reduction of their timings, and the reported
rate is the sum over ranks."""

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        # rank r took 10 * (r + 1) ms for 5 steps of 4096 tokens
        ms = bench.max_over_ranks(dist, 10.0 * (rank + 1), torch.device("cpu"))
        rate = bench.whole_job_rate(world, 4096, 5, ms)
        out[rank] = (ms, rate)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_report_the_slowest_rank():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1]
    ms, rate = out[0]
    assert ms == 20.0                              # max over ranks
    assert rate == pytest.approx(2 * 4096 * 5 / 0.020)


def test_single_process_path_needs_no_collective():
    assert bench.max_over_ranks(None, 12.5, torch.device("cpu")) == 12.5
    assert bench.whole_job_rate(1, 4096, 10, 20.0) == pytest.approx(4096 * 10 / 0.020)
