"""The multi-GPU path is replicas only: each rank runs the whole block on its own batch and bench.py
reports the whole job's tokens/s over the slowest rank's time.  These checks run the ranks' host
logic as two gloo processes on the CPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow replica
        total = bench.max_over_ranks(ms, "cpu")
        out[rank] = (total, bench.whole_job_rate(4, 100, world, total))
        # the reference arm: rank 0 alone runs it, the others return nothing
        if rank != 0:
            out[rank + 10] = bench.reference_arm(type("A", (), {"config": 1, "steps": 1, "warmup": 0, "seed": 0}), rank)
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_the_whole_job_rate():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0
    # 2 replicas x 4 tokens x 100 steps in 15 ms
    assert out[0][1] == pytest.approx(2 * 4 * 100 / 0.015)
    assert out[11] is None


def test_whole_job_rate_scales_with_replicas():
    assert bench.whole_job_rate(4, 10, 1, 1000.0) == pytest.approx(40.0)
    assert bench.whole_job_rate(4, 10, 8, 1000.0) == pytest.approx(320.0)
