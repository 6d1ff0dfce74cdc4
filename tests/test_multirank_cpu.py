"""The N > 1 timing frame of bench.py on CPU with two gloo ranks.

Each rank runs its own replica of the stage (the path shards by microbatch
with no collective); torch.distributed only frames the timing: a barrier,
and the max over ranks of every timed quantity.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    dist.barrier()
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 5.0], dist, "cpu")
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        for r in range(world):
            assert out[r] == [2.0, 10.0, 5.0]


def test_whole_job_rate():
    import bench

    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    # two ranks each doing 1 TFLOP in 1 s: 2 TFLOP/s for the job
    assert abs(bench.whole_job_tflops(1e12, 2, 1000.0) - 2.0) < 1e-12
