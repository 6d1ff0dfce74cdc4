"""The N > 1 path of bench.py on CPU with two gloo ranks.

Each rank runs its own replica of the stage on its own microbatches (the path
shards by microbatch with no collective); torch.distributed only frames the
timing: a barrier, and the max over ranks of every timed quantity.  The
replica test runs a small stage per rank (the float64 oracle standing in for
the GPU kernels, in the library's ZB-H1 order) and checks that what a rank
computes depends on its own microbatches only: equal to the same stage run in
one process, whatever the other rank does.
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
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        for r in range(world):
            assert out[r] == [2.0, 10.0, 5.0]


STAGE = dict(kind="transformer", n_layers=2, hidden=64, ffn=128, n_heads=4, n_kv_heads=2, head_dim=16,
             eps=1e-5, attention="standin", seq_len=0)


def _replica(rank, p=4, m=6):
    """One rank's replica: stage `rank` of the pipeline order on microbatches drawn with seed = rank.
    Returns (dx per microbatch, float64 weight gradients per layer)."""
    import numpy as np

    from backward_split_linear_gb300 import synth
    from oracle import schedule as OS
    from oracle import stage as S

    c = STAGE
    inp = synth.stage_inputs(c["kind"], c["n_layers"], c["hidden"], c["ffn"], c["n_heads"], c["n_kv_heads"],
                             c["head_dim"], tokens=24, n_mb=m, seed=rank)
    params = synth.params_f64(inp["params"])
    orc = S.StageOracle(params, c)
    dx = {}
    for kind, mb in OS.orders_for("zbh1", p, m)[rank % p]:
        if kind == "F":
            orc.forward(mb, synth.bf16_to_f64(inp["x"][mb]))
        elif kind == "B":
            dx[mb] = orc.backward_input(mb, synth.bf16_to_f64(inp["dy"][mb]))
        else:
            orc.backward_weight(mb)
    return [dx[i] for i in range(m)], [{k: np.asarray(v) for k, v in g.items()} for g in orc.grads]


def _rank_replica(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    dist.barrier()
    dx, grads = _replica(rank)
    ms = bench.max_over_ranks([float(len(dx))], dist, "cpu")
    dist.barrier()
    out[rank] = (dx, grads, ms)
    dist.destroy_process_group()


def test_replicas_two_gloo_ranks_equal_single_process():
    import numpy as np

    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_replica, args=(world, port, out), nprocs=world, join=True)
        got = {r: out[r] for r in range(world)}
    for r in range(world):
        dx, grads, ms = got[r]
        ref_dx, ref_grads = _replica(r)
        assert ms == [6.0]
        assert all(np.array_equal(a, b) for a, b in zip(dx, ref_dx))
        for g, rg in zip(grads, ref_grads):
            assert g.keys() == rg.keys()
            assert all(np.array_equal(g[k], rg[k]) for k in g)
    # the two replicas ran on different microbatches and kept their own gradients
    assert not np.array_equal(got[0][1][0]["w_gu"], got[1][1][0]["w_gu"])


def test_whole_job_rate():
    import bench

    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    # two ranks each doing 1 TFLOP in 1 s: 2 TFLOP/s for the job
    assert abs(bench.whole_job_tflops(1e12, 2, 1000.0) - 2.0) < 1e-12
