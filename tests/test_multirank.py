"""The benchmark's multi-rank host logic on CPU: world size 2 over gloo.

Each rank runs its own replica (weak scaling, no collective on the data
path); the only collectives are the barrier around the timed region and the
max of the per-rank elapsed times, which these tests exercise.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        bench.barrier(world)
        elapsed = 10.0 + 5.0 * rank  # rank 1 is the slow one
        mx = bench.max_over_ranks(elapsed, world)
        out[rank] = mx
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_world_size_2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_is_identity_and_weak_scaling_value():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    # whole-job value counts every rank's work over the slowest rank's time
    flops = bench.causal_attn_flops(1, 32, 8192, 128)
    assert flops == pytest.approx(549822922752.0)
    assert bench.dense_attn_flops(4, 16, 4096, 4096, 64) == pytest.approx(274877906944.0)
    assert bench.softmax_bytes(4096, 32768) == 1073758208.0
