"""The bench's multi-process host logic (rank setup, barrier, max over ranks)
with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w, lr = bench.dist_setup()
    bench.barrier(w)
    m = bench.reduce_max(float(10 * (rank + 1)), w)
    out[rank] = m
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_barrier_and_max():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 20.0


def test_flop_model_counts():
    import bench
    f = bench.step_flops(2, 16, 16384, 128)
    N, C, d, BH = 128, 128, 128, 32
    assert f["attn"] == BH * (C * C * d * N * (N - 1) + C * C * d * N * (N + 1)
                              + C * d * d * (N - 1) * (N - 2))
    assert f["flash_equiv"] == 2 * BH * 16384 * 16384 * d
