"""The N>1 host path of bench.py on CPU: two gloo ranks, each a replica with its own
timing; the slowest rank's time and the sum of every rank's bytes make the job figure."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench._dist_env() == (world, rank, rank)
        mine = [1.0 + rank, 0.5 * (2 - rank), 3.0]
        got = bench.reduce_max_over_ranks(mine, torch.device("cpu"))
        value = bench.aggregate_value(world, 1e9, 10, got[0])
        q.put((rank, got, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_benchmark():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [2.0, 1.0, 3.0]                 # max over ranks, elementwise
        assert value == pytest.approx(2 * 1e9 * 10 / 2.0 / 1e9)
