"""Host-side logic of the multi-rank benchmark path, as two gloo ranks on the
CPU: replicas share nothing on the data path; only a barrier and the
max-over-ranks time cross ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        assert (w, r, lr) == (world, rank, rank)
        bench.barrier(world)
        slowest = bench.max_over_ranks(10.0 + rank * 5.0, world)
        out[rank] = (slowest, bench.job_throughput(768, 100, slowest, world))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_job_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        slowest, value = out[r]
        assert slowest == 15.0
        assert value == pytest.approx(2 * 768 * 100 / 0.015)
