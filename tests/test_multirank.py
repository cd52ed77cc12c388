"""The benchmark's multi-rank path (replicas only: one process per GPU, no data-path collective)
on CPU with gloo, world size 2: a barrier, the timing taken as the maximum over ranks, and the
whole-job throughput."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, l = bench.dist_setup()
    assert (w, r, l) == (world, rank, rank)
    dist.barrier()
    mine = 100.0 + 50.0 * rank          # ms: rank 1 is the slow one
    got = bench.max_over_ranks(mine, "cpu")
    value = bench.job_throughput(world, 256, 10, got)
    q.put((rank, got, value))
    dist.destroy_process_group()


def test_two_rank_timing_is_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, got, value in res:
        assert got == 150.0
        assert value == pytest.approx(2 * 256 * 10 / 0.150)


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_throughput(1, 256, 4, 1000.0) == pytest.approx(1024.0)
