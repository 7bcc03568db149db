"""The N>1 path of bench.py: independent replicas, one timing reduction.

Two gloo ranks on the CPU check that every rank ends up with the slowest
rank's time and that the job throughput counts every rank's units."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank)  # rank 1 is the slow one
        out[rank] = (slowest, bench.job_throughput(100.0, ws, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, thr = res[0]
    assert slowest == pytest.approx(15.0)
    assert thr == pytest.approx(2 * 100.0 / 15e-3)
