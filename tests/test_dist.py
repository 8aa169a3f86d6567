"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): barrier,
max of step times over ranks, and the whole-job (weak-scaling) value."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        r, lr, w = bench.dist_env()
        assert (r, lr, w) == (rank, rank, world)
        bench.barrier(world)
        # rank r takes (r + 1) ms per step on 1e6 bytes
        value, slowest = bench.job_throughput(10 ** 6, float(rank + 1), world)
        out[rank] = (value, slowest)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_weak_scaling_aggregation():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out),
                           nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    # slowest rank: 2 ms; job bytes: 2e6 -> 1 GB/s, the same on every rank
    for rank in range(world):
        value, slowest = res[rank]
        assert slowest == 2.0
        assert abs(value - 1.0) < 1e-12


def test_single_rank_is_identity():
    import bench
    value, slowest = bench.job_throughput(88_309_760, 0.0154, 1)
    assert slowest == 0.0154
    assert abs(value - 88_309_760 / 15.4e-6 / 1e9) < 1e-6
