"""The bench's multi-rank path on CPU: world size 2 over gloo.

Each rank runs a replica of the workload; the job time is the slowest rank's and the
throughput counts every rank's FLOPs.  No GPU is involved.
"""

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

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [2.0, 3.0][rank]  # rank 1 is the slow one
        value, tmax = bench.aggregate_throughput(local, 1e12, 10)
        out[rank] = (value, tmax)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_takes_slowest_rank():
    mp_ctx = mp.get_context("spawn")
    mgr = mp_ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for rank in (0, 1):
        value, tmax = out[rank]
        assert tmax == 3.0
        # 2 ranks x 10 steps x 1e12 FLOP / 3 s = 6.67 TFLOP/s
        assert value == pytest.approx(2 * 10 * 1e12 / 3.0 / 1e12)


def test_single_process_aggregation():
    import bench
    value, tmax = bench.aggregate_throughput(2.0, 1e12, 10)
    assert tmax == 2.0 and value == pytest.approx(5.0)
