"""The benchmark's multi-rank logic on CPU: two gloo ranks, no GPU.

Replicas-only scaling: each rank times its own copy of the workload; the job
reports the bytes of all ranks over the slowest rank's time.  This checks the
max-over-ranks reduction and the whole-job throughput with world size 2.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as tmp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = [120.0, 80.0][rank]
        m = bench.max_over_ranks(local_ms)
        v = bench.job_gbs(10 ** 9, 10, dist.get_world_size(), m)
        dist.barrier()
        out[rank] = (m, v)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = tmp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    tmp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True,
                        start_method="spawn")
    assert out[0] == out[1]
    m, v = out[0]
    assert m == 120.0                                   # the slowest rank's time
    assert v == pytest.approx(2 * 10 * 1e9 / 0.120 / 1e9)


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_gbs(4 * 10 ** 9, 2, 1, 1000.0) == pytest.approx(8.0)
