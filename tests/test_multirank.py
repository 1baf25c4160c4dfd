"""Host logic of the multi-process bench path on CPU: two gloo ranks, each
timed differently; the reported time is the slowest rank's on every rank, and
the whole-job throughput counts every replica's tokens (weak scaling).  The
layer itself has no exchange step on one GPU, so replicas share no data."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(100.0 + 7.5 * rank, world, "cpu")
        value = bench.replica_throughput(16384, world, 10, ms)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_replica_throughput_gloo(world):
    port = _free_port()
    mgr = tmp.get_context("spawn").Manager()   # no fork of a multi-threaded process
    out = mgr.dict()
    tmp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    slowest = 100.0 + 7.5 * (world - 1)
    for r in range(world):
        ms, value = out[r]
        assert ms == slowest
        assert value == pytest.approx(16384 * world * 10 / (slowest / 1e3))


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.replica_throughput(100, 1, 4, 2000.0) == pytest.approx(200.0)
