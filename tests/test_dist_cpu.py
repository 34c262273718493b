"""Multi-rank host logic of the benchmark on the CPU (gloo, world size 2).

The attention path needs no data exchange between GPUs: under torchrun every
rank runs its own replica and only the timing is reduced.  This checks that
reduction -- the slowest rank's time sets the whole-job throughput -- with
two gloo ranks.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        slowest = bench.max_over_ranks(local_ms, dist, "cpu")
        out[rank] = (slowest, bench.aggregate_tflops(world, 2.0e12, slowest))
    finally:
        dist.destroy_process_group()


def test_two_replicas_reduce_to_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, value = res[rank]
        assert slowest == 5.0
        assert value == pytest.approx(2 * 2.0e12 / 5e-3 / 1e12)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(4.5, None, "cpu") == 4.5
    assert bench.aggregate_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)
