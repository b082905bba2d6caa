"""Replica bookkeeping of the benchmark across ranks, on CPU with the gloo backend.

The layer has no exchange step, so N GPUs run N independent replicas; the only collective
is the max-reduce of the timed region. Two gloo ranks with different local times must
agree on the slowest one and report the whole job's throughput from it.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.5][rank]
        ms = bench.max_over_ranks(local_ms, world)
        value = bench.replica_throughput(1_000_000, ms, world)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == 5.5
    # two replicas of 1 MB each per step over 5.5 ms
    assert value == pytest.approx(2 * 1_000_000 / 5.5e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.replica_throughput(4e9, 1000.0, 1) == pytest.approx(4.0)
