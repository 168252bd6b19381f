"""The multi-process path of bench.py on CPU (gloo, world size 2): the joint
block has no exchange step for one sample, so N processes run N independent
replicas; the whole-job throughput is every rank's units over the slowest
rank's step time, the same number on every rank."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, step_ms, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        value, slowest = bench.replica_throughput(4608, step_ms[rank], world, "cpu")
        out[rank] = (value, slowest)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_all_units_over_the_slowest_rank():
    world = 2
    step_ms = [1.0, 1.25]                    # rank 1 is the slower replica
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), step_ms, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        value, slowest = res[rank]
        assert slowest == pytest.approx(1.25)
        assert value == pytest.approx(2 * 4608 / 1.25e-3)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    value, slowest = bench.replica_throughput(100, 2.0, 1, "cpu")
    assert (value, slowest) == (pytest.approx(5e4), 2.0)
