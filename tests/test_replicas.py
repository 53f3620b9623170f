"""The replica bench's cross-rank logic on CPU: two gloo ranks on 127.0.0.1."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # each replica measured a different time; the job takes the slowest
        ms = bench.max_over_ranks(10.0 + rank * 2.5, torch.device("cpu"), world)
        out[rank] = (ms, bench.whole_job_rate(64, world, 100, ms / 1e3))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, rate = res[0]
    assert ms == 12.5
    assert rate == pytest.approx(64 * world * 100 / 12.5e-3)


def test_single_replica_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, torch.device("cpu"), 1) == 3.25
    assert bench.whole_job_rate(64, 1, 10, 0.5) == 64 * 10 / 0.5
