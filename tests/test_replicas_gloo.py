"""The N-replica timing aggregation of bench.py on CPU: two gloo ranks, each
reporting its own elapsed time; the job rate is the units of all ranks over
the slowest rank's time."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [100.0, 250.0][rank]
    rate, job_ms = bench.replica_rate(64, ms)
    out[rank] = (rate, job_ms)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_rate_two_gloo_ranks():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:   # no fork of a multi-threaded process
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        rate, job_ms = res[r]
        assert job_ms == 250.0
        assert rate == pytest.approx(2 * 64 / 0.25)


def test_replica_rate_single_process():
    import bench
    rate, ms = bench.replica_rate(10, 500.0)
    assert ms == 500.0 and rate == pytest.approx(20.0)
