"""The multi-GPU path of the benchmark is replicas only: every rank runs the
workload on its own inputs, the job's time is the slowest rank's, and its
throughput counts every rank's bytes. The host logic runs here as two gloo
ranks on the CPU."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.replica_barrier(world)
        # rank r timed (10 + r) ms for the device pass and (20 - r) ms end to end
        ms, ms_e2e = bench.replica_max([10.0 + rank, 20.0 - rank], world)
        out[rank] = (ms, ms_e2e, bench.job_tbps(world, 1e9, 5, ms))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_every_rank():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        got = dict(out)
    for r in range(world):
        ms, ms_e2e, tb = got[r]
        assert ms == 11.0 and ms_e2e == 20.0       # max over ranks, on every rank
        assert tb == pytest.approx(2 * 1e9 * 5 / 11e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.replica_max([3.0, 4.0], 1) == [3.0, 4.0]
    bench.replica_barrier(1)
    assert bench.job_tbps(1, 2e12, 1, 1000.0) == pytest.approx(2.0)
