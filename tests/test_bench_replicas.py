"""The multi-GPU path of bench.py is replicas only: every rank runs its own
batch, the job's time is the slowest rank's, and the job's throughput counts
every replica.  The host logic runs here on two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [120.0, 150.0][rank]  # the ranks' local times of K steps
    job_ms = bench.slowest_rank(ms, torch.device("cpu"), True)
    value = bench.job_throughput(512, world, 1000, job_ms)
    q.put((rank, job_ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, job_ms, value in got:
        assert job_ms == 150.0
        assert value == pytest.approx(512 * 2 * 1000 / 0.150)


def test_single_rank_is_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank(123.0, torch.device("cpu"), False) == 123.0
    assert bench.job_throughput(512, 1, 10, 1000.0) == pytest.approx(5120.0)
