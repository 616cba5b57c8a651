"""Replica sharding and the job-throughput reduction, as world-size-2 gloo process groups on CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_exact_speculative_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seconds = [2.0, 3.0][rank]          # rank 1 is the slow one
        units = [64.0, 80.0][rank]
        value, slowest, total = replicas.job_throughput(seconds, units)
        q.put((rank, replicas.rank_seed(7, rank), value, slowest, total))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_slowest_time_and_summed_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, v0, t0, u0), (r1, s1, v1, t1, u1) = out
    assert (r0, r1) == (0, 1)
    assert s0 != s1                                  # every rank verifies its own sequences
    assert t0 == t1 == 3.0 and u0 == u1 == 144.0     # slowest time, summed work, on every rank
    assert v0 == v1 == pytest.approx(48.0)


def test_single_process_needs_no_group():
    assert replicas.job_throughput(2.0, 10.0) == (5.0, 2.0, 10.0)
    assert replicas.rank_seed(0, 0) == 0 and replicas.rank_seed(0, 1) == replicas.RANK_SEED_STRIDE
