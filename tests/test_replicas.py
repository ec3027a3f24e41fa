"""Replica mode of bench.py on CPU: world size 2 over gloo.  The path shards into independent
replicas with no data-path exchange; the only collective is the max-over-ranks reduction of the
timed region, and the job's value counts the units of every rank."""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads
    # each replica reports its own time; the slowest sets the job's time
    secs = [0.010, 0.025][rank]
    t = bench.max_over_ranks(secs, world)
    w = bench.work(workloads.make("decode"))
    v = bench.job_throughput("decode", w, t, world)
    q.put((rank, t, v, bench.throughput("decode", w, t)))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, v0, one0), (r1, t1, v1, one1) = res
    assert t0 == t1 == pytest.approx(0.025)
    assert v0 == v1 == pytest.approx(2 * one0)


def test_single_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1) == 0.5
