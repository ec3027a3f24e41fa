"""Replica mode of bench.py on CPU: world size 2 over gloo.  The path shards into independent
replicas with no data-path exchange; the only collective is the max-over-ranks reduction of the
timed region, and the job's value counts the units of every rank.  Without a GPU, a rank's step is
its host half through the C ABI (block table and task table) with the oracle standing in for the
device half."""

import os
import socket
import sys
import time

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


def _step_rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np
    import bench
    import oracle
    import paged_kv_varlen_xy_gb300 as xy
    import workloads
    wl = workloads.tiny()   # every replica runs the same batch (weak scaling: N ranks, N batches)
    vals = wl.tensors("cpu")
    bits = {k: v.contiguous().view(torch.int16).numpy().view(np.uint16) for k, v in vals.items()}
    t0 = time.perf_counter()
    bt, _ = xy.xy_build_block_table(wl.context_lens, wl.block_size, wl.free_list, wl.max_blocks)
    qt, kc = xy.default_tiles(wl.num_heads_q, wl.num_heads_kv, wl.head_dim)
    tasks = xy.xy_build_task_table(wl.cu_seqlens_q, wl.context_lens, wl.num_heads_q, wl.num_heads_kv, wl.head_dim,
                                   wl.causal, 8, qt, kc, xy.XY_SCHEDULE_DYNAMIC)["tasks"]
    ref = oracle.step.run_step(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                               bits["q"], bits["k_new"], bits["v_new"], bits["k_pool"], bits["v_pool"], wl.scale,
                               wl.causal)
    secs = time.perf_counter() - t0
    t = bench.max_over_ranks(secs, world)
    q.put((rank, secs, t, bt.tobytes(), tasks.tobytes(), ref["out"].tobytes(),
           np.array_equal(bt, ref["block_table"])))
    dist.destroy_process_group()


def test_two_replicas_each_run_a_step():
    # each rank plans and runs its own step; the replicas agree bit for bit (no rank reads another's
    # data) and the job's time is the slower rank's
    from paged_kv_varlen_xy_gb300 import build
    build.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_step_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, s0, t0, bt0, tk0, out0, ok0), (_, s1, t1, bt1, tk1, out1, ok1) = res
    assert ok0 and ok1, "host block table differs from the oracle's allocation"
    assert bt0 == bt1 and tk0 == tk1 and out0 == out1
    assert t0 == t1 == pytest.approx(max(s0, s1))
