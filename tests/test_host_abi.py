"""CPU checks of the C ABI: libxy loads without a GPU, exports every declared symbol, and its host
calls (block table, task table) agree bit-exactly with the oracle and reject bad input."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads
from paged_kv_varlen_xy_gb300 import build as xybuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def xy():
    xybuild.build()
    import paged_kv_varlen_xy_gb300 as m
    m.lib()
    return m


def _declared():
    text = open(os.path.join(ROOT, "include", "xy.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(xy_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(xy):
    names = _declared()
    assert len(names) >= 8
    L = ctypes.CDLL(xy.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert sorted(xy.C_ABI) == names


def test_status_strings(xy):
    assert xy.status_string(0) == "ok"
    for code in range(-10, 0):
        assert xy.status_string(code) != "unknown status"
    assert xy.status_string(-99) == "unknown status"


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_block_table_matches_oracle_on_configs(xy, name):
    wl = workloads.make(name)
    mine, used = xy.xy_build_block_table(wl.context_lens, wl.block_size, wl.free_list, wl.max_blocks)
    ref = oracle.allocate_block_table(wl.context_lens, wl.block_size, wl.free_list, wl.max_blocks)
    assert np.array_equal(mine, ref)
    assert used == int(np.sum(-(-wl.context_lens.astype(np.int64) // wl.block_size)))


def test_block_table_fuzz(xy):
    rng = np.random.default_rng(0)
    for _ in range(50):
        S = int(rng.integers(1, 20))
        bs = int(2 ** rng.integers(4, 9))
        ctx = rng.integers(1, 2000, size=S)
        need = int(np.sum(-(-ctx // bs)))
        P = need + int(rng.integers(0, 10))
        free = rng.permutation(P).astype(np.int32)
        MB = int(np.max(-(-ctx // bs))) + int(rng.integers(0, 3))
        mine, _ = xy.xy_build_block_table(ctx, bs, free, MB)
        assert np.array_equal(mine, oracle.allocate_block_table(ctx, bs, free, MB))


def test_block_table_errors(xy):
    with pytest.raises(xy.XYError) as e:
        xy.xy_build_block_table([16, 17], 16, np.arange(2), 2)
    assert e.value.status == -9            # pool exhausted
    with pytest.raises(xy.XYError) as e:
        xy.xy_build_block_table([33], 16, np.arange(8), 2)
    assert e.value.status == -10           # more blocks than the table has columns
    with pytest.raises(xy.XYError) as e:
        xy.xy_build_block_table([3], 12, np.arange(8), 2)
    assert e.value.status == -1            # page size must be a power of two >= 16


def _tiles(G):
    return max(1, 64 // G), 4096


@pytest.mark.parametrize("schedule", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_task_table_matches_oracle_on_configs(xy, name, schedule):
    wl = workloads.make(name)
    qt, ch = _tiles(wl.group)
    if schedule >= 2:
        qt = xy.default_tiles(wl.num_heads_q, wl.num_heads_kv, wl.head_dim)[0]
    args = (wl.cu_seqlens_q, wl.context_lens, wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, 152, qt, ch,
            schedule)
    mine = xy.xy_build_task_table(*args)
    ref = oracle.build_task_table(*args)
    assert np.array_equal(mine["tasks"], ref["tasks"])
    assert np.array_equal(mine["merges"], ref["merges"])
    assert mine["workspace_bytes"] == ref["workspace_bytes"]
    assert mine["stats"]["max_cta_load"] == int(ref["cta_loads"].max())
    assert mine["stats"]["min_cta_load"] == int(ref["cta_loads"].min())
    assert mine["stats"]["total_load"] == int(ref["loads"].sum())
    assert mine["stats"]["balance"] == pytest.approx(ref["balance"], rel=1e-15)


def test_task_table_fuzz(xy):
    rng = np.random.default_rng(1)
    for _ in range(60):
        S = int(rng.integers(1, 12))
        q = rng.integers(1, 300, size=S)
        ctx = q + rng.integers(0, 3000, size=S)
        Hkv = int(rng.integers(1, 5))
        Hq = Hkv * int(rng.integers(1, 9))
        args = (oracle.pack_cu_seqlens(q), ctx, Hq, Hkv, int(rng.choice([64, 128])), bool(rng.integers(0, 2)),
                int(rng.integers(1, 200)), int(rng.integers(1, 70)), int(rng.choice([16, 64, 100, 256, 4096])),
                int(rng.integers(0, 5)))
        mine = xy.xy_build_task_table(*args)
        ref = oracle.build_task_table(*args)
        assert np.array_equal(mine["tasks"], ref["tasks"])
        assert np.array_equal(mine["merges"], ref["merges"])
        assert mine["workspace_bytes"] == ref["workspace_bytes"]


@pytest.mark.parametrize("schedule", [0, 1, 2, 3, 4])
def test_task_table_sort_regimes(xy, schedule):
    # the builder sorts loads with one counting pass when they span fewer than 2^16 steps of their
    # common power of two, else with an LSD radix sort: both give the oracle's stable order,
    # equal loads (ties) included
    narrow = ([1] * 40 + [3, 3], [700, 700, 650] + [512] * 37 + [40, 41], 4096)
    wide = ([1, 5, 300, 2, 77, 1], [1, 2000, 300, 70000, 900, 65536], 4096)
    unsplit = ([1, 2, 1, 1, 40], [1, 100000, 70000, 2, 99999], 131072)   # > 2^16 steps at every schedule
    for q, ctx, chunk in (narrow, wide, unsplit):
        args = (oracle.pack_cu_seqlens(q), np.array(ctx), 8, 2, 128, True, 7, 16, chunk, schedule)
        mine = xy.xy_build_task_table(*args)
        ref = oracle.build_task_table(*args)
        assert np.array_equal(mine["tasks"], ref["tasks"])
        assert np.array_equal(mine["merges"], ref["merges"])


def test_task_table_errors(xy):
    with pytest.raises(xy.XYError) as e:
        xy.xy_build_task_table([1, 3], [5], 4, 2, 64, True, 8, 8, 64)
    assert e.value.status == -2            # cu_seqlens[0] != 0
    with pytest.raises(xy.XYError) as e:
        xy.xy_build_task_table([0, 3, 3], [5, 5], 4, 2, 64, True, 8, 8, 64)
    assert e.value.status == -2            # not strictly increasing
    with pytest.raises(xy.XYError) as e:
        xy.xy_build_task_table([0, 6], [5], 4, 2, 64, True, 8, 8, 64)
    assert e.value.status == -4            # context shorter than the query
    with pytest.raises(xy.XYError) as e:
        xy.xy_build_task_table([0, 6], [9], 6, 4, 64, True, 8, 8, 64)
    assert e.value.status == -1            # Hq not a multiple of Hkv
    with pytest.raises(xy.XYError) as e:
        xy.xy_build_task_table([0, 3], [5], 4, 2, 64, True, 8, 8, 64, schedule=5)
    assert e.value.status == -1            # unknown schedule


def test_task_table_empty_batch(xy):
    r = xy.xy_build_task_table([0], [], 4, 2, 64, True, 8, 8, 64)
    assert r["tasks"].shape == (0, 8) and r["workspace_bytes"] == 0 and r["stats"]["balance"] == 1.0


def test_task_table_capacity_retry_and_out_arrays():
    # outputs written into caller arrays (one builder call), or retried when they are too small
    import paged_kv_varlen_xy_gb300 as xy
    cu = np.array([0, 1, 2, 40, 41], dtype=np.int32)
    ctx = np.array([900, 50, 7000, 33], dtype=np.int32)
    ref = xy.xy_build_task_table(cu, ctx, 16, 4, 128, 1, 9, 16, 256, 3)
    big_t, big_m = np.zeros((4096, 8), np.int32), np.zeros((512, 8), np.int32)
    r = xy.xy_build_task_table(cu, ctx, 16, 4, 128, 1, 9, 16, 256, 3, tasks_out=big_t, merges_out=big_m)
    assert np.shares_memory(r["tasks"], big_t) and np.shares_memory(r["merges"], big_m)
    small_t, small_m = np.zeros((3, 8), np.int32), np.zeros((1, 8), np.int32)
    r2 = xy.xy_build_task_table(cu, ctx, 16, 4, 128, 1, 9, 16, 256, 3, tasks_out=small_t, merges_out=small_m)
    for a in (r, r2):
        assert np.array_equal(a["tasks"], ref["tasks"]) and np.array_equal(a["merges"], ref["merges"])
        assert a["workspace_bytes"] == ref["workspace_bytes"]
    n, m = xy.task_table_bound(cu, ctx, 4, 16, 256)
    assert n >= int(np.sum(ref["tasks"][:, 0] >= 0)) and m >= len(ref["merges"])


def test_step_tables_pack_both_builders_outputs():
    import paged_kv_varlen_xy_gb300 as xy
    cu = np.array([0, 1, 2, 40, 41], dtype=np.int32)
    ctx = np.array([900, 50, 7000, 33], dtype=np.int32)
    free = np.random.default_rng(0).permutation(1000).astype(np.int32)
    args = (cu, ctx, free, 16, 448, 16, 4, 128, True, 9, 16, 256, 3)
    small = np.zeros(64, dtype=np.uint8)
    st, tbl = xy.xy_build_step_tables(*args, small.ctypes.data, small.nbytes)
    assert st == -10 and tbl.bytes > small.nbytes          # XY_ERR_CAPACITY, size reported
    buf = np.full(tbl.bytes + 100, 0xAB, dtype=np.uint8)
    st, tbl = xy.xy_build_step_tables(*args, buf.ctypes.data, buf.nbytes)
    assert st == 0
    for o in (tbl.err_off, tbl.cu_off, tbl.ctx_off, tbl.bt_off, tbl.tasks_off, tbl.merges_off):
        assert o % 256 == 0
    i32 = lambda off, n: buf[off:off + 4 * n].view(np.int32)
    bt, used = xy.xy_build_block_table(ctx, 16, free, 448)
    ref = xy.xy_build_task_table(cu, ctx, 16, 4, 128, True, 9, 16, 256, 3)
    assert i32(tbl.err_off, 1)[0] == 0
    assert np.array_equal(i32(tbl.cu_off, 5), cu) and np.array_equal(i32(tbl.ctx_off, 4), ctx)
    assert np.array_equal(i32(tbl.bt_off, bt.size).reshape(bt.shape), bt) and tbl.pages_used == used
    assert np.array_equal(i32(tbl.tasks_off, 8 * tbl.num_tasks).reshape(-1, 8), ref["tasks"])
    assert np.array_equal(i32(tbl.merges_off, 8 * tbl.num_merges).reshape(-1, 8), ref["merges"])
    assert tbl.workspace_bytes == ref["workspace_bytes"] and tbl.stats.balance == ref["stats"]["balance"]
    assert tbl.bytes == tbl.merges_off + 32 * tbl.num_merges


def test_default_kv_chunk_policy(xy):
    # the chunk with the least estimated makespan: four contexts of 128K keys beside many short
    # ones split into 32768-key tasks on 152 CTAs, 16384 on the pure-decode kernels' twice as many
    # CTAs; a single 1M-key context into 8192-key tasks (256 longer tasks would leave a second
    # round on some CTAs); contexts that no candidate splits take the longest chunk
    skew = workloads.make("skew")
    assert xy.default_kv_chunk(skew.context_lens, 64, 8, 152) == 32768
    assert xy.default_kv_chunk(skew.context_lens, 64, 8, 152, kv_fp8=True, pure_decode=True) == 16384
    assert xy.default_kv_chunk(skew.context_lens, 64, 8, 152, pure_decode=True) == 16384
    # G = 32 pure decode over 8-bit pages keeps one CTA per SM slot
    assert xy.default_kv_chunk(skew.context_lens, 256, 8, 152, kv_fp8=True, pure_decode=True) == 32768
    assert xy.default_kv_chunk([1 << 20], 8, 8, 152) == 8192
    assert xy.default_kv_chunk([100, 4096, 8000], 32, 8, 152) == 65536
    assert xy.default_kv_chunk([], 32, 8, 152) == 65536
    rng = np.random.default_rng(5)
    for _ in range(50):
        ctx = rng.integers(0, 300000, size=int(rng.integers(1, 40)))
        c = xy.default_kv_chunk(ctx, 8, 8, int(rng.integers(1, 300)), kv_fp8=bool(rng.integers(2)))
        assert c in (8192, 16384, 32768, 65536) and c % 256 == 0
    for bad in (dict(context_lens=[-1]), dict(num_ctas=0), dict(num_heads_q=6, num_heads_kv=4)):
        args = dict(context_lens=[10], num_heads_q=8, num_heads_kv=8, num_ctas=152)
        args.update(bad)
        with pytest.raises(xy.XYError):
            xy.default_kv_chunk(**args)
