"""The split step over 8-bit pages through the C ABI alone (no step.py): xy_build_fp8_step_tables
on the host, xy_kv_append_paged_fp8 and xy_paged_attention_fp8_mixed on the device.  Host tests
check the builder's tables against the host calls they compose; GPU tests check the step against
the oracle (codes and scales bit for bit, outputs within the bf16 tolerance)."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads


@pytest.fixture(scope="module")
def xy():
    from paged_kv_varlen_xy_gb300 import build
    build.build()
    import paged_kv_varlen_xy_gb300 as m
    return m


def _tables(xy, wl, num_ctas=37, max_blocks=None):
    mb = max_blocks or wl.max_blocks
    staging = np.zeros(1 << 22, dtype=np.uint8)
    st, t = xy.xy_build_fp8_step_tables(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, mb,
                                        wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, num_ctas,
                                        staging.ctypes.data, staging.nbytes)
    assert st == 0
    return staging, t, mb


def _i32(staging, off, n):
    return staging[off:off + 4 * n].view(np.int32)


@pytest.mark.parametrize("q_lens,ctx", [([40, 300, 1, 1, 1], [300, 900, 700, 33, 1]),
                                        ([1, 1, 17, 64], [4000, 90, 500, 64]),
                                        ([1, 1, 1], [10, 20, 30]),
                                        ([5, 9], [5, 300])])
def test_builder_tables_compose_the_host_calls(xy, q_lens, ctx):
    wl = workloads.custom(q_lens, ctx, 8, 2, 128, 16, seed=3)
    staging, t, mb = _tables(xy, wl)
    cu, L = wl.cu_seqlens_q, wl.context_lens
    multi = np.asarray(q_lens) > 1
    tile = [i for i in range(len(q_lens)) if multi[i]]
    dec = [i for i in range(len(q_lens)) if not multi[i]]
    assert list(range(t.tile_seq_begin, t.tile_seq_end)) == tile
    assert list(range(t.dec_seq_begin, t.dec_seq_end)) == dec
    S = len(q_lens)
    bt, _ = xy.xy_build_block_table(L, wl.block_size, wl.free_list, mb)
    assert np.array_equal(_i32(staging, t.bt_off, S * mb).reshape(S, mb), bt)
    assert np.array_equal(_i32(staging, t.cu_off, S + 1), cu)
    assert _i32(staging, t.err_off, 1)[0] == 0
    # the tile part's page list and its block table over the copies
    pages = _i32(staging, t.tile_pages_off, t.tile_num_pages)
    want = [int(p) for i in tile for p in bt[i][: -(-int(L[i]) // wl.block_size)]]
    assert pages.tolist() == want
    if tile:
        bt_t = _i32(staging, t.tile_bt_off, len(tile) * mb).reshape(len(tile), mb)
        for r, i in enumerate(tile):
            n = -(-int(L[i]) // wl.block_size)
            assert np.array_equal(pages[bt_t[r][:n]], bt[i][:n]) and (bt_t[r][n:] == -1).all()
    # each part's task table is xy_build_task_table's for its sub-batch (dynamic deal)
    for idx, off_cu, off_t, off_m, nt, nm, fp8 in (
            (tile, t.tile_cu_off, t.tile_tasks_off, t.tile_merges_off, t.tile_num_tasks, t.tile_num_merges, False),
            (dec, t.dec_cu_off, t.dec_tasks_off, t.dec_merges_off, t.dec_num_tasks, t.dec_num_merges, True)):
        if not idx:
            assert nt == 0
            continue
        a, b = idx[0], idx[-1] + 1
        sub_cu = (cu[a:b + 1] - cu[a]).astype(np.int32)
        assert np.array_equal(_i32(staging, off_cu, b - a + 1), sub_cu)
        qt, _ = xy.default_tiles(8, 2, 128, kv_fp8=fp8, pure_decode=fp8)
        ch = xy.default_kv_chunk(L[a:b], 8, 2, 37, kv_fp8=fp8, pure_decode=fp8)
        r = xy.xy_build_task_table(sub_cu, L[a:b], 8, 2, 128, True, 37, qt, ch, xy.XY_SCHEDULE_DYNAMIC)
        assert np.array_equal(_i32(staging, off_t, 8 * nt).reshape(nt, 8), r["tasks"])
        assert np.array_equal(_i32(staging, off_m, 8 * nm).reshape(nm, 8), r["merges"])


def test_builder_rejects_interleaved_kinds_and_reports_capacity(xy):
    wl = workloads.custom([1, 5, 1, 5], [10, 20, 30, 40], 8, 2, 128, 16, seed=4)
    staging = np.zeros(1 << 16, dtype=np.uint8)
    with pytest.raises(xy.XYError) as e:
        xy.xy_build_fp8_step_tables(wl.cu_seqlens_q, wl.context_lens, wl.free_list, 16, wl.max_blocks, 8, 2, 128,
                                    True, 37, staging.ctypes.data, staging.nbytes)
    assert e.value.status == -5
    wl = workloads.custom([5, 1], [20, 30], 8, 2, 128, 16, seed=4)
    st, t = xy.xy_build_fp8_step_tables(wl.cu_seqlens_q, wl.context_lens, wl.free_list, 16, wl.max_blocks, 8, 2, 128,
                                        True, 37, staging.ctypes.data, 64)
    assert st == -10 and t.bytes > 64


@pytest.mark.gpu
@pytest.mark.parametrize("q_lens,ctx,G", [([40, 300, 1, 1, 1], [300, 900, 700, 33, 1], 4),
                                          ([1, 1, 17, 64, 3], [9000, 90, 500, 64, 3], 8),
                                          ([512, 512] + [1] * 30, [600, 4000] + list(range(100, 3100, 100)), 4)])
def test_mixed_step_through_the_c_abi_matches_the_oracle(xy, q_lens, ctx, G):
    dev = torch.device("cuda")
    wl = workloads.custom(q_lens, ctx, 2 * G, 2, 128, 16, seed=77)
    vals = wl.tensors(dev)
    P, Hkv, bs, d = vals["k_pool"].shape
    codes = [torch.zeros(P, Hkv, bs, d, dtype=torch.uint8, device=dev) for _ in range(2)]
    scales = [torch.zeros(P, Hkv, bs, dtype=torch.float32, device=dev) for _ in range(2)]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    rows = [vals[n].permute(0, 2, 1, 3).reshape(P * bs, Hkv, d).contiguous() for n in ("k_pool", "v_pool")]
    xy.xy_kv_append_fp8(rows[0], rows[1], torch.arange(P * bs, dtype=torch.int64, device=dev), codes[0], codes[1],
                        scales[0], scales[1], err)
    staging, t, mb = _tables(xy, wl, num_ctas=xy.xy_default_num_ctas(0))
    tables = torch.from_numpy(staging[:t.bytes].copy()).to(dev)
    S = wl.num_seqs

    def dv(off, n):
        return tables[off:off + 4 * n].view(torch.int32)

    cu, ctxd, bt = dv(t.cu_off, S + 1), dv(t.ctx_off, S), dv(t.bt_off, S * mb).view(S, mb)
    slots = torch.empty(wl.num_tokens, dtype=torch.int64, device=dev)
    xy.xy_kv_append_paged_fp8(vals["k_new"], vals["v_new"], cu, ctxd, bt, codes[0], codes[1], scales[0], scales[1],
                              err, slot_mapping=slots)
    n = max(t.tile_num_pages, 1)
    copy_k = torch.empty(n, Hkv, bs, d, dtype=torch.bfloat16, device=dev)
    copy_v = torch.empty_like(copy_k)
    ws = [torch.empty(max(16, x), dtype=torch.uint8, device=dev) for x in (t.tile_workspace_bytes,
                                                                          t.dec_workspace_bytes)]
    counters = torch.zeros(4, dtype=torch.int32, device=dev)
    out = torch.full_like(vals["q"], float("nan"))
    for _ in range(2):   # the claim counters return to zero: a second call runs every task again
        xy.xy_paged_attention_fp8_mixed(vals["q"], tables, t, codes[0], codes[1], scales[0], scales[1], S, mb,
                                        wl.scale, True, xy.xy_default_num_ctas(0), copy_k, copy_v, ws[0], ws[1],
                                        counters, err, out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert counters.cpu().tolist() == [0, 0, 0, 0]

    def bits(x):
        return x.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.step.run_step_fp8(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, mb,
                                   bits(vals["q"]), bits(vals["k_new"]), bits(vals["v_new"]), bits(vals["k_pool"]),
                                   bits(vals["v_pool"]), wl.scale, True)
    assert np.array_equal(slots.cpu().numpy(), ref["slots"])
    assert np.array_equal(codes[0].cpu().numpy(), ref["k_codes"])
    assert np.array_equal(codes[1].cpu().numpy(), ref["v_codes"])
    assert np.array_equal(scales[0].cpu().numpy().view(np.uint32), ref["k_scales"].view(np.uint32))
    assert np.array_equal(scales[1].cpu().numpy().view(np.uint32), ref["v_scales"].view(np.uint32))
    got = oracle.bf16_bits_to_f64(bits(out))
    diff = np.abs(got - ref["out"])
    assert np.isfinite(got).all() and diff.max() <= 2e-2 and diff.mean() <= 2e-3, (diff.max(), diff.mean())
