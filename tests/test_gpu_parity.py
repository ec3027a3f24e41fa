"""GPU parity: the CUDA path through the C ABI against the oracle on the same seeded inputs.

Block table, slot mapping and appended pages are compared bit for bit; attention outputs (bf16,
fp32 accumulation) against the fp64 oracle within max-abs 2e-2 and mean-abs 2e-3.  Small batches
are compared on every row; the full-size workloads on sampled sequences and rows, in the launch
configuration bench.py times."""

import numpy as np
import pytest
import torch

import workloads
from gpu_cases import assert_parity, run, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_varlen_xy_gb300 import build
    build.build()


def test_tiny_mixed_batch_every_row():
    r = run(workloads.tiny())
    assert_parity(r)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [16, 256])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_batch_every_row(d, bs, causal):
    # several 64-row tiles with ragged tails, GQA 4, prior context, decode rows
    wl = workloads.custom([1, 17, 130, 77, 40, 1], [1, 40, 130, 500, 333, 700], 8, 2, d, bs, causal=causal,
                          seed=100 + d + bs + int(causal))
    assert_parity(run(wl))


@pytest.mark.parametrize("kv_chunk", [128, 256, 384])
def test_split_kv_and_combine_every_row(kv_chunk):
    wl = workloads.custom([3, 1, 50, 1], [700, 520, 190, 64], 8, 2, 128, 16, seed=kv_chunk)
    r = run(wl, kv_chunk=kv_chunk)
    assert len(r["batch"].plan.host["merges"]) > 0
    assert_parity(r)


@pytest.mark.parametrize("G", [1, 2, 8, 16])
def test_gqa_groups(G):
    wl = workloads.custom([1, 5, 33, 2], [90, 5, 70, 130], 2 * G, 2, 128, 16, seed=G)
    assert_parity(run(wl))


def test_nan_in_unused_slots_never_reaches_outputs():
    # the whole pool starts as NaN; the step appends every context token (q = L), so only
    # slots past each context end and untouched pages stay NaN
    wl = workloads.custom([5, 37, 64, 70], [5, 37, 64, 70], 4, 2, 128, 16, seed=3)
    r = run(wl, pool_fill=float("nan"))
    assert_parity(r, check_pages=False)
    wl = workloads.custom([5, 37, 64, 70], [5, 37, 64, 70], 4, 2, 128, 16, seed=3)
    r = run(wl, pool_fill=float("nan"), kv_chunk=128)
    assert_parity(r, check_pages=False)


def test_num_ctas_variants():
    wl = workloads.custom([1, 9, 1, 100], [300, 9, 20, 130], 8, 4, 64, 16, seed=5)
    for n in (1, 3, 300):
        assert_parity(run(wl, num_ctas=n))


@pytest.mark.parametrize("G", [1, 4, 8])
def test_verify_shaped_queries(G):
    # speculative-verify batches ([ATB] 投机解码技术): 2..8 new tokens per sequence over long
    # contexts; with G = 1 every task is decode-shaped, with G = 4 and 8 some become tiles
    rng = np.random.default_rng(40 + G)
    q = rng.integers(2, 9, size=24)
    ctx = q + rng.integers(500, 6000, size=24)
    wl = workloads.custom(q, ctx, 4 * G, 4, 128, 16, True, seed=60 + G, name="verify")
    assert_parity(run(wl))


@pytest.mark.parametrize("schedule", [0, 1, 2, 3, 4])
def test_kind_switches_in_one_launch(schedule):
    # short decode tasks (one or two 64-key stages) interleaved with chunk tiles on few CTAs, so
    # every CTA switches between the decode path and the tile path many times in one launch
    rng = np.random.default_rng(7)
    dq = np.ones(48, dtype=np.int64)
    dctx = rng.integers(20, 130, size=48)
    cq = np.full(6, 256)
    cctx = cq + rng.integers(0, 1500, size=6)
    q = np.concatenate([dq[:24], cq[:3], dq[24:], cq[3:]])
    ctx = np.concatenate([dctx[:24], cctx[:3], dctx[24:], cctx[3:]])
    wl = workloads.custom(q, ctx, 16, 4, 128, 16, True, seed=71, name="switches")
    assert_parity(run(wl, num_ctas=5, kv_chunk=512, schedule=schedule))


def test_sharp_score_growth_across_tiles():
    # K pages scaled by powers of two in random page order (and the new tokens' K by the largest),
    # so a row's max jumps by far more than 2^24 between KV tiles: the tile softmax must raise its
    # reference and rescale P, l and O on the fly; outputs are nearly one-hot and must still match
    def spiky(vals):
        g = torch.Generator().manual_seed(5)
        f = torch.tensor([1.0, 4.0, 16.0, 64.0])[torch.randint(0, 4, (vals["k_pool"].shape[0],), generator=g)]
        vals["k_pool"].mul_(f.to(vals["k_pool"].device, torch.bfloat16).view(-1, 1, 1, 1))
        vals["k_new"].mul_(64.0)

    wl = workloads.custom([300, 1, 129, 64], [1500, 2000, 700, 64], 16, 4, 128, 16, True, seed=81, name="spiky")
    assert_parity(run(wl, transform=spiky))


def test_full_size_decode_sampled():
    wl = workloads.decode()
    rng = np.random.default_rng(0)
    seqs = sorted(rng.choice(wl.num_seqs, size=6, replace=False).tolist())
    seqs.append(int(np.argmax(wl.context_lens)))
    r = run(wl, rows=sample_rows(wl, seqs, rng), sample_seqs=seqs, schedule=4)
    assert_parity(r)


def test_full_size_prefill_sampled():
    wl = workloads.prefill()
    rng = np.random.default_rng(1)
    seqs = sorted({int(np.argmax(wl.q_lens)), int(np.argmin(wl.q_lens)), int(rng.integers(wl.num_seqs))})
    r = run(wl, rows=sample_rows(wl, seqs, rng, per_seq=12, q_tile=256 // wl.group), sample_seqs=seqs, schedule=4)
    assert_parity(r)


def test_full_size_mixed_sampled():
    wl = workloads.mixed()
    rng = np.random.default_rng(2)
    seqs = [0, 5, 8, 60, 127, int(np.argmax(wl.context_lens))]
    r = run(wl, rows=sample_rows(wl, seqs, rng, per_seq=8, q_tile=256 // wl.group), sample_seqs=seqs, schedule=4)
    assert_parity(r)


def test_full_size_skew_sampled():
    # every one of the four 131072-key sequences (all 64 heads of each), and two 512-key ones
    wl = workloads.skew()
    long_seqs = [int(i) for i in np.flatnonzero(wl.context_lens == wl.context_lens.max())]
    assert len(long_seqs) == 4
    rng = np.random.default_rng(3)
    short = [int(i) for i in rng.choice(np.flatnonzero(wl.context_lens < wl.context_lens.max()), 2, replace=False)]
    seqs = sorted(long_seqs + short)
    r = run(wl, rows=sample_rows(wl, seqs, rng), sample_seqs=seqs, per_seq_oracle=True, schedule=4)
    assert_parity(r)


def test_page_index_out_of_range_sets_error_bit():
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import step as xystep
    wl = workloads.custom([1, 1], [40, 20], 4, 2, 64, 16, seed=9)
    vals = wl.tensors("cuda")
    batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                              wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal)
    batch.block_table[0, 1] = wl.num_pages + 5          # a page outside the pool, inside the context
    xystep.run_step(batch, vals["q"], vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"], wl.scale)
    torch.cuda.synchronize()
    with pytest.raises(xy.XYDeviceError) as e:
        xystep.check(batch)
    assert e.value.bits & xy.XY_DEV_PAGE_OOB
    # the context is still usable
    r = run(workloads.tiny())
    assert_parity(r)


def test_host_validation_rejects_bad_arguments():
    import paged_kv_varlen_xy_gb300 as xy
    wl = workloads.tiny()
    vals = wl.tensors("cuda")
    from paged_kv_varlen_xy_gb300 import step as xystep
    batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                              wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal)
    pl = batch.plan
    out = torch.empty_like(vals["q"])
    with pytest.raises(xy.XYError) as e:    # head_dim 48 is not supported
        q48 = torch.zeros(vals["q"].shape[0], 4, 48, dtype=torch.bfloat16, device="cuda")
        kp48 = torch.zeros(64, 2, 16, 48, dtype=torch.bfloat16, device="cuda")
        xy.xy_paged_attention(q48, batch.cu, batch.ctx, batch.block_table, kp48, kp48, 0.1, True, pl.tasks,
                              pl.merges, pl.num_ctas, pl.workspace, batch.err, torch.empty_like(q48))
    assert e.value.status == -5
    with pytest.raises(xy.XYError) as e:    # misaligned pointer
        T = vals["q"].shape[0]
        qv = vals["q"].view(-1)[1: 1 + (T - 1) * 256].view(T - 1, 4, 64)
        xy.xy_paged_attention(qv, batch.cu, batch.ctx, batch.block_table, vals["k_pool"], vals["v_pool"], 0.1,
                              True, pl.tasks, pl.merges, pl.num_ctas, pl.workspace, batch.err, torch.empty_like(qv))
    assert e.value.status == -1
    torch.cuda.synchronize()
    assert int(batch.err.item()) == 0


def test_empty_batch_launches_nothing():
    import paged_kv_varlen_xy_gb300 as xy
    dev = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kp = torch.zeros(4, 1, 16, 64, dtype=torch.bfloat16, device=dev)
    empty = torch.zeros(0, 1, 64, dtype=torch.bfloat16, device=dev)
    slots = torch.zeros(0, dtype=torch.int64, device=dev)
    xy.xy_kv_append(empty, empty, slots, kp, kp, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_fused_append_equals_slot_mapping_then_append(fp8):
    # xy_kv_append_paged(_fp8) forms each token's slot in the copy kernel; its slots and pages must
    # equal those of xy_slot_mapping followed by xy_kv_append(_fp8), and the oracle's, bit for bit
    import oracle
    import paged_kv_varlen_xy_gb300 as xy
    from gpu_cases import bits
    wl = workloads.custom([5, 1, 300, 1, 40, 7], [5, 33, 900, 4096, 57, 7], 16, 4, 128, 16, seed=91)
    vals = wl.tensors("cuda")
    bt_host, _ = xy.xy_build_block_table(wl.context_lens, wl.block_size, wl.free_list, wl.max_blocks)
    cu = torch.from_numpy(wl.cu_seqlens_q).cuda()
    ctx = torch.from_numpy(wl.context_lens).cuda()
    bt = torch.from_numpy(bt_host).cuda()
    T, P = wl.num_tokens, wl.num_pages
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = oracle.step.run_step(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                               bits(vals["q"]), bits(vals["k_new"]), bits(vals["v_new"]), bits(vals["k_pool"]),
                               bits(vals["v_pool"]), wl.scale, wl.causal, rows=[])
    results = []
    for fused in (False, True):
        slots = torch.full((T,), -7, dtype=torch.int64, device="cuda")
        if fp8:
            _, Hkv, bs, d = vals["k_pool"].shape
            pools = [torch.zeros(P, Hkv, bs, d, dtype=torch.uint8, device="cuda") for _ in range(2)]
            scl = [torch.zeros(P, Hkv, bs, dtype=torch.float32, device="cuda") for _ in range(2)]
            if fused:
                xy.xy_kv_append_paged_fp8(vals["k_new"], vals["v_new"], cu, ctx, bt, pools[0], pools[1], scl[0], scl[1],
                                          err, slot_mapping=slots)
            else:
                xy.xy_slot_mapping(cu, ctx, bt, wl.block_size, P, slots, err)
                xy.xy_kv_append_fp8(vals["k_new"], vals["v_new"], slots, pools[0], pools[1], scl[0], scl[1], err)
            pools += scl
        else:
            pools = [vals["k_pool"].clone(), vals["v_pool"].clone()]
            if fused:
                xy.xy_kv_append_paged(vals["k_new"], vals["v_new"], cu, ctx, bt, pools[0], pools[1], err,
                                      slot_mapping=slots)
            else:
                xy.xy_slot_mapping(cu, ctx, bt, wl.block_size, P, slots, err)
                xy.xy_kv_append(vals["k_new"], vals["v_new"], slots, pools[0], pools[1], err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert np.array_equal(slots.cpu().numpy(), ref["slots"])
        results.append([x.cpu() for x in pools])
    for a, b in zip(*results):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    if not fp8:
        assert np.array_equal(bits(results[1][0]), ref["k_pages"])
        assert np.array_equal(bits(results[1][1]), ref["v_pages"])


def test_fused_append_flags_a_page_outside_the_pool():
    import paged_kv_varlen_xy_gb300 as xy
    wl = workloads.custom([3, 1], [40, 20], 4, 2, 64, 16, seed=9)
    vals = wl.tensors("cuda")
    bt_host, _ = xy.xy_build_block_table(wl.context_lens, wl.block_size, wl.free_list, wl.max_blocks)
    bt_host[0, 2] = wl.num_pages + 3     # the page of sequence 0's new tokens lies outside the pool
    cu, ctx, bt = (torch.from_numpy(a).cuda() for a in (wl.cu_seqlens_q, wl.context_lens, bt_host))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.zeros(wl.num_tokens, dtype=torch.int64, device="cuda")
    before = vals["k_pool"].clone()
    xy.xy_kv_append_paged(vals["k_new"], vals["v_new"], cu, ctx, bt, vals["k_pool"], vals["v_pool"], err,
                          slot_mapping=slots)
    torch.cuda.synchronize()
    assert int(err.item()) & xy.XY_DEV_PAGE_OOB
    s = slots.cpu().numpy()
    assert (s[:3] == -1).all() and s[3] >= 0
    # only the one token with a valid slot was written
    changed = (vals["k_pool"] != before).any(dim=-1).any(dim=-1).any(dim=-1).sum().item()
    assert changed == 1


def test_full_size_verify_sampled():
    # the bench's speculative-verify batch (64 sequences of 2..8 new tokens over 512..8192 keys) in its
    # launch configuration: every row of eight sampled sequences
    wl = workloads.verify()
    rng = np.random.default_rng(6)
    seqs = sorted(rng.choice(wl.num_seqs, size=8, replace=False).tolist())
    cu = wl.cu_seqlens_q
    rows = [(t, h) for i in seqs for t in range(int(cu[i]), int(cu[i + 1])) for h in range(wl.num_heads_q)]
    r = run(wl, rows=rows, sample_seqs=seqs, schedule=4)
    assert_parity(r)


@pytest.mark.parametrize("config,launches", [("prefill", 200), ("mixed", 30), ("verify", 100)])
def test_repeated_launches_bit_identical(config, launches):
    # Each task's result does not depend on which CTA runs it or on how the warps of a CTA drift
    # against one another, so back-to-back launches of the bench's batches (dynamic deal) give
    # bit-identical outputs and raise no device error (a barrier phase overtaken by a fast warp
    # would show here as a wait that gives up, or as a wrong output).
    from paged_kv_varlen_xy_gb300 import step as xystep
    import paged_kv_varlen_xy_gb300 as xy

    wl = workloads.make(config)
    dev = torch.device("cuda")
    vals = wl.tensors(dev)
    batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                              wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, device=dev, schedule=4)
    first = xystep.run_step(batch, vals["q"], vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"], wl.scale)
    pl = batch.plan
    ref = first.view(torch.int16)
    outs = [torch.empty_like(first) for _ in range(2)]
    differ = []
    for i in range(launches):
        out = outs[i & 1]
        xy.xy_paged_attention_dynamic(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"],
                                      vals["v_pool"], wl.scale, batch.causal, pl.tasks, pl.merges, pl.num_ctas,
                                      pl.workspace, pl.task_counter, batch.err, out)
        if i % 16 == 15 and not torch.equal(out.view(torch.int16), ref):
            differ.append(i)
    torch.cuda.synchronize()
    xystep.check(batch)
    assert not differ, f"launches {differ} differ from the first"
    assert torch.equal(outs[(launches - 1) & 1].view(torch.int16), ref)


@pytest.mark.parametrize("G,kv_chunk", [(4, None), (4, 256), (8, 384), (2, None)])
def test_single_query_tile_tasks_every_row(G, kv_chunk):
    # tile tasks of at most 128 rows (one query tile, group B idle) over two or more K/V tiles:
    # whole 128-row tiles (the TMA store epilogue), partial ones, odd and even tile counts, ragged
    # ends, split partials
    rng = np.random.default_rng(90 + G)
    qt = 128 // G
    q = [qt, qt - 3, 5, qt, 9, qt // 2, qt]
    ctx = [qi + int(rng.integers(130, 1500)) for qi in q]
    ctx[0] = q[0] + 256   # an even number of 128-key tiles from the start
    ctx[3] = q[3] + 383
    wl = workloads.custom(q, ctx, 2 * G, 2, 128, 16, True, seed=70 + G, name="paired")
    assert_parity(run(wl, q_tile=qt, kv_chunk=kv_chunk, schedule=4))
    assert_parity(run(wl, q_tile=qt, kv_chunk=kv_chunk, schedule=3))


def test_single_query_tile_tasks_sharp_score_growth_and_nan_pool():
    # the lazy rescale of one-tile tasks whose row maxima jump between K/V tiles; stale NaN rows
    # past kv_end never reach the outputs
    G = 4
    q = [32, 20, 32]
    ctx = [32 + 700, 20 + 300, 32 + 1000]
    wl = workloads.custom(q, ctx, 8, 2, 128, 16, True, seed=81, name="paired_sharp")

    def grow(vals):
        # pages scaled by powers of two in random page order, as in the sharp-growth test above
        g = torch.Generator().manual_seed(6)
        f = torch.tensor([1.0, 4.0, 16.0, 64.0])[torch.randint(0, 4, (vals["k_pool"].shape[0],), generator=g)]
        vals["k_pool"].mul_(f.to(vals["k_pool"].device, torch.bfloat16).view(-1, 1, 1, 1))
        vals["k_new"].mul_(64.0)

    assert_parity(run(wl, q_tile=32, schedule=4, transform=grow))
    # the whole pool starts as NaN and every context token is appended (q = L), so only slots past
    # each context end stay NaN; 32-token query tiles past the first 96 tokens span two or more
    # K/V tiles
    wl = workloads.custom([300, 200, 150], [300, 200, 150], 8, 2, 128, 16, True, seed=82, name="paired_nan")
    assert_parity(run(wl, q_tile=32, schedule=4, pool_fill=float("nan")), check_pages=False)
