"""The packed-upload Planner gives the same tables and the same step results as PagedBatch, across
batches of different sizes planned with one Planner (buffers reused and grown), and when the deal
needs more records than the size bound allowed for."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import MAX_ABS, MEAN_ABS, bits

pytestmark = pytest.mark.gpu


def _step_both(planner, wl, vals):
    from paged_kv_varlen_xy_gb300 import step as xystep
    outs = []
    pools = []
    for use_planner in (False, True):
        kp, vp = vals["k_pool"].clone(), vals["v_pool"].clone()
        if use_planner:
            b = planner.plan(wl.cu_seqlens_q, wl.context_lens, wl.free_list)
        else:
            b = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                                  wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, num_ctas=planner.num_ctas)
        if use_planner:
            out = planner.run(b, vals["q"], vals["k_new"], vals["v_new"], kp, vp, wl.scale)
        else:
            out = xystep.run_step(b, vals["q"], vals["k_new"], vals["v_new"], kp, vp, wl.scale)
        torch.cuda.synchronize()
        xystep.check(b)
        outs.append((b, out))
        pools.append((kp, vp))
    (b0, o0), (b1, o1) = outs
    assert np.array_equal(b0.block_table_host, b1.block_table_host)
    assert np.array_equal(b0.block_table.cpu().numpy(), b1.block_table.cpu().numpy())
    assert np.array_equal(b0.plan.tasks.cpu().numpy(), b1.plan.tasks.cpu().numpy())
    assert np.array_equal(b0.plan.merges.cpu().numpy(), b1.plan.merges.cpu().numpy())
    assert np.array_equal(b0.slots.cpu().numpy(), b1.slots.cpu().numpy())
    assert torch.equal(pools[0][0], pools[1][0]) and torch.equal(pools[0][1], pools[1][1])
    assert np.array_equal(bits(o0), bits(o1))   # same kernels, same inputs
    return b1, o1


def test_planner_matches_pagedbatch_across_batches():
    from paged_kv_varlen_xy_gb300 import build
    from paged_kv_varlen_xy_gb300 import step as xystep
    build.build()
    planner = xystep.Planner(16, 4, 128, 16, 512, True)
    # small, larger (buffers grow), small again (buffers reused)
    for q, L, seed in (([3, 1, 1], [40, 300, 17], 1), ([1] * 40 + [64, 100], list(range(100, 4100, 100)) + [900, 2000], 2),
                       ([5, 1], [5, 1000], 3)):
        wl = workloads.custom(q, L, 16, 4, 128, 16, True, seed=seed)
        wl.max_blocks = 512
        vals = wl.tensors("cuda")
        k0, v0 = bits(vals["k_pool"]), bits(vals["v_pool"])
        b, out = _step_both(planner, wl, vals)
        if seed != 2:  # all rows of the small batches against the oracle
            ref = oracle.step.run_step(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                                       bits(vals["q"]), bits(vals["k_new"]), bits(vals["v_new"]), k0, v0, wl.scale,
                                       wl.causal)
            diff = np.abs(oracle.bf16_bits_to_f64(bits(out)) - ref["out"])
            assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS


def test_planner_grows_its_buffers_on_the_first_batch():
    from paged_kv_varlen_xy_gb300 import build
    from paged_kv_varlen_xy_gb300 import step as xystep
    build.build()
    # 300 sequences x 64 block-table columns = 76.8 KB of block table: more than the first
    # staging buffer holds, so plan() grows it and builds again
    planner = xystep.Planner(8, 2, 128, 16, 64, True, num_ctas=7)
    rng = np.random.default_rng(3)
    ctx = rng.integers(1, 1000, size=300)
    wl = workloads.custom(np.ones(300), ctx, 8, 2, 128, 16, True, seed=5)
    wl.max_blocks = 64
    _step_both(planner, wl, wl.tensors("cuda"))


def test_planner_fp8_run_matches_run_step_fp8():
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import build
    from paged_kv_varlen_xy_gb300 import step as xystep
    build.build()
    wl = workloads.custom([1, 1, 9, 1], [700, 40, 300, 2000], 16, 4, 128, 16, True, seed=9)
    vals = wl.tensors("cuda")
    P, Hkv, bs, d = vals["k_pool"].shape
    res = []
    for use_planner in (False, True):
        codes = [torch.zeros(P, Hkv, bs, d, dtype=torch.uint8, device="cuda") for _ in range(2)]
        scl = [torch.zeros(P, Hkv, bs, dtype=torch.float32, device="cuda") for _ in range(2)]
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        rows = [vals[n].permute(0, 2, 1, 3).reshape(P * bs, Hkv, d).contiguous() for n in ("k_pool", "v_pool")]
        xy.xy_kv_append_fp8(rows[0], rows[1], torch.arange(P * bs, dtype=torch.int64, device="cuda"), codes[0],
                            codes[1], scl[0], scl[1], err)
        if use_planner:
            planner = xystep.Planner(16, 4, 128, 16, wl.max_blocks, True, kv_fp8=True, kv_chunk=256)
            b = planner.plan(wl.cu_seqlens_q, wl.context_lens, wl.free_list)
            out = planner.run(b, vals["q"], vals["k_new"], vals["v_new"], codes[0], codes[1], wl.scale,
                              k_scales=scl[0], v_scales=scl[1])
        else:
            b = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks, 16, 4,
                                  128, True, kv_fp8=True, kv_chunk=256)
            out = xystep.run_step_fp8(b, vals["q"], vals["k_new"], vals["v_new"], codes[0], codes[1], scl[0], scl[1],
                                      wl.scale)
        torch.cuda.synchronize()
        xystep.check(b)
        assert int(err.item()) == 0
        res.append((bits(out), codes[0].cpu(), scl[1].cpu()))
    assert np.array_equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1]) and torch.equal(res[0][2], res[1][2])


def test_split_planner_matches_fp8_split_batch_across_batches():
    # over 8-bit pages: the packed-upload split planner gives the tables and the outputs of
    # Fp8SplitBatch, bit for bit, for batches of different sizes planned by one planner
    from paged_kv_varlen_xy_gb300 import step as xystep
    import paged_kv_varlen_xy_gb300 as xy
    dev = torch.device("cuda")
    shapes = [([40, 1, 1], [300, 700, 33]), ([300, 17, 1, 1, 1, 1], [900, 3000, 40, 9000, 1, 64]),
              ([64, 1], [64, 5])]
    MB = 600  # one block-table width for every batch of the planner (>= 9000 / 16)
    planner = xystep.Fp8SplitPlanner(8, 2, 128, 16, MB, True, device=dev, num_ctas=37)
    for k, (ql, cl) in enumerate(shapes):
        wl = workloads.custom(ql, cl, 8, 2, 128, 16, True, seed=200 + k, name="split")
        vals = wl.tensors(dev)
        P, Hkv, bs, d = vals["k_pool"].shape
        codes = [torch.zeros(P, Hkv, bs, d, dtype=torch.uint8, device=dev) for _ in range(2)]
        scales = [torch.zeros(P, Hkv, bs, dtype=torch.float32, device=dev) for _ in range(2)]
        rows = [vals[n].permute(0, 2, 1, 3).reshape(P * bs, Hkv, d).contiguous() for n in ("k_pool", "v_pool")]
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        xy.xy_kv_append_fp8(rows[0], rows[1], torch.arange(P * bs, dtype=torch.int64, device=dev), codes[0],
                            codes[1], scales[0], scales[1], err)
        outs, batches = [], []
        for use_planner in (False, True):
            cc = [c.clone() for c in codes]
            ss = [x.clone() for x in scales]
            if use_planner:
                b = planner.plan(wl.cu_seqlens_q, wl.context_lens, wl.free_list)
            else:
                b = xystep.Fp8SplitBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, MB,
                                         wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, device=dev,
                                         num_ctas=37)
            out = xystep.run_step_fp8_split(b, vals["q"], vals["k_new"], vals["v_new"], cc[0], cc[1], ss[0], ss[1],
                                            wl.scale)
            torch.cuda.synchronize()
            xystep.check(b)
            outs.append(bits(out))
            batches.append(b)
        b0, b1 = batches
        assert np.array_equal(b0.block_table.cpu().numpy(), b1.block_table.cpu().numpy())
        for part in ("tile", "decode"):
            p0, p1 = getattr(b0, part), getattr(b1, part)
            assert (p0 is None) == (p1 is None)
            if p0 is not None:
                assert np.array_equal(p0["plan"].tasks.cpu().numpy(), p1["plan"].tasks.cpu().numpy())
                assert np.array_equal(p0["plan"].merges.cpu().numpy(), p1["plan"].merges.cpu().numpy())
        assert np.array_equal(outs[0], outs[1])
        ref = oracle.step.run_step_fp8(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, MB,
                                       bits(vals["q"]), bits(vals["k_new"]), bits(vals["v_new"]), bits(vals["k_pool"]),
                                       bits(vals["v_pool"]), wl.scale, wl.causal)
        diff = np.abs(oracle.bf16_bits_to_f64(outs[1]) - ref["out"])
        assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS
