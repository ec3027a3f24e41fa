"""8-bit (E4M3) KV pages on the GPU against the oracle: the quantizing append bit for bit, and
attention over the 8-bit pages against the oracle's attention over the dequantized pages."""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("d", [64, 128])
def test_append_fp8_bit_exact(d):
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import build
    build.build()
    rng = np.random.default_rng(d)
    P, Hkv, bs, T = 37, 4, 16, 300
    g = torch.Generator().manual_seed(d)
    scale = torch.tensor([1e-3, 1.0, 40.0])[torch.randint(0, 3, (T, Hkv, 1), generator=g)]
    k_new = (torch.randn(T, Hkv, d, generator=g) * scale).to(torch.bfloat16)
    v_new = (torch.randn(T, Hkv, d, generator=g) * scale).to(torch.bfloat16)
    k_new[5, 1] = 0                                    # an all-zero row
    slots = rng.permutation(P * bs)[:T].astype(np.int64)
    slots[7] = -1
    kp = torch.randint(0, 256, (P, Hkv, bs, d), generator=g, dtype=torch.uint8)
    vp = torch.randint(0, 256, (P, Hkv, bs, d), generator=g, dtype=torch.uint8)
    ks = torch.rand(P, Hkv, bs, generator=g)
    vs = torch.rand(P, Hkv, bs, generator=g)
    ref = oracle.kv_append_fp8(kp.numpy(), vp.numpy(), ks.numpy(), vs.numpy(), _bits(k_new), _bits(v_new), slots)
    dev = [t.cuda() for t in (k_new, v_new, kp, vp, ks, vs)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xy.xy_kv_append_fp8(dev[0], dev[1], torch.from_numpy(slots).cuda(), dev[2], dev[3], dev[4], dev[5], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(dev[2].cpu().numpy(), ref[0]) and np.array_equal(dev[3].cpu().numpy(), ref[1])
    assert np.array_equal(dev[4].cpu().numpy().view(np.uint32), ref[2].view(np.uint32))
    assert np.array_equal(dev[5].cpu().numpy().view(np.uint32), ref[3].view(np.uint32))


# ---------------------------------------------------------------------------------------------
# attention over 8-bit pages

# the task-table deals over 8-bit pages: greedy static and dynamic (the default)
GREEDY, DYN = 3, 4


def _run_fp8(wl, kv_chunk=None, row_scale=None, split=False, schedule=None, num_ctas=None, layout="separate"):
    """One step over 8-bit pages on the GPU and in the oracle, on workload wl's bf16 values
    (optionally with each pool / new row multiplied by a power of two from row_scale).
    layout: the code pools as two allocations ("separate"), as one allocation with V after K
    ("one": the attention fetches a page's K and V codes with one 3-D copy), or as one allocation
    with V before K ("v_first": two copies per page)."""
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import build
    from paged_kv_varlen_xy_gb300 import step as xystep
    build.build()
    dev = torch.device("cuda")
    vals = wl.tensors("cpu")
    if row_scale is not None:
        g = torch.Generator().manual_seed(wl.seed)
        for name in ("k_pool", "v_pool", "k_new", "v_new"):
            shp = vals[name].shape[:-1] + (1,)
            f = torch.tensor(row_scale, dtype=torch.float32)[torch.randint(0, len(row_scale), shp, generator=g)]
            vals[name] = (vals[name].float() * f).to(torch.bfloat16)
    P, Hkv, bs, d = vals["k_pool"].shape
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if layout == "separate":
        codes = {n: torch.zeros(P, Hkv, bs, d, dtype=torch.uint8, device=dev) for n in ("k", "v")}
    else:
        both = torch.zeros(2, P, Hkv, bs, d, dtype=torch.uint8, device=dev)
        codes = {"k": both[0], "v": both[1]} if layout == "one" else {"k": both[1], "v": both[0]}
    scl = {n: torch.zeros(P, Hkv, bs, dtype=torch.float32, device=dev) for n in ("k", "v")}
    slots_all = torch.arange(P * bs, dtype=torch.int64, device=dev)
    krows = vals["k_pool"].permute(0, 2, 1, 3).reshape(P * bs, Hkv, d).contiguous().to(dev)
    vrows = vals["v_pool"].permute(0, 2, 1, 3).reshape(P * bs, Hkv, d).contiguous().to(dev)
    xy.xy_kv_append_fp8(krows, vrows, slots_all, codes["k"], codes["v"], scl["k"], scl["v"], err)
    q, kn, vn = (vals[n].to(dev) for n in ("q", "k_new", "v_new"))
    if split:
        batch = xystep.Fp8SplitBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                                     wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, device=dev)
        out = xystep.run_step_fp8_split(batch, q, kn, vn, codes["k"], codes["v"], scl["k"], scl["v"], wl.scale)
    else:
        batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                                  wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, device=dev,
                                  kv_chunk=kv_chunk, kv_fp8=True, schedule=schedule, num_ctas=num_ctas)
        out = xystep.run_step_fp8(batch, q, kn, vn, codes["k"], codes["v"], scl["k"], scl["v"], wl.scale)
    torch.cuda.synchronize()
    ref = oracle.step.run_step_fp8(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                                   _bits(vals["q"]), _bits(vals["k_new"]), _bits(vals["v_new"]),
                                   _bits(vals["k_pool"]), _bits(vals["v_pool"]), wl.scale, wl.causal)
    return dict(err=int(err.item()) | int(batch.err.item()), batch=batch, out=oracle.bf16_bits_to_f64(_bits(out)),
                ref=ref, codes={n: c.cpu().numpy() for n, c in codes.items()},
                scales={n: s.cpu().numpy() for n, s in scl.items()})


def _assert_fp8_parity(r, per_row_scale=False):
    """Bit-exact slots, codes and scales; outputs within the bf16 tolerance (with per_row_scale,
    relative to each output row's largest magnitude when that exceeds 1: bf16 rounds relatively)."""
    from gpu_cases import MAX_ABS, MEAN_ABS
    assert r["err"] == 0, f"device error word {r['err']:#x}"
    assert np.array_equal(r["batch"].slots.cpu().numpy(), r["ref"]["slots"])
    assert np.array_equal(r["codes"]["k"], r["ref"]["k_codes"]) and np.array_equal(r["codes"]["v"], r["ref"]["v_codes"])
    assert np.array_equal(r["scales"]["k"].view(np.uint32), r["ref"]["k_scales"].view(np.uint32))
    assert np.array_equal(r["scales"]["v"].view(np.uint32), r["ref"]["v_scales"].view(np.uint32))
    assert np.isfinite(r["out"]).all()
    diff = np.abs(r["out"] - r["ref"]["out"])
    if per_row_scale:
        diff = diff / np.maximum(1.0, np.abs(r["ref"]["out"]).max(axis=-1, keepdims=True))
    assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS, (diff.max(), diff.mean())


@pytest.mark.parametrize("schedule", [GREEDY, DYN])
@pytest.mark.parametrize("G,bs", [(1, 16), (4, 16), (8, 64), (16, 256)])
def test_fp8_decode_matches_oracle(G, bs, schedule):
    # decode rows over ragged contexts (1 key, partial pages, partial 64-key stages, several chunks)
    ctx = [1, 15, 16, 17, 63, 64, 65, 200, 1000, 2500, 777, 4096]
    wl = workloads.custom(np.ones(len(ctx)), ctx, 4 * G, 4, 128, bs, seed=40 + G, name="fp8_decode")
    r = _run_fp8(wl, schedule=schedule)
    assert r["batch"].plan.dynamic == (schedule == DYN)
    _assert_fp8_parity(r)


@pytest.mark.parametrize("schedule", [GREEDY, DYN])
@pytest.mark.parametrize("G", [1, 4, 8, 32])
def test_fp8_mixed_batch_matches_oracle(G, schedule):
    # prefill, chunked-prefill and verify-shaped queries (causal): tasks of up to 64 rows (up to
    # four 16-row groups) on the ring for batches that are not pure decode
    q_lens = [37, 1, 5, 100, 1, 16, 3]
    ctx = [37, 900, 64, 612, 129, 16, 2050]
    wl = workloads.custom(q_lens, ctx, 2 * G, 2, 128, 16, seed=50 + G, name="fp8_mixed")
    _assert_fp8_parity(_run_fp8(wl, schedule=schedule))


@pytest.mark.parametrize("schedule", [GREEDY, DYN])
def test_fp8_split_kv_and_row_magnitudes(schedule):
    # KV chunks of 256 keys (split partials and the combine) and rows of very different magnitude
    # (the largest V scale grows along a task: O is rescaled as it does)
    ctx = [3000, 1, 700, 5000, 257]
    wl = workloads.custom(np.ones(len(ctx)), ctx, 32, 8, 128, 16, seed=61, name="fp8_split")
    _assert_fp8_parity(_run_fp8(wl, kv_chunk=256, row_scale=[2.0 ** -12, 1.0, 2.0 ** 4], schedule=schedule),
                       per_row_scale=True)


@pytest.mark.parametrize("schedule", [GREEDY, DYN])
@pytest.mark.parametrize("name", ["decode", "skew"])
def test_fp8_full_size_sampled_rows(name, schedule):
    # the full decode / skew batches over 8-bit pages in the bench's launch configuration; the oracle
    # checks sampled sequences (all their rows), pages and codes of those sequences bit for bit
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import build
    from paged_kv_varlen_xy_gb300 import step as xystep
    from gpu_cases import MAX_ABS, MEAN_ABS
    build.build()
    wl = workloads.make(name)
    vals = wl.tensors("cuda")
    P, Hkv, bs, d = vals["k_pool"].shape
    codes = [torch.empty(P, Hkv, bs, d, dtype=torch.uint8, device="cuda") for _ in range(2)]
    scl = [torch.empty(P, Hkv, bs, dtype=torch.float32, device="cuda") for _ in range(2)]
    batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                              wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, kv_fp8=True,
                              schedule=schedule)
    rows = [vals[n].permute(0, 2, 1, 3).reshape(P * bs, Hkv, d).contiguous() for n in ("k_pool", "v_pool")]
    xy.xy_kv_append_fp8(rows[0], rows[1], torch.arange(P * bs, dtype=torch.int64, device="cuda"), codes[0], codes[1],
                        scl[0], scl[1], batch.err)
    del rows
    out = xystep.run_step_fp8(batch, vals["q"], vals["k_new"], vals["v_new"], codes[0], codes[1], scl[0], scl[1],
                              wl.scale)
    torch.cuda.synchronize()
    xystep.check(batch)
    # sampled sequences; under the dynamic deal (the bench's launch) the skew sample also holds one of
    # the 131072-key sequences: its 16 split chunks per tile, their merge and, on this pure decode
    # batch with G = 8, the two-CTA-per-SM kernel (the oracle quantizes its 512 pages, about two
    # minutes of host time, so the greedy-deal run keeps to the short ones)
    rng = np.random.default_rng(7)
    ok_seqs = [i for i in range(wl.num_seqs) if wl.context_lens[i] <= 8192]
    sample = sorted(rng.choice(ok_seqs, size=min(6, len(ok_seqs)), replace=False).tolist())
    if name == "skew" and schedule == DYN:
        sample = sorted(sample[:5] + [int(np.argmax(wl.context_lens))])
    bt = batch.block_table_host
    pages = np.unique(np.concatenate([bt[i][bt[i] >= 0] for i in sample]))
    idx = torch.from_numpy(pages).long().cuda()
    cu = wl.cu_seqlens_q
    rows = [(t, h) for i in sample for t in range(int(cu[i]), int(cu[i + 1])) for h in range(wl.num_heads_q)]
    ref = oracle.step.run_step_fp8(cu, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                                   _bits(vals["q"]), _bits(vals["k_new"]), _bits(vals["v_new"]),
                                   _bits(vals["k_pool"].index_select(0, idx)), _bits(vals["v_pool"].index_select(0, idx)),
                                   wl.scale, wl.causal, pool_pages=pages, rows=rows)
    assert np.array_equal(codes[0].index_select(0, idx).cpu().numpy(), ref["k_codes"])
    assert np.array_equal(codes[1].index_select(0, idx).cpu().numpy(), ref["v_codes"])
    assert np.array_equal(scl[0].index_select(0, idx).cpu().numpy().view(np.uint32), ref["k_scales"].view(np.uint32))
    assert np.array_equal(scl[1].index_select(0, idx).cpu().numpy().view(np.uint32), ref["v_scales"].view(np.uint32))
    got = oracle.bf16_bits_to_f64(_bits(out))
    got = np.stack([got[t, h] for (t, h) in rows])
    diff = np.abs(got - ref["out"])
    assert np.isfinite(got).all() and diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS, (diff.max(), diff.mean())


@pytest.mark.parametrize("decode", [True, False])
def test_fp8_dynamic_deal_bit_identical_and_counter_reused(decode):
    # a task's result does not depend on the CTA that runs it: the dynamic deal's outputs equal the
    # greedy deal's bit for bit (same tasks, same split rows); every launch returns the counter to
    # zero, so repeated launches need no reset; one CTA and more CTAs than tasks run every task
    import paged_kv_varlen_xy_gb300 as xy
    rng = np.random.default_rng(23)
    ctx = [int(x) for x in rng.integers(1, 3000, size=50)]
    q_lens = [1] * 50 if decode else [int(x) for x in rng.integers(1, 40, size=50)]
    wl = workloads.custom(q_lens, ctx, 16, 2, 128, 16, seed=24, name="fp8_dyn")
    outs = {}
    for schedule, n in ((GREEDY, None), (DYN, None), (DYN, 1), (DYN, 300)):
        r = _run_fp8(wl, kv_chunk=512, schedule=schedule, num_ctas=n)
        _assert_fp8_parity(r)
        outs[(schedule, n)] = r
    base = _bits_f64(outs[(GREEDY, None)]["out"])
    for key, r in outs.items():
        assert np.array_equal(_bits_f64(r["out"]), base), key
    r = outs[(DYN, None)]
    batch, pl = r["batch"], r["batch"].plan
    assert len(pl.host["merges"]) > 0, "expected split tasks"
    assert pl.task_counter.cpu().tolist() == [0, 0]
    q = wl.tensors("cpu")["q"].cuda()  # the values _run_fp8 used
    k, v = (torch.from_numpy(r["codes"][n]).cuda() for n in ("k", "v"))
    ks, vs = (torch.from_numpy(r["scales"][n]).cuda() for n in ("k", "v"))
    for _ in range(3):
        out = torch.empty_like(q)
        xy.xy_paged_attention_fp8_dynamic(q, batch.cu, batch.ctx, batch.block_table, k, v, ks, vs, wl.scale,
                                          wl.causal, pl.tasks, pl.merges, pl.num_ctas, pl.workspace,
                                          pl.task_counter, batch.err, out)
        torch.cuda.synchronize()
        assert int(batch.err.item()) == 0
        assert pl.task_counter.cpu().tolist() == [0, 0]
        assert np.array_equal(_bits(out), base)


def test_fp8_greedy_table_with_holes_through_the_dynamic_call():
    # hole records of a greedy table are skipped by the claiming CTAs: every task runs once
    import paged_kv_varlen_xy_gb300 as xy
    wl = workloads.custom([1] * 6, [5000, 30, 30, 30, 900, 17], 8, 2, 128, 16, seed=19, name="fp8_holes")
    r = _run_fp8(wl, kv_chunk=1024, schedule=GREEDY, num_ctas=5)
    _assert_fp8_parity(r)
    batch, pl = r["batch"], r["batch"].plan
    assert (pl.host["tasks"][:, 0] == -1).any(), "expected hole records"
    q = wl.tensors("cpu")["q"].cuda()  # the values _run_fp8 used
    k, v = (torch.from_numpy(r["codes"][n]).cuda() for n in ("k", "v"))
    ks, vs = (torch.from_numpy(r["scales"][n]).cuda() for n in ("k", "v"))
    counter = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    xy.xy_paged_attention_fp8_dynamic(q, batch.cu, batch.ctx, batch.block_table, k, v, ks, vs, wl.scale, wl.causal,
                                      pl.tasks, pl.merges, pl.num_ctas, pl.workspace, counter, batch.err, out)
    torch.cuda.synchronize()
    assert int(batch.err.item()) == 0 and counter.cpu().tolist() == [0, 0]
    assert np.array_equal(_bits(out), _bits_f64(r["out"]))


def _bits_f64(x):
    """bf16 values held as float64 (exactly) -> their bf16 bit patterns."""
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_dequant_pages_bit_exact():
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import build
    build.build()
    g = torch.Generator().manual_seed(3)
    P, Hkv, bs, d = 40, 4, 16, 128
    codes = [torch.randint(0, 256, (P, Hkv, bs, d), generator=g, dtype=torch.uint8) for _ in range(2)]
    for c in codes:
        c[(c & 0x7F) == 0x7F] = 0                                   # no NaN codes
    scl = [torch.rand(P, Hkv, bs, generator=g) * 4 for _ in range(2)]
    pages = torch.tensor([7, 0, 39, 7, 12], dtype=torch.int32)
    outs = [torch.empty(5, Hkv, bs, d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = [t.cuda() for t in codes + scl]
    xy.xy_dequant_pages_fp8(dev[0], dev[1], dev[2], dev[3], pages.cuda(), outs[0], outs[1], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for n in range(2):
        ref = oracle.dequantize_to_bf16_bits(codes[n].numpy()[pages.numpy()], scl[n].numpy()[pages.numpy()])
        assert np.array_equal(_bits(outs[n]), ref)


@pytest.mark.parametrize("q_lens,ctx", [([37, 100, 5, 1, 1, 1], [37, 612, 2050, 900, 129, 16]),
                                         ([1, 1, 1, 64, 3], [700, 33, 4000, 300, 1500]),
                                         ([200, 17], [200, 5000])])
def test_fp8_split_tile_and_decode_parts(q_lens, ctx):
    # prefill / chunk sequences on the tile path over bf16 copies, decode sequences on the 8-bit
    # path, in one step; against the oracle's attention over the exactly dequantized pages
    from paged_kv_varlen_xy_gb300 import build
    from paged_kv_varlen_xy_gb300 import step as xystep
    build.build()
    wl = workloads.custom(q_lens, ctx, 16, 4, 128, 16, True, seed=71)
    r = _run_fp8(wl, split=True)
    _assert_fp8_parity(r)


@pytest.mark.parametrize("layout", ["one", "v_first"])
@pytest.mark.parametrize("config", ["decode16", "decode256", "verify"])
def test_code_pools_in_one_allocation(layout, config):
    # K and V code pools in one allocation: V after K (one 3-D copy per page brings both) or V
    # before K (a copy per page and pool), over 16- and 256-token pages, one-token and multi-token
    # sequences (the tiny two-CTA kernel and the wide decode path)
    rng = np.random.default_rng(11)
    if config == "verify":
        q = rng.integers(2, 9, size=12)
        wl = workloads.custom(q, q + rng.integers(100, 3000, size=12), 16, 4, 128, 16, True, seed=12, name="v1")
    else:
        bs = 16 if config == "decode16" else 256
        wl = workloads.custom(np.ones(20, dtype=np.int64), rng.integers(50, 3000, size=20), 16, 4, 128, bs, True,
                              seed=13, name="d1")
    _assert_fp8_parity(_run_fp8(wl, layout=layout, schedule=4))
    _assert_fp8_parity(_run_fp8(wl, layout=layout, kv_chunk=256, schedule=3))
