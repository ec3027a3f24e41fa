"""GPU parity of the dynamic deal (XY_SCHEDULE_DYNAMIC tables run by xy_paged_attention_dynamic:
persistent CTAs claim tasks in table order from a device counter while the kernel runs, on the
unified tcgen05 kernel or the decode-path kernel, whichever the static call would launch).

The attention outputs are compared with the oracle as in the static-deal tests; besides, a task's
result does not depend on which CTA runs it, so the dynamic and static deals of the same tasks
give outputs identical bit for bit."""

import numpy as np
import pytest
import torch

import workloads
from gpu_cases import assert_parity, bits, run, sample_rows

pytestmark = pytest.mark.gpu

DYN = 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_varlen_xy_gb300 import build
    build.build()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [16, 256])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_batch_every_row(d, bs, causal):
    wl = workloads.custom([1, 17, 130, 77, 40, 1], [1, 40, 130, 500, 333, 700], 8, 2, d, bs, causal=causal,
                          seed=300 + d + bs + int(causal))
    r = run(wl, schedule=DYN)
    assert r["batch"].plan.dynamic
    assert_parity(r)


@pytest.mark.parametrize("kv_chunk", [128, 256, 384])
def test_split_kv_and_combine_every_row(kv_chunk):
    wl = workloads.custom([3, 1, 50, 1], [700, 520, 190, 64], 8, 2, 128, 16, seed=kv_chunk + 7)
    r = run(wl, kv_chunk=kv_chunk, schedule=DYN)
    assert len(r["batch"].plan.host["merges"]) > 0
    assert_parity(r)


@pytest.mark.parametrize("G", [1, 2, 8, 16])
def test_gqa_groups(G):
    wl = workloads.custom([1, 5, 33, 2], [90, 5, 70, 130], 2 * G, 2, 128, 16, seed=40 + G)
    assert_parity(run(wl, schedule=DYN))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 4, 16])
@pytest.mark.parametrize("bs", [16, 256])
def test_pure_decode_half_size_ctas(d, G, bs):
    # one new token per sequence under the dynamic deal: the half-size decode-path CTAs, two per SM
    # slot (G <= 16 rows per task); 256-key chunks split the longer contexts into partials + combine
    ctx = [1, 17, 300, 64, 1000, 2049, 5, 130, 777]
    wl = workloads.custom([1] * len(ctx), ctx, 2 * G, 2, d, bs, seed=500 + d + G + bs)
    r = run(wl, kv_chunk=256, schedule=DYN)
    assert len(r["batch"].plan.host["merges"]) > 0
    assert_parity(r)

    def nan_outside_contexts(vals):
        # every slot no context token occupies (the rest of each last page, unused pages) is NaN;
        # the page boxes bring whole pages, so this checks that those slots never reach an output
        import oracle
        bt = oracle.allocate_block_table(wl.context_lens, wl.block_size, wl.free_list, wl.max_blocks)
        unused = torch.ones(wl.num_pages, wl.block_size, dtype=torch.bool)
        for i, L in enumerate(wl.context_lens.tolist()):
            for b in range(-(-L // wl.block_size)):
                unused[int(bt[i][b]), :min(wl.block_size, L - b * wl.block_size)] = False
        m = unused.to(vals["k_pool"].device).view(wl.num_pages, 1, wl.block_size, 1)
        for k in ("k_pool", "v_pool"):
            vals[k].masked_fill_(m, float("nan"))

    assert_parity(run(wl, kv_chunk=256, schedule=DYN, transform=nan_outside_contexts))


def test_more_ctas_than_tasks_and_one_cta():
    # 300 CTAs for a handful of tasks: most claim the end of the table at once; one CTA runs all
    wl = workloads.custom([1, 9, 1, 100], [300, 9, 20, 130], 8, 4, 64, 16, seed=15)
    for n in (1, 3, 300):
        assert_parity(run(wl, num_ctas=n, schedule=DYN))


@pytest.mark.parametrize("mixed", [False, True])
def test_counter_returns_to_zero_and_is_reused(mixed):
    # every launch leaves the claim counter at zero, so back-to-back launches need no reset
    import paged_kv_varlen_xy_gb300 as xy
    q_lens = [1, 40, 1, 200, 1] if mixed else [1] * 5
    wl = workloads.custom(q_lens, [3000, 40, 700, 300, 64], 8, 2, 128, 16, seed=16)
    r = run(wl, num_ctas=37, kv_chunk=512, schedule=DYN)
    assert_parity(r)
    pl = r["batch"].plan
    assert pl.task_counter.cpu().tolist() == [0, 0]
    vals = wl.tensors(torch.device("cuda"))
    batch = r["batch"]
    first = None
    for _ in range(3):
        out = torch.empty_like(vals["q"])
        xy.xy_paged_attention_dynamic(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"],
                                      vals["v_pool"], wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas,
                                      pl.workspace, pl.task_counter, batch.err, out)
        torch.cuda.synchronize()
        assert int(batch.err.item()) == 0
        assert pl.task_counter.cpu().tolist() == [0, 0]
        first = bits(out) if first is None else first
        assert np.array_equal(bits(out), first)


@pytest.mark.parametrize("mixed", [False, True])
def test_bit_identical_to_static_deal(mixed):
    rng = np.random.default_rng(5)
    ctx = [int(x) for x in rng.integers(300, 3000, size=40)]
    q_lens = [int(x) for x in rng.integers(1, 200, size=40)] if mixed else [1] * 40
    wl = workloads.custom(q_lens, ctx, 16, 2, 128, 16, seed=17)
    outs = []
    for schedule in (3, DYN):
        vals = wl.tensors(torch.device("cuda"))
        from paged_kv_varlen_xy_gb300 import step as xystep
        batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                                  wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, kv_chunk=1024,
                                  schedule=schedule)
        out = xystep.run_step(batch, vals["q"], vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"],
                              wl.scale)
        torch.cuda.synchronize()
        xystep.check(batch)
        outs.append(bits(out))
    assert np.array_equal(outs[0], outs[1])


def test_static_table_with_holes_through_the_dynamic_call():
    # a greedy table (hole records) run by the dynamic call: holes are skipped, every task once
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import step as xystep
    wl = workloads.custom([1, 1, 1, 1, 1, 1], [5000, 30, 30, 30, 900, 17], 8, 2, 128, 16, seed=18)
    r_ref = run(wl, kv_chunk=1024, num_ctas=5, schedule=3)
    assert_parity(r_ref)
    assert (r_ref["batch"].plan.host["tasks"][:, 0] == -1).any(), "expected hole records"
    dev = torch.device("cuda")
    vals = wl.tensors(dev)
    batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                              wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, num_ctas=5, kv_chunk=1024,
                              schedule=3)
    P = wl.num_pages
    xy.xy_slot_mapping(batch.cu, batch.ctx, batch.block_table, wl.block_size, P, batch.slots, batch.err)
    xy.xy_kv_append(vals["k_new"], vals["v_new"], batch.slots, vals["k_pool"], vals["v_pool"], batch.err)
    out = torch.empty_like(vals["q"])
    counter = torch.zeros(2, dtype=torch.int32, device=dev)
    pl = batch.plan
    xy.xy_paged_attention_dynamic(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"], vals["v_pool"],
                                  wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas, pl.workspace, counter,
                                  batch.err, out)
    torch.cuda.synchronize()
    xystep.check(batch)
    # the static call ran the same kernel on the same tasks
    import oracle
    got = oracle.bf16_bits_to_f64(bits(out))
    assert np.array_equal(got, r_ref["gpu_out"])
    assert np.abs(got - r_ref["ref"]["out"]).max() <= 2e-2


@pytest.mark.parametrize("G", [1, 4, 8])
def test_verify_shaped_queries(G):
    # speculative-verify batches: 2..8 new tokens per sequence over long contexts
    rng = np.random.default_rng(80 + G)
    q = rng.integers(2, 9, size=24)
    ctx = q + rng.integers(500, 6000, size=24)
    wl = workloads.custom(q, ctx, 4 * G, 4, 128, 16, True, seed=90 + G, name="verify")
    assert_parity(run(wl, schedule=DYN))


def test_nan_in_unused_slots_never_reaches_outputs():
    wl = workloads.custom([5, 37, 64, 70], [5, 37, 64, 70], 4, 2, 128, 16, seed=33)
    assert_parity(run(wl, pool_fill=float("nan"), schedule=DYN), check_pages=False)
    assert_parity(run(wl, pool_fill=float("nan"), kv_chunk=128, schedule=DYN), check_pages=False)


def test_full_size_decode_sampled():
    wl = workloads.decode()
    rng = np.random.default_rng(10)
    seqs = sorted(rng.choice(wl.num_seqs, size=6, replace=False).tolist())
    seqs.append(int(np.argmax(wl.context_lens)))
    assert_parity(run(wl, rows=sample_rows(wl, seqs, rng), sample_seqs=seqs, schedule=DYN))


def test_full_size_skew_sampled():
    wl = workloads.skew()
    seqs = [int(np.argmax(wl.context_lens)), int(np.argmin(wl.context_lens))]
    rng = np.random.default_rng(13)
    assert_parity(run(wl, rows=sample_rows(wl, seqs, rng), sample_seqs=seqs, schedule=DYN))


def test_full_size_mixed_sampled():
    wl = workloads.mixed()
    rng = np.random.default_rng(12)
    seqs = [0, 5, 8, 60, 127, int(np.argmax(wl.context_lens))]
    r = run(wl, rows=sample_rows(wl, seqs, rng, per_seq=8, q_tile=256 // wl.group), sample_seqs=seqs, schedule=DYN)
    assert_parity(r)


def test_full_size_prefill_sampled():
    wl = workloads.prefill()
    rng = np.random.default_rng(11)
    seqs = sorted({int(np.argmax(wl.q_lens)), int(np.argmin(wl.q_lens)), int(rng.integers(wl.num_seqs))})
    r = run(wl, rows=sample_rows(wl, seqs, rng, per_seq=12, q_tile=256 // wl.group), sample_seqs=seqs, schedule=DYN)
    assert_parity(r)


@pytest.mark.parametrize("mixed", [False, True])
@pytest.mark.parametrize("dynamic", [False, True])
def test_trace_accounts_for_every_task(dynamic, mixed):
    # the per-CTA trace: every non-hole task counted once, its rows x keys summed, start <= end
    # (static mixed batches run on the unified tcgen05 kernel, the rest on the decode-path kernel)
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import step as xystep
    q_lens = [300, 1, 1, 77, 1, 1, 1, 40, 1, 1, 1, 3] if mixed else [1] * 12
    wl = workloads.custom(q_lens, [4000, 30, 30, 300, 900, 17, 1, 2500, 64, 65, 640, 3], 8, 2, 128, 16, seed=21)
    dev = torch.device("cuda")
    vals = wl.tensors(dev)
    n = 7
    batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                              wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, num_ctas=n, kv_chunk=512,
                              schedule=DYN if dynamic else 3)
    pl = batch.plan
    trace = torch.zeros(n, 4, dtype=torch.int64, device=dev)
    out = torch.empty_like(vals["q"])
    xy.xy_paged_attention_traced(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"], vals["v_pool"],
                                 wl.scale, wl.causal, pl.tasks, pl.merges, n, pl.workspace,
                                 pl.task_counter if dynamic else None, trace, batch.err, out)
    torch.cuda.synchronize()
    xystep.check(batch)
    tr = trace.cpu().numpy()
    tasks = pl.host["tasks"]
    real = tasks[tasks[:, 0] >= 0]
    assert tr[:, 2].sum() == len(real)
    assert tr[:, 3].sum() == int((real[:, 3].astype(np.int64) * 4 * (real[:, 5] - real[:, 4])).sum())
    assert (tr[:, 1] >= tr[:, 0]).all() and (tr[:, 0] > 0).all()
    if not dynamic:
        # the static deal: CTA c runs the non-hole records at positions c, c + n, ...
        for c in range(n):
            mine = tasks[c::n]
            mine = mine[mine[:, 0] >= 0]
            assert tr[c, 2] == len(mine)
    s = xy.trace_summary(tr)
    assert 0 < s["busy_balance"] <= 1 and s["tail_us"] >= 0


@pytest.mark.parametrize("mixed", [False, True])
def test_many_tasks_per_cta_wrap_the_claim_queue(mixed):
    # two CTAs for ~200 tasks: each CTA's 8-slot claim queue wraps around many times
    rng = np.random.default_rng(31)
    S = 60
    ctx = [int(x) for x in rng.integers(20, 900, size=S)]
    q = [int(min(c, rng.integers(2, 150))) if (mixed and i % 7 == 0) else 1 for i, c in enumerate(ctx)]
    wl = workloads.custom(q, ctx, 8, 2, 128, 16, True, seed=33 + int(mixed))
    r = run(wl, num_ctas=2, kv_chunk=256, schedule=DYN)
    assert len(r["batch"].plan.host["tasks"]) > 100
    assert_parity(r)
    assert r["batch"].plan.task_counter.cpu().tolist() == [0, 0]
