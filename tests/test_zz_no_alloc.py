"""xy_paged_attention_noalloc: the attention entry point for callers that cannot allocate device
memory (for example a server that gives all free HBM to the KV page pool at start-up).  Its
split-KV scratch is a fixed array inside libxy.  Given the same task table it runs the same
kernels as xy_paged_attention, which takes a caller workspace, so the two outputs must agree bit
for bit, call after call; both are also checked against the oracle.

The scratch array keeps whatever the previous call left in it.  A batch with more split rows runs
through it first, so a later, smaller batch would show any leftover partial that leaked into its
merge.

This file is collected last so that a run stopping at the first failure has run every other
test before it; it also passes on its own in a fresh process."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import MAX_ABS, MEAN_ABS, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def xy():
    from paged_kv_varlen_xy_gb300 import build
    build.build()
    import paged_kv_varlen_xy_gb300 as m
    return m


def _prepared(xy, q_lens, ctx, seed, kv_chunk):
    """A bf16 batch with its pages appended once (both entry points then read the same pages), the
    oracle's output for every row, and the host copy of the pool before the append."""
    from paged_kv_varlen_xy_gb300 import step as xystep
    wl = workloads.custom(q_lens, ctx, 8, 2, 128, 16, seed=seed)
    vals = wl.tensors("cuda")
    k0, v0 = bits(vals["k_pool"]), bits(vals["v_pool"])
    batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                              wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, kv_chunk=kv_chunk)
    xy.xy_slot_mapping(batch.cu, batch.ctx, batch.block_table, wl.block_size, wl.num_pages, batch.slots, batch.err)
    xy.xy_kv_append(vals["k_new"], vals["v_new"], batch.slots, vals["k_pool"], vals["v_pool"], batch.err)
    torch.cuda.synchronize()
    assert int(batch.err.item()) == 0
    ref = oracle.step.run_step(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                               bits(vals["q"]), bits(vals["k_new"]), bits(vals["v_new"]), k0, v0, wl.scale, wl.causal)
    return wl, vals, batch, ref["out"]


def _noalloc(xy, wl, vals, batch):
    pl = batch.plan
    out = torch.full_like(vals["q"], float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xy.xy_paged_attention_noalloc(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"], vals["v_pool"],
                                  wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas, pl.host["workspace_bytes"],
                                  err, out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


def _workspace(xy, wl, vals, batch):
    pl = batch.plan
    out = torch.full_like(vals["q"], float("nan"))
    xy.xy_paged_attention(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"], vals["v_pool"],
                          wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas, pl.workspace, batch.err, out)
    torch.cuda.synchronize()
    assert int(batch.err.item()) == 0
    return out


def _assert_oracle(out, ref):
    got = oracle.bf16_bits_to_f64(bits(out))
    diff = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS, (diff.max(), diff.mean())


def test_noalloc_matches_workspace_entry_point_on_two_calls(xy):
    # a larger batch first: more split rows than the compared batch, so its partials fill more of
    # the library's scratch than the compared batch overwrites
    big = _prepared(xy, [1] * 8 + [40, 64], [4000, 3100, 2600, 5000, 1900, 3500, 7000, 6100, 900, 2000], seed=20,
                   kv_chunk=128)
    small = _prepared(xy, [3, 1, 50, 1, 17], [300, 257, 190, 64, 900], seed=21, kv_chunk=128)
    ws_big, ws_small = big[2].plan.host["workspace_bytes"], small[2].plan.host["workspace_bytes"]
    assert small[2].plan.merges.shape[0] > 0
    assert 0 < ws_small < ws_big <= xy.XY_NOALLOC_SCRATCH_BYTES
    out_big = _noalloc(xy, *big[:3])
    _assert_oracle(out_big, big[3])

    wl, vals, batch, ref = small
    expect = _workspace(xy, wl, vals, batch)
    _assert_oracle(expect, ref)
    for _ in range(2):
        out = _noalloc(xy, wl, vals, batch)
        assert torch.equal(out.view(torch.int16), expect.view(torch.int16)), "differs from xy_paged_attention"
        _assert_oracle(out, ref)


def test_noalloc_rejects_batches_beyond_its_scratch(xy):
    wl, vals, batch, _ = _prepared(xy, [3, 1, 50, 1, 17], [300, 257, 190, 64, 900], seed=21, kv_chunk=128)
    pl = batch.plan
    out = torch.empty_like(vals["q"])
    with pytest.raises(xy.XYError) as e:
        xy.xy_paged_attention_noalloc(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"],
                                      vals["v_pool"], wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas,
                                      xy.XY_NOALLOC_SCRATCH_BYTES + 1, batch.err, out)
    assert e.value.status == -6
