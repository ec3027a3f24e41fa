"""xy_paged_attention_noalloc: the attention entry point for callers that cannot allocate device
memory (for example a server that gives all free HBM to the KV page pool at start-up).  Its
split-KV scratch is a fixed array inside libxy; its output must match xy_paged_attention's, which
takes a caller workspace, call after call.

This file is collected last so that a run stopping at the first failure has run every other
test before it; it also passes on its own in a fresh process."""

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


@pytest.fixture(scope="module")
def xy():
    from paged_kv_varlen_xy_gb300 import build
    build.build()
    import paged_kv_varlen_xy_gb300 as m
    return m


def _prepared(xy, kv_chunk):
    from paged_kv_varlen_xy_gb300 import step as xystep
    wl = workloads.custom([3, 1, 50, 1, 17], [300, 257, 190, 64, 900], 8, 2, 128, 16, seed=21)
    vals = wl.tensors("cuda")
    batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                              wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, kv_chunk=kv_chunk)
    # append once so that both entry points read the same pages
    xy.xy_slot_mapping(batch.cu, batch.ctx, batch.block_table, wl.block_size, wl.num_pages, batch.slots, batch.err)
    xy.xy_kv_append(vals["k_new"], vals["v_new"], batch.slots, vals["k_pool"], vals["v_pool"], batch.err)
    return wl, vals, batch


def test_noalloc_matches_workspace_entry_point_on_two_calls(xy):
    wl, vals, batch = _prepared(xy, kv_chunk=128)
    pl = batch.plan
    assert pl.merges.shape[0] > 0 and 0 < pl.host["workspace_bytes"] <= xy.XY_NOALLOC_SCRATCH_BYTES
    ref = torch.empty_like(vals["q"])
    xy.xy_paged_attention(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"], vals["v_pool"],
                          wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas, pl.workspace, batch.err, ref)
    torch.cuda.synchronize()
    assert int(batch.err.item()) == 0
    ref64 = ref.float().cpu().numpy().astype(np.float64)
    for _ in range(2):
        out = torch.full_like(vals["q"], float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        xy.xy_paged_attention_noalloc(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"],
                                      vals["v_pool"], wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas,
                                      pl.host["workspace_bytes"], err, out)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        diff = np.abs(out.float().cpu().numpy().astype(np.float64) - ref64)
        assert np.isfinite(diff).all()
        assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS


def test_noalloc_rejects_batches_beyond_its_scratch(xy):
    wl, vals, batch = _prepared(xy, kv_chunk=128)
    pl = batch.plan
    out = torch.empty_like(vals["q"])
    with pytest.raises(xy.XYError) as e:
        xy.xy_paged_attention_noalloc(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"],
                                      vals["v_pool"], wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas,
                                      xy.XY_NOALLOC_SCRATCH_BYTES + 1, batch.err, out)
    assert e.value.status == -6
