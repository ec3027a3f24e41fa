"""One step of the path through the C ABI: block table (host), task table (host), slot mapping,
KV append and paged attention (device).  Composition of libxy calls only; no arithmetic here."""

import numpy as np
import torch

from . import (Plan, check_err_word, xy_build_block_table, xy_kv_append, xy_kv_append_fp8, xy_paged_attention,
               xy_paged_attention_fp8, xy_slot_mapping)


class PagedBatch:
    """Per-batch metadata on the device: cu_seqlens_q, context_lens, block table, slot mapping
    buffer and the attention plan.  Built from host arrays (the scheduler's view of the batch)."""

    def __init__(self, cu_seqlens_q, context_lens, free_list, block_size, max_blocks, num_heads_q, num_heads_kv,
                 head_dim, causal, device="cuda", num_ctas=None, q_tile=None, kv_chunk=None, schedule=3,
                 kv_fp8=False):
        dev = torch.device(device)
        self.cu_host = np.asarray(cu_seqlens_q, dtype=np.int32)
        self.ctx_host = np.asarray(context_lens, dtype=np.int32)
        self.block_table_host, self.pages_used = xy_build_block_table(self.ctx_host, block_size, free_list, max_blocks)
        self.plan = Plan(self.cu_host, self.ctx_host, num_heads_q, num_heads_kv, head_dim, causal, device=dev,
                         num_ctas=num_ctas, q_tile=q_tile, kv_chunk=kv_chunk, schedule=schedule, kv_fp8=kv_fp8)
        self.cu = torch.from_numpy(self.cu_host).to(dev)
        self.ctx = torch.from_numpy(self.ctx_host).to(dev)
        self.block_table = torch.from_numpy(self.block_table_host).to(dev)
        self.slots = torch.empty(int(self.cu_host[-1]), dtype=torch.int64, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.block_size = block_size
        self.causal = causal


def run_step(batch, q, k_new, v_new, k_pages, v_pages, scale, out=None, stream=None):
    """a2 slot mapping -> a3 KV append -> a5..a10 attention, all enqueued on `stream`.
    Returns out [T, Hq, d] bf16.  Device-side errors accumulate in batch.err (see check())."""
    out = torch.empty_like(q) if out is None else out
    P = k_pages.shape[0]
    xy_slot_mapping(batch.cu, batch.ctx, batch.block_table, batch.block_size, P, batch.slots, batch.err, stream)
    xy_kv_append(k_new, v_new, batch.slots, k_pages, v_pages, batch.err, stream)
    pl = batch.plan
    xy_paged_attention(q, batch.cu, batch.ctx, batch.block_table, k_pages, v_pages, scale, batch.causal, pl.tasks,
                       pl.merges, pl.num_ctas, pl.workspace, batch.err, out, stream)
    return out


def run_step_fp8(batch, q, k_new, v_new, k_pages, v_pages, k_scales, v_scales, scale, out=None, stream=None):
    """run_step over 8-bit pages (E4M3 codes + per-row fp32 scales); batch built with kv_fp8=True."""
    out = torch.empty_like(q) if out is None else out
    P = k_pages.shape[0]
    xy_slot_mapping(batch.cu, batch.ctx, batch.block_table, batch.block_size, P, batch.slots, batch.err, stream)
    xy_kv_append_fp8(k_new, v_new, batch.slots, k_pages, v_pages, k_scales, v_scales, batch.err, stream)
    pl = batch.plan
    xy_paged_attention_fp8(q, batch.cu, batch.ctx, batch.block_table, k_pages, v_pages, k_scales, v_scales, scale,
                           batch.causal, pl.tasks, pl.merges, pl.num_ctas, pl.workspace, batch.err, out, stream)
    return out


def check(batch):
    check_err_word(batch.err)
