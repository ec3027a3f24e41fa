"""One step of the path composed from the oracle's functions (test infrastructure only).

Block table from the free list, slot mapping, KV append, then attention for all rows or for a
sample of rows.  To check full-size batches, the page pool may be given as a subset: the physical
pages ``pool_pages`` whose contents ``k_pool``/``v_pool`` hold (every page the sampled sequences
use); physical ids are renumbered to local ones, which does not change attention (the result is
invariant under a permutation of physical pages).
"""

import numpy as np

from .attention import attention_rows, paged_attention
from .bf16 import bf16_bits_to_f64
from .fp8 import dequantize, kv_append_fp8, quantize_rows
from .paged import allocate_block_table, kv_append, slot_mapping


def _localize(bt, slots, block_size, pool_pages):
    """Block table and slots renumbered to positions in pool_pages (None: unchanged)."""
    if pool_pages is None:
        return bt, slots
    pool_pages = np.asarray(pool_pages)
    lut = {int(p): i for i, p in enumerate(pool_pages)}
    local_bt = np.array([[lut.get(int(p), -1) if p >= 0 else -1 for p in row] for row in bt], dtype=np.int32)
    local_slots = np.array([(lut[int(s) // block_size] * block_size + int(s) % block_size)
                            if int(s) // block_size in lut else -1 for s in slots], dtype=np.int64)
    return local_bt, local_slots


def run_step(cu_seqlens_q, context_lens, free_list, block_size, max_blocks, q_bits, k_new_bits, v_new_bits,
             k_pool_bits, v_pool_bits, scale, causal, pool_pages=None, rows=None):
    """Returns dict(block_table, slots, k_pages, v_pages, out).

    q_bits [T, Hq, d], k_new_bits/v_new_bits [T, Hkv, d]: uint16 bf16 bit patterns.
    k_pool_bits/v_pool_bits [n, Hkv, bs, d]: the pool before the append (all P pages, or the
    pages listed in pool_pages).  rows: list of (token, query head), or None for every row.
    out is float64, [T, Hq, d] or [len(rows), d]; k_pages/v_pages are the pool (subset) after
    the append, as bits.
    """
    bt = allocate_block_table(context_lens, block_size, free_list, max_blocks)
    slots = slot_mapping(cu_seqlens_q, context_lens, bt, block_size)
    local_bt, local_slots = _localize(bt, slots, block_size, pool_pages)
    kp, vp = kv_append(k_pool_bits, v_pool_bits, k_new_bits, v_new_bits, local_slots)
    q = bf16_bits_to_f64(q_bits)
    kf, vf = bf16_bits_to_f64(kp), bf16_bits_to_f64(vp)
    if rows is None:
        out = paged_attention(q, cu_seqlens_q, context_lens, local_bt, kf, vf, scale, causal)
    else:
        out = attention_rows(rows, q, cu_seqlens_q, context_lens, local_bt, kf, vf, scale, causal)
    return dict(block_table=bt, slots=slots, k_pages=kp, v_pages=vp, out=out)


def run_step_fp8(cu_seqlens_q, context_lens, free_list, block_size, max_blocks, q_bits, k_new_bits, v_new_bits,
                 k_pool_bits, v_pool_bits, scale, causal, pool_pages=None, rows=None):
    """The step over 8-bit pages.  The pool before the step holds the bf16 rows k_pool_bits /
    v_pool_bits [n, Hkv, bs, d] (all P pages, or the pages listed in pool_pages, as in run_step)
    quantized row by row (as if each had been appended); the new tokens are appended quantized,
    and attention runs on the dequantized pages (all rows, or the (token, query head) pairs in
    rows).  Returns dict(block_table, slots, k_codes, v_codes, k_scales, v_scales (the pool after
    the append), out)."""
    bt = allocate_block_table(context_lens, block_size, free_list, max_blocks)
    slots = slot_mapping(cu_seqlens_q, context_lens, bt, block_size)
    local_bt, local_slots = _localize(bt, slots, block_size, pool_pages)
    kc, ks = quantize_rows(k_pool_bits)
    vc, vs = quantize_rows(v_pool_bits)
    kc, vc, ks, vs = kv_append_fp8(kc, vc, ks, vs, k_new_bits, v_new_bits, local_slots)
    q = bf16_bits_to_f64(q_bits)
    kf, vf = dequantize(kc, ks), dequantize(vc, vs)
    if rows is None:
        out = paged_attention(q, cu_seqlens_q, context_lens, local_bt, kf, vf, scale, causal)
    else:
        out = attention_rows(rows, q, cu_seqlens_q, context_lens, local_bt, kf, vf, scale, causal)
    return dict(block_table=bt, slots=slots, k_codes=kc, v_codes=vc, k_scales=ks, v_scales=vs, out=out)
