"""Oracle: a plain, slow, obviously correct CPU restatement of the paged-KV varlen attention path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the C-ABI library under
``paged_kv_varlen_xy_gb300/csrc`` and its Python binding) imports, links or calls
anything here.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may use it.  The oracle shares no code,
header, table or constant with the CUDA path; the two meet only through the seeded
input generators in ``workloads.py`` (which hold none of the method's arithmetic).

Arithmetic is NumPy float64 with explicit loops over sequences and heads; bf16
values are read bit-exactly (bf16 -> fp64 is exact) and integer work (block table,
slot mapping, append, task table) is exact.

Sources (web pages on the subject; cited by title and section):

* [XY]    "XY-Serve 深度实战：当昇腾 NPU 终于学会「驯服动态负载」" (chenxutan.com/d/5031):
          §1.1 (prefill/decode definition), §2.2 component 1 (dynamic decomposer),
          component 2 (attention task reorder), component 3 (Meta-Attention kernel),
          §2.3 technique 1 (virtual padding), §4.2 (KV cache allocator),
          §4.3 (Meta-Attention module), §4.4 (decomposer / load-balance analysis).
* [MindIE] MindIE serving notes (hwcomputing.csdn.net/6a130621662f9a54cb76c319):
          "KV Cache 的 Block 级管理" (256-token blocks), "Prefill Chunking".
* [CANN]  cann-recipes-infer Paged KV Cache / Packed Sequence notes (dpshk.com/news/5336026):
          §2.2 (paged KV cache, page table), §2.3 (packed sequence, cu_seqlens),
          §3.1 (page pool layout), §3.2 (page allocation), §3.3 (packed paged_attention
          call), §4.4 (fault checks), §5.2 (scale metadata beside the pages), §5.3
          (page-size rule).
* [ATB]   ATB dynamic batching / speculative decoding / KV reuse notes
          (ai6s.net/6a38a2a6662f9a54cb828d66): "KV缓存复用", "端到端推理调优".

Readings where the pages are silent or inconsistent are stated in the docstring of the
function that takes them.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against
closed forms, worked examples printed on the pages (``tests/golden/``), brute force
on tiny inputs and a textbook library routine (``torch`` SDPA in fp64).  No function
is "parity unpinned".
"""

from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits
from .paged import (
    pack_cu_seqlens,
    allocate_block_table,
    slot_mapping,
    kv_append,
    gather_kv,
)
from .attention import (
    paged_attention,
    attention_row,
    attention_rows,
    split_row_partials,
    combine_partials,
    virtual_mask,
)
from .tasks import build_task_table, TASK_FIELDS, MERGE_FIELDS
from .fp8 import e4m3_to_f64, f64_to_e4m3, quantize_rows, dequantize, dequantize_to_bf16_bits, kv_append_fp8
from . import step

__all__ = [
    "bf16_bits_to_f64",
    "f64_to_bf16_bits",
    "pack_cu_seqlens",
    "allocate_block_table",
    "slot_mapping",
    "kv_append",
    "gather_kv",
    "paged_attention",
    "attention_row",
    "attention_rows",
    "split_row_partials",
    "combine_partials",
    "virtual_mask",
    "e4m3_to_f64",
    "f64_to_e4m3",
    "quantize_rows",
    "dequantize",
    "dequantize_to_bf16_bits",
    "kv_append_fp8",
    "build_task_table",
    "TASK_FIELDS",
    "MERGE_FIELDS",
    "step",
]
