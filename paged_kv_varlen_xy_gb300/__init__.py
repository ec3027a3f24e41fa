"""Python binding of libxy (unified paged-KV varlen attention on GB300).

Argument marshalling only: every step of the path runs in libxy's C++ host code or CUDA
kernels.  The functions carry the C-ABI's names (``xy_*``, declared in ``include/xy.h``);
torch tensors supply device memory and the current CUDA stream, numpy arrays the host inputs
of the host-side builders.  If libxy.so has not been built the import still succeeds, but
every call raises; there is no fallback path.
"""

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libxy.so")

XY_DEV_PAGE_OOB = 0x1
XY_DEV_SLOT_OOB = 0x2
XY_DEV_BAD_TASK = 0x4
XY_DEV_TIMEOUT = 0x8

C_ABI = ("xy_status_string", "xy_last_error_string", "xy_version", "xy_default_num_ctas", "xy_build_block_table",
         "xy_slot_mapping", "xy_kv_append", "xy_build_task_table", "xy_paged_attention",
         "xy_paged_attention_noalloc", "xy_selftest_bounded_wait", "xy_kv_append_fp8",
         "xy_paged_attention_fp8", "xy_build_step_tables", "xy_dequant_pages_fp8", "xy_paged_attention_dynamic",
         "xy_paged_attention_traced", "xy_paged_attention_fp8_dynamic", "xy_kv_append_paged",
         "xy_kv_append_paged_fp8", "xy_default_tiles", "xy_build_fp8_step_tables",
         "xy_paged_attention_fp8_mixed", "xy_default_kv_chunk")

# size of the library-owned split-KV scratch used by xy_paged_attention_noalloc
XY_NOALLOC_SCRATCH_BYTES = 32 << 20
# 8-bit pages: rows per task when G <= this (include/xy.h)
XY_FP8_NARROW_ROWS = 16


class XYError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        detail = ""
        if status == -7:  # XY_ERR_CUDA: add the CUDA error text the library recorded
            detail = " [" + lib().xy_last_error_string().decode(errors="replace") + "]"
        super().__init__(f"{where}: {status_string(status)} (status {status}){detail}")


class XYDeviceError(RuntimeError):
    def __init__(self, bits):
        self.bits = bits
        names = [n for b, n in ((XY_DEV_PAGE_OOB, "page index out of range"), (XY_DEV_SLOT_OOB, "slot out of range"),
                                (XY_DEV_BAD_TASK, "malformed task"), (XY_DEV_TIMEOUT, "bounded wait expired"))
                 if bits & b]
        super().__init__("libxy device error: " + ", ".join(names or [hex(bits)]))


class TaskStats(ctypes.Structure):
    _fields_ = [("total_load", ctypes.c_int64), ("max_cta_load", ctypes.c_int64),
                ("min_cta_load", ctypes.c_int64), ("balance", ctypes.c_double)]


class StepTables(ctypes.Structure):
    """xy_step_tables: where xy_build_step_tables put each table in the staging buffer."""
    _fields_ = [("err_off", ctypes.c_size_t), ("cu_off", ctypes.c_size_t), ("ctx_off", ctypes.c_size_t),
                ("bt_off", ctypes.c_size_t), ("tasks_off", ctypes.c_size_t), ("merges_off", ctypes.c_size_t),
                ("bytes", ctypes.c_size_t), ("workspace_bytes", ctypes.c_size_t), ("num_tasks", ctypes.c_int),
                ("num_merges", ctypes.c_int), ("pages_used", ctypes.c_int), ("stats", TaskStats)]


class Fp8StepTables(ctypes.Structure):
    """xy_fp8_step_tables (include/xy.h): offsets, ranges and counts of a split 8-bit step."""
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "err_off", "cu_off", "ctx_off", "bt_off", "tile_cu_off", "tile_bt_off", "tile_pages_off", "tile_tasks_off",
        "tile_merges_off", "dec_cu_off", "dec_tasks_off", "dec_merges_off", "bytes", "tile_workspace_bytes",
        "dec_workspace_bytes")] + [(n, ctypes.c_int) for n in (
        "tile_seq_begin", "tile_seq_end", "dec_seq_begin", "dec_seq_end", "tile_tok_begin", "tile_tok_end",
        "dec_tok_begin", "dec_tok_end", "tile_num_pages", "tile_num_tasks", "tile_num_merges", "dec_num_tasks",
        "dec_num_merges", "pages_used")]


_lib = None


def lib():
    """The loaded libxy (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libxy.so is not built ({LIB_PATH}); run paged_kv_varlen_xy_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, I, I64, F, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    SZ = ctypes.c_size_t
    L.xy_status_string.argtypes = [I]
    L.xy_status_string.restype = ctypes.c_char_p
    L.xy_last_error_string.argtypes = []
    L.xy_last_error_string.restype = ctypes.c_char_p
    L.xy_version.argtypes = []
    L.xy_version.restype = I
    L.xy_default_num_ctas.argtypes = [I]
    L.xy_default_num_ctas.restype = I
    L.xy_build_block_table.argtypes = [P, I, I, P, I, I, P, P]
    L.xy_build_block_table.restype = I
    L.xy_slot_mapping.argtypes = [P, P, P, I, I, I, I, I, P, P, P]
    L.xy_slot_mapping.restype = I
    L.xy_kv_append.argtypes = [P, P, P, I, P, P, I, I, I, I, P, P]
    L.xy_kv_append.restype = I
    L.xy_kv_append_paged.argtypes = [P, P, P, P, P, I, I, I, P, P, I, I, I, I, P, P, P]
    L.xy_kv_append_paged.restype = I
    L.xy_kv_append_paged_fp8.argtypes = [P, P, P, P, P, I, I, I, P, P, P, P, I, I, I, I, P, P, P]
    L.xy_kv_append_paged_fp8.restype = I
    L.xy_build_task_table.argtypes = [P, P, I, I, I, I, I, I, I, I, I, P, I, P, P, I, P, P, P]
    L.xy_build_task_table.restype = I
    L.xy_default_tiles.argtypes = [I, I, I, I, I, P, P]
    L.xy_default_tiles.restype = I
    L.xy_default_kv_chunk.argtypes = [P, I, I, I, I, I, I, P]
    L.xy_default_kv_chunk.restype = I
    L.xy_build_fp8_step_tables.argtypes = [P, P, I, P, I, I, I, I, I, I, I, I, P, SZ, P]
    L.xy_build_fp8_step_tables.restype = I
    L.xy_paged_attention_fp8_mixed.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, I, P, P, I, P, SZ,
                                               P, SZ, P, P, P, P]
    L.xy_paged_attention_fp8_mixed.restype = I
    L.xy_paged_attention.argtypes = [P, P, P, P, I, P, P, I, I, I, I, I, I, I, F, I, P, I, P, I, I, P, SZ, P, P, P]
    L.xy_paged_attention.restype = I
    L.xy_paged_attention_noalloc.argtypes = [P, P, P, P, I, P, P, I, I, I, I, I, I, I, F, I, P, I, P, I, I, SZ, P, P,
                                             P]
    L.xy_paged_attention_noalloc.restype = I
    L.xy_selftest_bounded_wait.argtypes = [ctypes.c_uint32, P, P, P]
    L.xy_selftest_bounded_wait.restype = I
    L.xy_kv_append_fp8.argtypes = [P, P, P, I, P, P, P, P, I, I, I, I, P, P]
    L.xy_kv_append_fp8.restype = I
    L.xy_paged_attention_fp8.argtypes = [P, P, P, P, I, P, P, P, P, I, I, I, I, I, I, I, F, I, P, I, P, I, I, P, SZ,
                                         P, P, P]
    L.xy_paged_attention_fp8.restype = I
    L.xy_build_step_tables.argtypes = [P, P, I, P, I, I, I, I, I, I, I, I, I, I, I, P, SZ, P]
    L.xy_build_step_tables.restype = I
    L.xy_dequant_pages_fp8.argtypes = [P, P, P, P, I, I, I, I, P, I, P, P, P, P]
    L.xy_dequant_pages_fp8.restype = I
    L.xy_paged_attention_dynamic.argtypes = [P, P, P, P, I, P, P, I, I, I, I, I, I, I, F, I, P, I, P, I, I, P, SZ, P,
                                             P, P, P]
    L.xy_paged_attention_dynamic.restype = I
    L.xy_paged_attention_traced.argtypes = [P, P, P, P, I, P, P, I, I, I, I, I, I, I, F, I, P, I, P, I, I, P, SZ, P,
                                            P, P, P, P]
    L.xy_paged_attention_traced.restype = I
    L.xy_paged_attention_fp8_dynamic.argtypes = [P, P, P, P, I, P, P, P, P, I, I, I, I, I, I, I, F, I, P, I, P, I, I,
                                                 P, SZ, P, P, P, P]
    L.xy_paged_attention_fp8_dynamic.restype = I
    _lib = L
    return L


def status_string(status):
    return lib().xy_status_string(int(status)).decode()


def _check(status, where):
    if status != 0:
        raise XYError(status, where)


def _host_i32(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _dev(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    # the library launches on the current device (and picks per-device state by it)
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device} but the current CUDA device is cuda:{torch.cuda.current_device()}; "
                         "call inside torch.cuda.device(...) of the tensors' device")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    if s.device.index != torch.cuda.current_device():
        raise ValueError(f"stream is on {s.device} but the current CUDA device is cuda:{torch.cuda.current_device()}")
    return ctypes.c_void_p(s.cuda_stream)


def xy_version():
    return lib().xy_version()


def xy_default_num_ctas(device=0):
    n = lib().xy_default_num_ctas(int(device))
    if n < 0:
        raise XYError(n, "xy_default_num_ctas")
    return n


def xy_build_block_table(context_lens, block_size, free_list, max_blocks, out=None):
    """a1 (host): block table [S, max_blocks] int32 from the FIFO free list; returns (table, pages_used).
    out: optional C-contiguous int32 array [S, max_blocks] to write the table into."""
    ctx, pctx = _host_i32(context_lens)
    free, pfree = _host_i32(free_list)
    S = len(ctx)
    if out is None:
        table = np.empty((S, int(max_blocks)), dtype=np.int32)
    else:
        table = out
        if table.dtype != np.int32 or table.shape != (S, int(max_blocks)) or not table.flags.c_contiguous:
            raise ValueError("out must be a C-contiguous int32 array [S, max_blocks]")
    used = ctypes.c_int(0)
    _check(lib().xy_build_block_table(pctx, S, int(block_size), pfree, len(free), int(max_blocks),
                                      table.ctypes.data_as(ctypes.c_void_p), ctypes.byref(used)),
           "xy_build_block_table")
    return table, used.value


XY_SCHEDULE_AREA = 0
XY_SCHEDULE_SERPENTINE = 1
XY_SCHEDULE_MIXED = 2
XY_SCHEDULE_GREEDY = 3
XY_SCHEDULE_DYNAMIC = 4


def default_schedule(kv_fp8=False):
    """The task-table schedule a step uses unless told otherwise: the dynamic deal, over bf16 and
    8-bit pages alike (CTAs claim tasks while the kernel runs; over bf16 pages measured faster than
    the static deals on the prefill, mixed and skewed batches and level on decode; over 8-bit pages
    a little faster than the greedy deal on the device, and faster end to end, since the host only
    sorts the tasks instead of dealing them)."""
    return XY_SCHEDULE_DYNAMIC


_XY_ERR_CAPACITY = -10


def task_table_bound(cu_seqlens_q, context_lens, num_heads_kv, q_tile, kv_chunk):
    """Upper bounds on the tasks (before hole records) and merge records of a batch: every query
    tile counted with the chunks of its sequence's whole context."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    L = np.asarray(context_lens, dtype=np.int64)
    q = cu[1:] - cu[:-1]
    tiles = (q + q_tile - 1) // q_tile
    chunks = np.maximum(1, (L + kv_chunk - 1) // kv_chunk)
    return int(num_heads_kv * np.sum(tiles * chunks)), int(num_heads_kv * np.sum(tiles * (chunks > 1)))


def xy_build_task_table(cu_seqlens_q, context_lens, num_heads_q, num_heads_kv, head_dim, causal, num_ctas,
                        q_tile, kv_chunk, schedule=XY_SCHEDULE_AREA, tasks_out=None, merges_out=None):
    """a4 (host): returns dict(tasks [n,8] int32, merges [m,8] int32, workspace_bytes, stats).

    tasks_out / merges_out: optional C-contiguous int32 arrays [capacity, 8] to write into (the
    returned tasks / merges are then views of their first rows).  The builder runs once when they
    are large enough, else a second time into arrays of the reported size."""
    cu, pcu = _host_i32(cu_seqlens_q)
    ctx, pctx = _host_i32(context_lens)
    S = len(cu) - 1
    args = (pcu, pctx, S, int(num_heads_q), int(num_heads_kv), int(head_dim), int(bool(causal)), int(num_ctas),
            int(q_tile), int(kv_chunk), int(schedule))
    n, m, ws = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_size_t(0)
    L = lib()
    st = TaskStats()
    for arr in (tasks_out, merges_out):
        if arr is not None and (arr.dtype != np.int32 or arr.ndim != 2 or arr.shape[1] != 8
                                or not arr.flags.c_contiguous):
            raise ValueError("tasks_out / merges_out must be C-contiguous int32 arrays [capacity, 8]")
    if tasks_out is None or merges_out is None:
        n_est, m_est = task_table_bound(cu, ctx, num_heads_kv, q_tile, kv_chunk)
        n_est += 4 * int(num_ctas)  # room for hole records
    tasks = tasks_out if tasks_out is not None else np.zeros((max(1, n_est), 8), np.int32)
    merges = merges_out if merges_out is not None else np.zeros((max(1, m_est), 8), np.int32)
    status = L.xy_build_task_table(*args, tasks.ctypes.data_as(ctypes.c_void_p), tasks.shape[0], ctypes.byref(n),
                                   merges.ctypes.data_as(ctypes.c_void_p), merges.shape[0], ctypes.byref(m),
                                   ctypes.byref(ws), ctypes.byref(st))
    if status == _XY_ERR_CAPACITY:
        # n and m hold the sizes needed
        tasks = np.zeros((n.value, 8), dtype=np.int32)
        merges = np.zeros((max(1, m.value), 8), dtype=np.int32)
        status = L.xy_build_task_table(*args, tasks.ctypes.data_as(ctypes.c_void_p), n.value, ctypes.byref(n),
                                       merges.ctypes.data_as(ctypes.c_void_p), merges.shape[0], ctypes.byref(m),
                                       ctypes.byref(ws), ctypes.byref(st))
    _check(status, "xy_build_task_table")
    return dict(tasks=tasks[:n.value], merges=merges[:m.value], workspace_bytes=ws.value,
                stats=dict(total_load=st.total_load, max_cta_load=st.max_cta_load,
                           min_cta_load=st.min_cta_load, balance=st.balance))


def xy_build_step_tables(cu_seqlens_q, context_lens, free_list, block_size, max_blocks, num_heads_q, num_heads_kv,
                         head_dim, causal, num_ctas, q_tile, kv_chunk, schedule, staging_ptr, staging_bytes):
    """One step's block table, task table and merge records packed into the host buffer at
    staging_ptr (see include/xy.h).  Returns (status, StepTables): status 0, or XY_ERR_CAPACITY
    with StepTables.bytes the size needed; other errors raise."""
    cu, pcu = _host_i32(cu_seqlens_q)
    ctx, pctx = _host_i32(context_lens)
    free, pfree = _host_i32(free_list)
    out = StepTables()
    st = lib().xy_build_step_tables(pcu, pctx, len(ctx), pfree, len(free), int(block_size), int(max_blocks),
                                    int(num_heads_q), int(num_heads_kv), int(head_dim), int(bool(causal)),
                                    int(num_ctas), int(q_tile), int(kv_chunk), int(schedule),
                                    ctypes.c_void_p(staging_ptr), int(staging_bytes), ctypes.byref(out))
    if st != _XY_ERR_CAPACITY:
        _check(st, "xy_build_step_tables")
    return st, out


def xy_slot_mapping(cu_seqlens_q, context_lens, block_table, block_size, num_pages, slot_mapping, err_word,
                    stream=None):
    """a2 (device): fills slot_mapping [T] int64 on the stream."""
    import torch
    S = cu_seqlens_q.numel() - 1
    _check(lib().xy_slot_mapping(_dev(cu_seqlens_q, torch.int32, "cu_seqlens_q"),
                                 _dev(context_lens, torch.int32, "context_lens"),
                                 _dev(block_table, torch.int32, "block_table"), S, block_table.shape[1],
                                 slot_mapping.numel(), int(block_size), int(num_pages),
                                 _dev(slot_mapping, torch.int64, "slot_mapping"),
                                 _dev(err_word, torch.int32, "err_word"), _stream(stream)), "xy_slot_mapping")


def xy_kv_append(k_new, v_new, slot_mapping, k_pages, v_pages, err_word, stream=None):
    """a3 (device): writes k_new/v_new [T, Hkv, d] into k_pages/v_pages [P, Hkv, bs, d] at the slots."""
    import torch
    P, Hkv, bs, d = k_pages.shape
    if tuple(v_pages.shape) != tuple(k_pages.shape) or tuple(k_new.shape) != tuple(v_new.shape):
        raise ValueError("K and V shapes differ")
    if k_new.shape[1:] != (Hkv, d) or k_new.shape[0] != slot_mapping.numel():
        raise ValueError("k_new must be [T, Hkv, d] with T = len(slot_mapping)")
    bf = torch.bfloat16
    _check(lib().xy_kv_append(_dev(k_new, bf, "k_new"), _dev(v_new, bf, "v_new"),
                              _dev(slot_mapping, torch.int64, "slot_mapping"), k_new.shape[0],
                              _dev(k_pages, bf, "k_pages"), _dev(v_pages, bf, "v_pages"), P, Hkv, bs, d,
                              _dev(err_word, torch.int32, "err_word"), _stream(stream)), "xy_kv_append")


def xy_kv_append_paged(k_new, v_new, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, err_word,
                       slot_mapping=None, stream=None):
    """a2 + a3 in one launch (device): each new token's slot from cu_seqlens_q / context_lens /
    block_table (int32, device), its K/V rows copied there; slot_mapping int64 [T] (optional)
    receives the slots."""
    import torch
    P, Hkv, bs, d = k_pages.shape
    if tuple(v_pages.shape) != tuple(k_pages.shape) or tuple(k_new.shape) != tuple(v_new.shape):
        raise ValueError("K and V shapes differ")
    T = k_new.shape[0]
    if k_new.shape[1:] != (Hkv, d) or (slot_mapping is not None and slot_mapping.numel() != T):
        raise ValueError("k_new must be [T, Hkv, d] and slot_mapping [T]")
    bf, i32 = torch.bfloat16, torch.int32
    _check(lib().xy_kv_append_paged(_dev(k_new, bf, "k_new"), _dev(v_new, bf, "v_new"),
                                    _dev(cu_seqlens_q, i32, "cu_seqlens_q"), _dev(context_lens, i32, "context_lens"),
                                    _dev(block_table, i32, "block_table"), cu_seqlens_q.numel() - 1,
                                    block_table.shape[1], T, _dev(k_pages, bf, "k_pages"), _dev(v_pages, bf, "v_pages"),
                                    P, Hkv, bs, d,
                                    _dev(slot_mapping, torch.int64, "slot_mapping") if slot_mapping is not None
                                    else None, _dev(err_word, i32, "err_word"), _stream(stream)), "xy_kv_append_paged")


def xy_kv_append_paged_fp8(k_new, v_new, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, k_scales,
                           v_scales, err_word, slot_mapping=None, stream=None):
    """xy_kv_append_paged for 8-bit pages (the quantizing append of xy_kv_append_fp8)."""
    import torch
    P, Hkv, bs, d = k_pages.shape
    if tuple(v_pages.shape) != tuple(k_pages.shape) or tuple(k_new.shape) != tuple(v_new.shape):
        raise ValueError("K and V shapes differ")
    if tuple(k_scales.shape) != (P, Hkv, bs) or tuple(v_scales.shape) != (P, Hkv, bs):
        raise ValueError("scales must be [P, Hkv, bs]")
    T = k_new.shape[0]
    if k_new.shape[1:] != (Hkv, d) or (slot_mapping is not None and slot_mapping.numel() != T):
        raise ValueError("k_new must be [T, Hkv, d] and slot_mapping [T]")
    bf, u8, f32, i32 = torch.bfloat16, torch.uint8, torch.float32, torch.int32
    _check(lib().xy_kv_append_paged_fp8(
        _dev(k_new, bf, "k_new"), _dev(v_new, bf, "v_new"), _dev(cu_seqlens_q, i32, "cu_seqlens_q"),
        _dev(context_lens, i32, "context_lens"), _dev(block_table, i32, "block_table"), cu_seqlens_q.numel() - 1,
        block_table.shape[1], T, _dev(k_pages, u8, "k_pages"), _dev(v_pages, u8, "v_pages"),
        _dev(k_scales, f32, "k_scales"), _dev(v_scales, f32, "v_scales"), P, Hkv, bs, d,
        _dev(slot_mapping, torch.int64, "slot_mapping") if slot_mapping is not None else None,
        _dev(err_word, i32, "err_word"), _stream(stream)), "xy_kv_append_paged_fp8")


def xy_paged_attention(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, scale, causal, tasks, merges,
                       num_ctas, workspace, err_word, out, stream=None):
    """a5..a10 (device): out [T, Hq, d] bf16.  tasks/merges: device int32 [n, 8] / [m, 8] from
    xy_build_task_table with the same num_ctas; workspace: device uint8 tensor (or None when no merges)."""
    import torch
    T, Hq, d = q.shape
    P, Hkv, bs, d2 = k_pages.shape
    if d2 != d or tuple(out.shape) != tuple(q.shape) or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("shape mismatch between q, out and the page pools")
    bf = torch.bfloat16
    nm = merges.shape[0] if merges is not None else 0
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None and workspace.numel() else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().xy_paged_attention(
        _dev(q, bf, "q"), _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q"), _dev(context_lens, torch.int32, "context_lens"),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1], _dev(k_pages, bf, "k_pages"),
        _dev(v_pages, bf, "v_pages"), P, cu_seqlens_q.numel() - 1, T, Hq, Hkv, d, bs, float(scale), int(bool(causal)),
        _dev(tasks, torch.int32, "tasks"), tasks.shape[0],
        _dev(merges, torch.int32, "merges") if nm else None, nm, int(num_ctas), ws_ptr, ws_bytes,
        _dev(err_word, torch.int32, "err_word"), _dev(out, bf, "out"), _stream(stream)), "xy_paged_attention")


def xy_paged_attention_dynamic(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, scale, causal, tasks,
                               merges, num_ctas, workspace, task_counter, err_word, out, stream=None):
    """xy_paged_attention with a dynamic deal: the persistent CTAs claim tasks in table order from
    task_counter (device int32 [2], zero before the first call; every launch returns it to zero)
    while they run."""
    import torch
    T, Hq, d = q.shape
    P, Hkv, bs, d2 = k_pages.shape
    if d2 != d or tuple(out.shape) != tuple(q.shape) or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("shape mismatch between q, out and the page pools")
    bf = torch.bfloat16
    nm = merges.shape[0] if merges is not None else 0
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None and workspace.numel() else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().xy_paged_attention_dynamic(
        _dev(q, bf, "q"), _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q"), _dev(context_lens, torch.int32, "context_lens"),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1], _dev(k_pages, bf, "k_pages"),
        _dev(v_pages, bf, "v_pages"), P, cu_seqlens_q.numel() - 1, T, Hq, Hkv, d, bs, float(scale), int(bool(causal)),
        _dev(tasks, torch.int32, "tasks"), tasks.shape[0],
        _dev(merges, torch.int32, "merges") if nm else None, nm, int(num_ctas), ws_ptr, ws_bytes,
        _dev(task_counter, torch.int32, "task_counter"), _dev(err_word, torch.int32, "err_word"), _dev(out, bf, "out"),
        _stream(stream)), "xy_paged_attention_dynamic")


def xy_paged_attention_traced(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, scale, causal, tasks,
                              merges, num_ctas, workspace, task_counter, cta_trace, err_word, out, stream=None):
    """Paged attention with a per-CTA trace: cta_trace device int64 [num_ctas, 4] = {start ns, end ns,
    tasks run, rows x keys}.  task_counter: device int32 [2] for the dynamic deal (as
    xy_paged_attention_dynamic), or None for the static deal (as xy_paged_attention)."""
    import torch
    T, Hq, d = q.shape
    P, Hkv, bs, d2 = k_pages.shape
    if d2 != d or tuple(out.shape) != tuple(q.shape) or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("shape mismatch between q, out and the page pools")
    if tuple(cta_trace.shape) != (int(num_ctas), 4):
        raise ValueError("cta_trace must be [num_ctas, 4]")
    bf = torch.bfloat16
    nm = merges.shape[0] if merges is not None else 0
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None and workspace.numel() else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().xy_paged_attention_traced(
        _dev(q, bf, "q"), _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q"), _dev(context_lens, torch.int32, "context_lens"),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1], _dev(k_pages, bf, "k_pages"),
        _dev(v_pages, bf, "v_pages"), P, cu_seqlens_q.numel() - 1, T, Hq, Hkv, d, bs, float(scale), int(bool(causal)),
        _dev(tasks, torch.int32, "tasks"), tasks.shape[0],
        _dev(merges, torch.int32, "merges") if nm else None, nm, int(num_ctas), ws_ptr, ws_bytes,
        _dev(task_counter, torch.int32, "task_counter") if task_counter is not None else None,
        _dev(cta_trace, torch.int64, "cta_trace"), _dev(err_word, torch.int32, "err_word"), _dev(out, bf, "out"),
        _stream(stream)), "xy_paged_attention_traced")


def trace_summary(cta_trace):
    """Balance and tail of one traced launch (cta_trace [num_ctas, 4] host int64 array): CTA busy
    times (end - start), their min/max ratio, the span from the first start to the last end, and
    the tail: the last end minus the median end (how long the slowest CTAs run after most are done)."""
    tr = np.asarray(cta_trace, dtype=np.int64)
    used = tr[tr[:, 2] > 0]
    if len(used) == 0:
        return {"ctas_used": 0}
    busy = (used[:, 1] - used[:, 0]) / 1e3
    t0 = int(tr[:, 0].min())
    ends = (used[:, 1] - t0) / 1e3
    return {"ctas_used": int(len(used)), "busy_us_min": float(busy.min()), "busy_us_max": float(busy.max()),
            "busy_balance": float(busy.min() / busy.max()) if busy.max() > 0 else 1.0,
            "span_us": float(ends.max()), "tail_us": float(ends.max() - np.median(ends)),
            "work_balance": float(used[:, 3].min() / used[:, 3].max()),
            "tasks_min": int(used[:, 2].min()), "tasks_max": int(used[:, 2].max())}


def xy_paged_attention_noalloc(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, scale, causal, tasks,
                               merges, num_ctas, workspace_bytes, err_word, out, stream=None):
    """xy_paged_attention for callers that cannot allocate device memory: the split-KV scratch
    comes from a fixed array inside libxy (XY_NOALLOC_SCRATCH_BYTES).  workspace_bytes is the
    size xy_build_task_table reported; larger batches raise XYError (XY_ERR_WORKSPACE).  Calls
    on one device share that array, so they must not overlap on the GPU."""
    import torch
    T, Hq, d = q.shape
    P, Hkv, bs, d2 = k_pages.shape
    if d2 != d or tuple(out.shape) != tuple(q.shape) or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("shape mismatch between q, out and the page pools")
    bf = torch.bfloat16
    nm = merges.shape[0] if merges is not None else 0
    _check(lib().xy_paged_attention_noalloc(
        _dev(q, bf, "q"), _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q"), _dev(context_lens, torch.int32, "context_lens"),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1], _dev(k_pages, bf, "k_pages"),
        _dev(v_pages, bf, "v_pages"), P, cu_seqlens_q.numel() - 1, T, Hq, Hkv, d, bs, float(scale), int(bool(causal)),
        _dev(tasks, torch.int32, "tasks"), tasks.shape[0],
        _dev(merges, torch.int32, "merges") if nm else None, nm, int(num_ctas), int(workspace_bytes),
        _dev(err_word, torch.int32, "err_word"), _dev(out, bf, "out"), _stream(stream)),
        "xy_paged_attention_noalloc")


def xy_kv_append_fp8(k_new, v_new, slot_mapping, k_pages, v_pages, k_scales, v_scales, err_word, stream=None):
    """a3 for 8-bit pages: quantizes k_new/v_new [T, Hkv, d] bf16 into k_pages/v_pages [P, Hkv, bs, d]
    uint8 (E4M3 codes) with one fp32 scale per row in k_scales/v_scales [P, Hkv, bs]."""
    import torch
    P, Hkv, bs, d = k_pages.shape
    if tuple(v_pages.shape) != tuple(k_pages.shape) or tuple(k_new.shape) != tuple(v_new.shape):
        raise ValueError("K and V shapes differ")
    if tuple(k_scales.shape) != (P, Hkv, bs) or tuple(v_scales.shape) != (P, Hkv, bs):
        raise ValueError("scales must be [P, Hkv, bs]")
    if k_new.shape[1:] != (Hkv, d) or k_new.shape[0] != slot_mapping.numel():
        raise ValueError("k_new must be [T, Hkv, d] with T = len(slot_mapping)")
    bf, u8, f32 = torch.bfloat16, torch.uint8, torch.float32
    _check(lib().xy_kv_append_fp8(_dev(k_new, bf, "k_new"), _dev(v_new, bf, "v_new"),
                                  _dev(slot_mapping, torch.int64, "slot_mapping"), k_new.shape[0],
                                  _dev(k_pages, u8, "k_pages"), _dev(v_pages, u8, "v_pages"),
                                  _dev(k_scales, f32, "k_scales"), _dev(v_scales, f32, "v_scales"), P, Hkv, bs, d,
                                  _dev(err_word, torch.int32, "err_word"), _stream(stream)), "xy_kv_append_fp8")


def xy_paged_attention_fp8(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, k_scales, v_scales, scale,
                           causal, tasks, merges, num_ctas, workspace, err_word, out, stream=None):
    """xy_paged_attention over 8-bit pages: k_pages/v_pages [P, Hkv, bs, 128] uint8 E4M3 codes,
    k_scales/v_scales [P, Hkv, bs] fp32 (as written by xy_kv_append_fp8).  tasks from a task table
    built with q_tile <= 64 // G (Plan(..., kv_fp8=True))."""
    a = _fp8_args(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, k_scales, v_scales, scale, causal,
                  tasks, merges, num_ctas, workspace, out)
    import torch
    _check(lib().xy_paged_attention_fp8(*a, _dev(err_word, torch.int32, "err_word"),
                                        _dev(out, torch.bfloat16, "out"), _stream(stream)),
           "xy_paged_attention_fp8")


def xy_paged_attention_fp8_dynamic(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, k_scales, v_scales,
                                   scale, causal, tasks, merges, num_ctas, workspace, task_counter, err_word, out,
                                   stream=None):
    """xy_paged_attention_fp8 with a dynamic deal: the CTAs claim tasks in table order from
    task_counter (device int32 [2], zero before the first call; every launch returns it to zero)."""
    import torch
    a = _fp8_args(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, k_scales, v_scales, scale, causal,
                  tasks, merges, num_ctas, workspace, out)
    _check(lib().xy_paged_attention_fp8_dynamic(*a, _dev(task_counter, torch.int32, "task_counter"),
                                                _dev(err_word, torch.int32, "err_word"),
                                                _dev(out, torch.bfloat16, "out"), _stream(stream)),
           "xy_paged_attention_fp8_dynamic")


def _fp8_args(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, k_scales, v_scales, scale, causal,
              tasks, merges, num_ctas, workspace, out):
    """The arguments the two 8-bit-page entries share, up to the workspace size (`out` is checked
    against q here and passed by the caller)."""
    import torch
    T, Hq, d = q.shape
    P, Hkv, bs, d2 = k_pages.shape
    if d2 != d or tuple(out.shape) != tuple(q.shape) or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("shape mismatch between q, out and the page pools")
    if tuple(k_scales.shape) != (P, Hkv, bs) or tuple(v_scales.shape) != (P, Hkv, bs):
        raise ValueError("scales must be [P, Hkv, bs]")
    bf, u8, f32 = torch.bfloat16, torch.uint8, torch.float32
    nm = merges.shape[0] if merges is not None else 0
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None and workspace.numel() else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return (_dev(q, bf, "q"), _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q"),
            _dev(context_lens, torch.int32, "context_lens"), _dev(block_table, torch.int32, "block_table"),
            block_table.shape[1], _dev(k_pages, u8, "k_pages"), _dev(v_pages, u8, "v_pages"),
            _dev(k_scales, f32, "k_scales"), _dev(v_scales, f32, "v_scales"), P, cu_seqlens_q.numel() - 1, T, Hq, Hkv,
            d, bs, float(scale), int(bool(causal)), _dev(tasks, torch.int32, "tasks"), tasks.shape[0],
            _dev(merges, torch.int32, "merges") if nm else None, nm, int(num_ctas), ws_ptr, ws_bytes)


def xy_build_fp8_step_tables(cu_seqlens_q, context_lens, free_list, block_size, max_blocks, num_heads_q, num_heads_kv,
                             head_dim, causal, num_ctas, staging_ptr, staging_bytes):
    """Tables of a split step over 8-bit pages packed into a host staging buffer (see include/xy.h).
    Returns (status, Fp8StepTables); status XY_ERR_CAPACITY (-10) means the buffer was too small
    (tables.bytes says how large it must be); any other error raises XYError."""
    cu, cu_p = _host_i32(cu_seqlens_q)
    ctx, ctx_p = _host_i32(context_lens)
    fl, fl_p = _host_i32(free_list)
    out = Fp8StepTables()
    st = lib().xy_build_fp8_step_tables(cu_p, ctx_p, len(ctx), fl_p, len(fl), int(block_size), int(max_blocks),
                                        int(num_heads_q), int(num_heads_kv), int(head_dim), int(bool(causal)),
                                        int(num_ctas), ctypes.c_void_p(staging_ptr), int(staging_bytes),
                                        ctypes.byref(out))
    if st not in (0, _XY_ERR_CAPACITY):
        raise XYError(st, "xy_build_fp8_step_tables")
    return st, out


def xy_paged_attention_fp8_mixed(q, tables_dev, t, k_pages, v_pages, k_scales, v_scales, num_seqs, max_blocks, scale,
                                 causal, num_ctas, copy_k, copy_v, tile_ws, dec_ws, task_counters, err_word, out,
                                 stream=None):
    """Attention of a split step over 8-bit pages from the device tables of xy_build_fp8_step_tables
    (tables_dev: uint8 device tensor holding the staging bytes; t: the Fp8StepTables)."""
    import torch
    T, Hq, d = q.shape
    P, Hkv, bs, _ = k_pages.shape
    bf, u8, f32 = torch.bfloat16, torch.uint8, torch.float32
    copy_pages = copy_k.shape[0] if copy_k is not None else 0
    _check(lib().xy_paged_attention_fp8_mixed(
        _dev(q, bf, "q"), _dev(tables_dev, u8, "tables"), ctypes.byref(t), _dev(k_pages, u8, "k_pages"),
        _dev(v_pages, u8, "v_pages"), _dev(k_scales, f32, "k_scales"), _dev(v_scales, f32, "v_scales"), P,
        int(num_seqs), T, int(max_blocks), Hq, Hkv, d, bs, float(scale), int(bool(causal)), int(num_ctas),
        _dev(copy_k, bf, "copy_k") if copy_pages else None, _dev(copy_v, bf, "copy_v") if copy_pages else None,
        copy_pages, _dev(tile_ws, u8, "tile_ws") if tile_ws is not None else None,
        tile_ws.numel() if tile_ws is not None else 0, _dev(dec_ws, u8, "dec_ws") if dec_ws is not None else None,
        dec_ws.numel() if dec_ws is not None else 0, _dev(task_counters, torch.int32, "task_counters"),
        _dev(err_word, torch.int32, "err_word"), _dev(out, bf, "out"), _stream(stream)), "xy_paged_attention_fp8_mixed")


def xy_dequant_pages_fp8(k_pages, v_pages, k_scales, v_scales, pages, k_out, v_out, err_word, stream=None):
    """bf16 copies of the listed 8-bit pages: k_out/v_out [n, Hkv, bs, d] bf16 <- pages[i] of
    k_pages/v_pages [P, Hkv, bs, d] uint8 with k_scales/v_scales [P, Hkv, bs] fp32; pages int32 [n]."""
    import torch
    P, Hkv, bs, d = k_pages.shape
    n = pages.numel()
    if tuple(k_out.shape) != (n, Hkv, bs, d) or tuple(v_out.shape) != (n, Hkv, bs, d):
        raise ValueError("k_out / v_out must be [len(pages), Hkv, bs, d]")
    u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
    _check(lib().xy_dequant_pages_fp8(_dev(k_pages, u8, "k_pages"), _dev(v_pages, u8, "v_pages"),
                                      _dev(k_scales, f32, "k_scales"), _dev(v_scales, f32, "v_scales"), P, Hkv, bs, d,
                                      _dev(pages, torch.int32, "pages"), n, _dev(k_out, bf, "k_out"),
                                      _dev(v_out, bf, "v_out"), _dev(err_word, torch.int32, "err_word"),
                                      _stream(stream)), "xy_dequant_pages_fp8")


def xy_selftest_bounded_wait(limit_us, err_word, result, stream=None):
    """Self-test of the kernels' bounded waits (see include/xy.h): err_word int32 [1] and
    result int32 [3] on the device."""
    import torch
    if result.numel() < 3:
        raise ValueError("result must hold 3 int32")
    _check(lib().xy_selftest_bounded_wait(int(limit_us), _dev(err_word, torch.int32, "err_word"),
                                          _dev(result, torch.int32, "result"), _stream(stream)),
           "xy_selftest_bounded_wait")


def check_err_word(err_word):
    """Synchronise on err_word's value and raise XYDeviceError if any device check fired."""
    bits = int(err_word.item())
    if bits:
        raise XYDeviceError(bits)


def default_kv_chunk(context_lens, num_heads_q, num_heads_kv, num_ctas, kv_fp8=False, pure_decode=False):
    """xy_default_kv_chunk: the KV chunk (8192 .. 65536 keys) with the least estimated makespan
    for this batch's context lengths on num_ctas persistent CTAs."""
    ctx, pctx = _host_i32(context_lens)
    ch = ctypes.c_int()
    _check(lib().xy_default_kv_chunk(pctx, len(ctx), int(num_heads_q), int(num_heads_kv), int(bool(kv_fp8)),
                                     int(bool(pure_decode)), int(num_ctas), ctypes.byref(ch)), "xy_default_kv_chunk")
    return ch.value


def default_tiles(num_heads_q, num_heads_kv, head_dim=128, kv_fp8=False, pure_decode=False):
    """(q_tile, kv_chunk): the kernels' tile policy for a batch of this shape (xy_default_tiles:
    two 128-row tcgen05 tiles per task where the shape allows, else decode-path task heights; over
    8-bit pages one token per task for pure decode batches; 16384-key KV chunks, the shape-only
    default; default_kv_chunk picks one for a batch's lengths)."""
    qt, ch = ctypes.c_int(), ctypes.c_int()
    _check(lib().xy_default_tiles(int(num_heads_q), int(num_heads_kv), int(head_dim), int(bool(kv_fp8)),
                                  int(bool(pure_decode)), ctypes.byref(qt), ctypes.byref(ch)), "xy_default_tiles")
    return qt.value, ch.value


class Plan:
    """Per-batch state for xy_paged_attention: the task table (built on the host from host copies of
    cu_seqlens_q and context_lens) uploaded to the device, and the workspace it needs."""

    def __init__(self, cu_seqlens_q, context_lens, num_heads_q, num_heads_kv, head_dim, causal, device="cuda",
                 num_ctas=None, q_tile=None, kv_chunk=None, schedule=None, kv_fp8=False):
        import torch
        dev = torch.device(device)
        self.num_ctas = num_ctas or xy_default_num_ctas(dev.index or 0)
        cu = np.asarray(cu_seqlens_q)
        schedule = default_schedule(kv_fp8) if schedule is None else schedule
        self.dynamic = schedule == XY_SCHEDULE_DYNAMIC
        pure = len(cu) > 1 and int(cu[-1]) == len(cu) - 1
        dq, _ = default_tiles(num_heads_q, num_heads_kv, head_dim, kv_fp8, pure_decode=pure)
        self.q_tile = q_tile or dq
        self.kv_chunk = kv_chunk or default_kv_chunk(context_lens, num_heads_q, num_heads_kv, self.num_ctas, kv_fp8,
                                                     pure)
        self.schedule = schedule
        # the dynamic deal's claim counter (every launch returns it to zero)
        self.task_counter = torch.zeros(2, dtype=torch.int32, device=dev) if self.dynamic else None
        r = xy_build_task_table(cu_seqlens_q, context_lens, num_heads_q, num_heads_kv, head_dim, causal,
                                self.num_ctas, self.q_tile, self.kv_chunk, schedule)
        self.host = r
        self.stats = r["stats"]
        self.tasks = torch.from_numpy(r["tasks"]).to(dev)
        self.merges = torch.from_numpy(r["merges"]).to(dev)
        self.workspace = torch.empty(max(r["workspace_bytes"], 16), dtype=torch.uint8, device=dev)
        self.causal = causal


def paged_attention(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, scale, causal, plan=None,
                    out=None, err_word=None, check=True):
    """out = attention of the packed queries over the paged cache (signature of the pages' packed
    paged_attention call).  Builds a Plan from host copies of cu_seqlens_q/context_lens when none is given."""
    import torch
    if plan is None:
        plan = Plan(cu_seqlens_q.cpu().numpy(), context_lens.cpu().numpy(), q.shape[1], k_pages.shape[1], q.shape[2],
                    causal, device=q.device)
    out = torch.empty_like(q) if out is None else out
    own_err = err_word is None
    err_word = torch.zeros(1, dtype=torch.int32, device=q.device) if own_err else err_word
    if plan.dynamic:
        xy_paged_attention_dynamic(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, scale, causal,
                                   plan.tasks, plan.merges, plan.num_ctas, plan.workspace, plan.task_counter,
                                   err_word, out)
    else:
        xy_paged_attention(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, scale, causal, plan.tasks,
                           plan.merges, plan.num_ctas, plan.workspace, err_word, out)
    if check and own_err:
        check_err_word(err_word)
    return out
