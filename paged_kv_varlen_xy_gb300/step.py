"""One step of the path through the C ABI: block table (host), task table (host), slot mapping,
KV append and paged attention (device).  Composition of libxy calls only; no arithmetic here."""

import numpy as np
import torch

from . import (XY_SCHEDULE_DYNAMIC, Plan, check_err_word, default_kv_chunk, default_schedule, default_tiles,
               xy_build_block_table, xy_build_step_tables, xy_default_num_ctas, xy_kv_append_paged,
               xy_kv_append_paged_fp8, xy_paged_attention, xy_paged_attention_dynamic, xy_paged_attention_fp8,
               xy_paged_attention_fp8_dynamic)


class PagedBatch:
    """Per-batch metadata on the device: cu_seqlens_q, context_lens, block table, slot mapping
    buffer and the attention plan.  Built from host arrays (the scheduler's view of the batch)."""

    def __init__(self, cu_seqlens_q, context_lens, free_list, block_size, max_blocks, num_heads_q, num_heads_kv,
                 head_dim, causal, device="cuda", num_ctas=None, q_tile=None, kv_chunk=None, schedule=None,
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


class _PlanView:
    """The attention plan of a Planner batch (the fields run_step reads from Plan)."""

    def __init__(self, batch, num_ctas, workspace, tbl, host_np):
        self._b, self.num_ctas, self.workspace, self._tbl, self._h = batch, num_ctas, workspace, tbl, host_np

    @property
    def stats(self):
        st = self._tbl.stats
        return dict(total_load=st.total_load, max_cta_load=st.max_cta_load, min_cta_load=st.min_cta_load,
                    balance=st.balance)

    @property
    def host(self):
        t, h, n, m = self._tbl, self._h, self._b.num_tasks, self._b.num_merges
        return dict(tasks=h[t.tasks_off:t.tasks_off + 32 * n].view(np.int32).reshape(n, 8),
                    merges=h[t.merges_off:t.merges_off + 32 * m].view(np.int32).reshape(m, 8),
                    workspace_bytes=t.workspace_bytes, stats=self.stats)

    @property
    def tasks(self):
        return self._b._view("tasks", (self._b.num_tasks, 8))

    @property
    def merges(self):
        return self._b._view("merges", (self._b.num_merges, 8))


class _StepBatch:
    """A Planner batch: the attributes of PagedBatch.  Its device tables live in the planner's
    device buffer (valid until the planner's next plan()); tensor views of them are made on
    demand, while Planner.run passes their addresses straight to libxy."""

    def __init__(self, dbuf, off, S, MB, n, m):
        self._dbuf, self._off, self.S, self.MB, self.num_tasks, self.num_merges = dbuf, off, S, MB, n, m
        self._base = dbuf.data_ptr()

    def addr(self, name):
        return self._base + self._off[name]

    def _view(self, name, shape):
        n_el = int(np.prod(shape))
        o = self._off[name]
        return self._dbuf[o:o + 4 * n_el].view(torch.int32).view(*shape)

    cu = property(lambda self: self._view("cu", (self.S + 1,)))
    ctx = property(lambda self: self._view("ctx", (self.S,)))
    block_table = property(lambda self: self._view("bt", (self.S, self.MB)))
    err = property(lambda self: self._view("err", (1,)))

    def _hv(self, name, n):
        o = self._off[name]
        return self._host_np[o:o + 4 * n].view(np.int32)

    # host views of the staged tables (valid until the planner's next plan())
    cu_host = property(lambda self: self._hv("cu", self.S + 1))
    ctx_host = property(lambda self: self._hv("ctx", self.S))
    block_table_host = property(lambda self: self._hv("bt", self.S * self.MB).reshape(self.S, self.MB))


class Planner:
    """Reusable builder of per-step metadata for one stream: the host-built block table, task and
    merge tables, cu_seqlens_q, context_lens and a zeroed error word are packed into one pinned
    staging buffer and reach the device in one host->device copy; the device buffer, split-KV
    workspace and slot-mapping buffer are kept between steps and grown when a batch needs more.
    A serving loop that re-plans every step calls plan() then run() once per step (PagedBatch
    instead builds and uploads each table separately).  Two device table buffers alternate: a
    batch's device tables stay valid until the plan() after next, its host views until the next
    plan().  plan(stream=s) uploads on s, which must then be ordered after the kernels of the batch
    planned two plans earlier (on the default stream that order holds by itself)."""

    _ALIGN = 256

    def __init__(self, num_heads_q, num_heads_kv, head_dim, block_size, max_blocks, causal, device="cuda",
                 num_ctas=None, q_tile=None, kv_chunk=None, schedule=None, kv_fp8=False):
        self.dev = torch.device(device)
        self.Hq, self.Hkv, self.d = num_heads_q, num_heads_kv, head_dim
        self.block_size, self.max_blocks, self.causal, self.kv_fp8 = block_size, max_blocks, causal, kv_fp8
        self.num_ctas = num_ctas or xy_default_num_ctas(self.dev.index or 0)
        # q_tile per batch over 8-bit pages (it depends on whether the batch is pure decode)
        self._q_tile_arg = q_tile
        schedule = default_schedule(kv_fp8) if schedule is None else schedule
        self.dynamic = schedule == XY_SCHEDULE_DYNAMIC
        tiles = default_tiles(num_heads_q, num_heads_kv, head_dim, kv_fp8)
        # the KV chunk per batch (default_kv_chunk of its lengths) unless one is given
        self._kv_chunk_arg = kv_chunk
        self.kv_chunk = kv_chunk or tiles[1]
        self.q_tile, self.schedule = q_tile or tiles[0], schedule
        # the dynamic deal's claim counter (every launch returns it to zero)
        self._counter = torch.zeros(2, dtype=torch.int32, device=self.dev) if self.dynamic else None
        self._host = None
        self._dev_bufs = [None, None]   # device tables, alternating between plans
        self._flip = 0
        self._ws = torch.empty(16, dtype=torch.uint8, device=self.dev)
        self._slots = torch.empty(1, dtype=torch.int64, device=self.dev)
        self._slot_views = {}
        self._copied = torch.cuda.Event()   # recorded after each upload
        self._pending = False
        self.last_upload_bytes = 0

    def _ensure(self, nbytes):
        """Staging and device buffers of at least nbytes (the staging buffer's contents are lost
        when it grows)."""
        if self._host is None or self._host.numel() < nbytes:
            size = max(nbytes, 2 * (self._host.numel() if self._host is not None else 0), 1 << 16)
            self._wait_upload()
            self._host = torch.empty(size, dtype=torch.uint8).pin_memory()
            self._host_np = self._host.numpy()
            self._host_ptr = self._host.data_ptr()
            self._dev_bufs = [None, None]
        for i in range(2):
            if self._dev_bufs[i] is None:
                self._dev_bufs[i] = torch.empty(self._host.numel(), dtype=torch.uint8, device=self.dev)

    def _wait_upload(self):
        if self._pending:
            self._copied.synchronize()   # the previous upload has left the staging buffer
            self._pending = False

    def wait_upload(self):
        """Block until the last plan's upload has left the pinned staging buffer (plan() does this
        first; a caller may do it beforehand to keep the wait out of its own timing)."""
        self._wait_upload()

    def plan(self, cu_seqlens_q, context_lens, free_list, stream=None, block_table=None):
        """Build and upload the metadata of one batch; returns a batch for run() (or run_step).
        block_table: a host int32 [S, max_blocks] table from the caller's own page allocator (a
        prefix cache whose rows share pages, say) that replaces the FIFO table before the upload."""
        self._ensure(1 << 16)
        self._wait_upload()   # the staging buffer is written below
        T = int(cu_seqlens_q[-1])
        pure = T == len(context_lens)
        if self.kv_fp8 and self._q_tile_arg is None:
            self.q_tile = default_tiles(self.Hq, self.Hkv, self.d, True, pure_decode=pure)[0]
        if self._kv_chunk_arg is None:
            self.kv_chunk = default_kv_chunk(context_lens, self.Hq, self.Hkv, self.num_ctas, self.kv_fp8, pure)
        for _ in range(2):
            st, tbl = xy_build_step_tables(cu_seqlens_q, context_lens, free_list, self.block_size, self.max_blocks,
                                           self.Hq, self.Hkv, self.d, self.causal, self.num_ctas, self.q_tile,
                                           self.kv_chunk, self.schedule, self._host_ptr, self._host.numel())
            if st == 0:
                break
            self._ensure(tbl.bytes)   # too small: grow and build again
        used_bytes = tbl.bytes
        if block_table is not None:
            S = len(context_lens)
            bt = np.ascontiguousarray(block_table, dtype=np.int32)
            if bt.shape != (S, self.max_blocks):
                raise ValueError("block_table must be [S, max_blocks] int32")
            self._host_np[tbl.bt_off:tbl.bt_off + bt.nbytes] = bt.view(np.uint8).ravel()
        stm = torch.cuda.current_stream(self.dev) if stream is None else stream
        self._flip ^= 1
        dbuf = self._dev_bufs[self._flip]
        with torch.cuda.stream(stm):
            dbuf[:used_bytes].copy_(self._host[:used_bytes], non_blocking=True)
        self._copied.record(stm)
        self._pending = True
        self.last_upload_bytes = used_bytes
        ws = tbl.workspace_bytes
        if self._ws.numel() < ws:
            self._ws = torch.empty(max(ws, 2 * self._ws.numel()), dtype=torch.uint8, device=self.dev)
        S = len(context_lens)
        T = int(cu_seqlens_q[-1])
        if self._slots.numel() < T:
            self._slots = torch.empty(max(T, 2 * self._slots.numel()), dtype=torch.int64, device=self.dev)
            self._slot_views = {}
        slots = self._slot_views.get(T)
        if slots is None:
            slots = self._slot_views[T] = self._slots[:T]
        off = {"err": tbl.err_off, "cu": tbl.cu_off, "ctx": tbl.ctx_off, "bt": tbl.bt_off, "tasks": tbl.tasks_off,
               "merges": tbl.merges_off}
        b = _StepBatch(dbuf, off, S, self.max_blocks, tbl.num_tasks, tbl.num_merges)
        b._host_np = self._host_np
        b.T = T
        b.pages_used = tbl.pages_used
        b.slots = slots
        b.block_size, b.causal = self.block_size, self.causal
        b.ws_bytes = ws
        b.plan = _PlanView(b, self.num_ctas, self._ws, tbl, self._host_np)
        return b

    def run(self, batch, q, k_new, v_new, k_pages, v_pages, scale, out=None, stream=None, k_scales=None,
            v_scales=None):
        """One step on a batch from plan(): slot mapping -> KV append -> paged attention (-> split-KV
        combine), the same libxy calls as run_step / run_step_fp8 with the batch's tables passed by
        address.  8-bit pages (kv_fp8 planners) take k_scales / v_scales.  Returns out."""
        import ctypes
        from . import _check, _dev, _stream, lib
        L = lib()
        out = torch.empty_like(q) if out is None else out
        T, Hq, d = q.shape
        P, Hkv, bs, _ = k_pages.shape
        if T != batch.T or Hq != self.Hq or Hkv != self.Hkv or d != self.d or bs != self.block_size:
            raise ValueError("tensor shapes differ from the planner's batch")
        st = _stream(stream)
        cu, ctx, bt, err = (ctypes.c_void_p(batch.addr(k)) for k in ("cu", "ctx", "bt", "err"))
        slots = _dev(batch.slots, torch.int64, "slots")
        tasks, merges = ctypes.c_void_p(batch.addr("tasks")), ctypes.c_void_p(batch.addr("merges"))
        ws = ctypes.c_void_p(self._ws.data_ptr())
        common = (batch.S, T, Hq, Hkv, d, bs, float(scale), int(bool(self.causal)), tasks, batch.num_tasks,
                  merges if batch.num_merges else None, batch.num_merges, self.num_ctas, ws, self._ws.numel(), err)
        bf = torch.bfloat16
        if self.kv_fp8:
            u8, f32 = torch.uint8, torch.float32
            _check(L.xy_kv_append_paged_fp8(_dev(k_new, bf, "k_new"), _dev(v_new, bf, "v_new"), cu, ctx, bt, batch.S,
                                            batch.MB, T, _dev(k_pages, u8, "k_pages"), _dev(v_pages, u8, "v_pages"),
                                            _dev(k_scales, f32, "k_scales"), _dev(v_scales, f32, "v_scales"), P, Hkv,
                                            bs, d, slots, err, st), "xy_kv_append_paged_fp8")
            pools = (_dev(q, bf, "q"), cu, ctx, bt, batch.MB, _dev(k_pages, u8, "k_pages"),
                     _dev(v_pages, u8, "v_pages"), _dev(k_scales, f32, "k_scales"), _dev(v_scales, f32, "v_scales"), P)
            if self.dynamic:
                _check(L.xy_paged_attention_fp8_dynamic(*pools, *common[:-1], ctypes.c_void_p(self._counter.data_ptr()),
                                                        err, _dev(out, bf, "out"), st),
                       "xy_paged_attention_fp8_dynamic")
            else:
                _check(L.xy_paged_attention_fp8(*pools, *common, _dev(out, bf, "out"), st), "xy_paged_attention_fp8")
        else:
            _check(L.xy_kv_append_paged(_dev(k_new, bf, "k_new"), _dev(v_new, bf, "v_new"), cu, ctx, bt, batch.S,
                                        batch.MB, T, _dev(k_pages, bf, "k_pages"), _dev(v_pages, bf, "v_pages"), P,
                                        Hkv, bs, d, slots, err, st), "xy_kv_append_paged")
            if self.dynamic:
                _check(L.xy_paged_attention_dynamic(_dev(q, bf, "q"), cu, ctx, bt, batch.MB,
                                                    _dev(k_pages, bf, "k_pages"), _dev(v_pages, bf, "v_pages"), P,
                                                    *common[:-1], ctypes.c_void_p(self._counter.data_ptr()), err,
                                                    _dev(out, bf, "out"), st), "xy_paged_attention_dynamic")
            else:
                _check(L.xy_paged_attention(_dev(q, bf, "q"), cu, ctx, bt, batch.MB, _dev(k_pages, bf, "k_pages"),
                                            _dev(v_pages, bf, "v_pages"), P, *common, _dev(out, bf, "out"), st),
                       "xy_paged_attention")
        return out


def run_step(batch, q, k_new, v_new, k_pages, v_pages, scale, out=None, stream=None):
    """a2 slot mapping -> a3 KV append -> a5..a10 attention, all enqueued on `stream`.
    Returns out [T, Hq, d] bf16.  Device-side errors accumulate in batch.err (see check())."""
    out = torch.empty_like(q) if out is None else out
    xy_kv_append_paged(k_new, v_new, batch.cu, batch.ctx, batch.block_table, k_pages, v_pages, batch.err,
                       slot_mapping=batch.slots, stream=stream)
    pl = batch.plan
    if pl.dynamic:
        xy_paged_attention_dynamic(q, batch.cu, batch.ctx, batch.block_table, k_pages, v_pages, scale, batch.causal,
                                   pl.tasks, pl.merges, pl.num_ctas, pl.workspace, pl.task_counter, batch.err, out,
                                   stream)
    else:
        xy_paged_attention(q, batch.cu, batch.ctx, batch.block_table, k_pages, v_pages, scale, batch.causal,
                           pl.tasks, pl.merges, pl.num_ctas, pl.workspace, batch.err, out, stream)
    return out


def run_step_fp8(batch, q, k_new, v_new, k_pages, v_pages, k_scales, v_scales, scale, out=None, stream=None):
    """run_step over 8-bit pages (E4M3 codes + per-row fp32 scales); batch built with kv_fp8=True."""
    out = torch.empty_like(q) if out is None else out
    xy_kv_append_paged_fp8(k_new, v_new, batch.cu, batch.ctx, batch.block_table, k_pages, v_pages, k_scales, v_scales,
                           batch.err, slot_mapping=batch.slots, stream=stream)
    pl = batch.plan
    if pl.dynamic:
        xy_paged_attention_fp8_dynamic(q, batch.cu, batch.ctx, batch.block_table, k_pages, v_pages, k_scales,
                                       v_scales, scale, batch.causal, pl.tasks, pl.merges, pl.num_ctas, pl.workspace,
                                       pl.task_counter, batch.err, out, stream)
    else:
        xy_paged_attention_fp8(q, batch.cu, batch.ctx, batch.block_table, k_pages, v_pages, k_scales, v_scales,
                               scale, batch.causal, pl.tasks, pl.merges, pl.num_ctas, pl.workspace, batch.err, out,
                               stream)
    return out


def split_ranges(q_lens):
    """(multi, single): the sequence ranges [a, b) of sequences with several new tokens and of
    one-token sequences, when each kind is one contiguous range (either may be empty); None when
    the kinds interleave (the rule xy_build_fp8_step_tables applies)."""
    multi = np.asarray(q_lens) > 1
    S = len(multi)
    changes = int(np.count_nonzero(multi[1:] != multi[:-1])) if S > 1 else 0
    if changes > 1:
        return None
    k = int(np.argmax(multi[1:] != multi[:-1])) + 1 if changes else S
    first = (0, k) if S else (0, 0)
    second = (k, S)
    if S and multi[0]:
        return first, second
    return second, first


class _Part:
    """The plan of one part of a split batch (the fields the bench and tests read from Plan)."""

    def __init__(self, tasks, merges, num_ctas, workspace, task_counter):
        self.tasks, self.merges, self.num_ctas, self.workspace = tasks, merges, num_ctas, workspace
        self.schedule, self.task_counter, self.dynamic = XY_SCHEDULE_DYNAMIC, task_counter, True
        self.stats = {"balance": None}


class _SplitBatch:
    """A batch of Fp8SplitPlanner.plan(): device views of its tables (cu, ctx, block_table, err,
    slots) and, per part, its sequence and token ranges and plan (tile / decode, None when empty)."""


class Fp8SplitPlanner:
    """Reusable planner of steps over 8-bit pages whose one-token (decode) sequences run on the
    8-bit decode path and whose multi-token sequences run on the tcgen05 tile path over bf16
    copies of their pages.  The tables (xy_build_fp8_step_tables: split, block table, page list
    and compact block table of the tile part, both task and merge tables) are built by libxy into
    one pinned staging buffer and reach the device in one copy; the device buffers, workspaces,
    slot buffer, claim counters and page-copy buffers are kept between steps and grown when a batch
    needs more.  Two device table buffers alternate between plans: a batch's device tables stay
    valid until the plan() after next (plan(stream=s) must be ordered after the kernels of the
    batch planned two plans earlier).  This class only marshals arguments."""

    def __init__(self, num_heads_q, num_heads_kv, head_dim, block_size, max_blocks, causal, device="cuda",
                 num_ctas=None):
        G = num_heads_q // num_heads_kv
        if head_dim != 128 or 128 % G:
            raise ValueError("the split path needs head_dim 128 and G dividing 128")
        self.dev = torch.device(device)
        self.Hq, self.Hkv, self.d, self.bs, self.MB, self.causal = (num_heads_q, num_heads_kv, head_dim, block_size,
                                                                   max_blocks, causal)
        self.num_ctas = num_ctas or xy_default_num_ctas(self.dev.index or 0)
        self._host = None
        self._dev_bufs = [None, None]   # device tables, alternating between plans
        self._flip = 0
        self._ws = [torch.empty(16, dtype=torch.uint8, device=self.dev) for _ in range(2)]
        self._slots = torch.empty(1, dtype=torch.int64, device=self.dev)
        self._copies = None
        # the two parts' claim counters (words 0-1 tile part, 2-3 decode part; each launch returns
        # its pair to zero)
        self._counters = torch.zeros(4, dtype=torch.int32, device=self.dev)
        self._copied = torch.cuda.Event() if self.dev.type == "cuda" else None
        self._pending = False
        self.last_upload_bytes = 0

    def _wait_upload(self):
        if self._pending:
            self._copied.synchronize()   # the previous upload has left the staging buffer
            self._pending = False

    def wait_upload(self):
        """Block until the last plan's upload has left the pinned staging buffer (plan() does this
        first; a caller may do it beforehand to keep the wait out of its own timing)."""
        self._wait_upload()

    def _ensure(self, nbytes):
        if self._host is None or self._host.numel() < nbytes:
            size = max(nbytes, 2 * (self._host.numel() if self._host is not None else 0), 1 << 16)
            self._wait_upload()
            self._host = torch.empty(size, dtype=torch.uint8).pin_memory()
            self._host_np = self._host.numpy()
            self._dev_bufs = [torch.empty(size, dtype=torch.uint8, device=self.dev) for _ in range(2)]

    def plan(self, cu_seqlens_q, context_lens, free_list, stream=None):
        from . import xy_build_fp8_step_tables
        cu = np.asarray(cu_seqlens_q, dtype=np.int32)
        ctx = np.asarray(context_lens, dtype=np.int32)
        self._ensure(1 << 16)
        self._wait_upload()   # the staging buffer is written below
        for _ in range(2):
            st, t = xy_build_fp8_step_tables(cu, ctx, free_list, self.bs, self.MB, self.Hq, self.Hkv, self.d,
                                             self.causal, self.num_ctas, self._host.data_ptr(), self._host.numel())
            if st == 0:
                break
            self._ensure(t.bytes)   # too small: grow and build again
        total = t.bytes
        stm = torch.cuda.current_stream(self.dev) if stream is None else stream
        self._flip ^= 1
        dbuf = self._dev_bufs[self._flip]
        with torch.cuda.stream(stm):
            dbuf[:total].copy_(self._host[:total], non_blocking=True)
        self._copied.record(stm)
        self._pending = True
        self.last_upload_bytes = total

        def dv(off, shape):
            n_el = int(np.prod(shape))
            return dbuf[off:off + 4 * n_el].view(torch.int32).view(*shape)

        S, MB, bs = len(ctx), self.MB, self.bs
        b = _SplitBatch()
        b.t, b.tables = t, dbuf
        b.pages_used = t.pages_used
        b.cu_host, b.ctx_host = cu, ctx
        b.cu, b.ctx, b.block_table = dv(t.cu_off, (S + 1,)), dv(t.ctx_off, (S,)), dv(t.bt_off, (S, MB))
        b.err = dv(t.err_off, (1,))
        b.block_table_host = self._host_np[t.bt_off:t.bt_off + 4 * S * MB].view(np.int32).reshape(S, MB).copy()
        T = int(cu[-1])
        if self._slots.numel() < T:
            self._slots = torch.empty(max(T, 2 * self._slots.numel()), dtype=torch.int64, device=self.dev)
        b.slots = self._slots[:T]
        b.block_size, b.causal, b.Hkv, b.d, b.MB, b.num_ctas = bs, self.causal, self.Hkv, self.d, MB, self.num_ctas
        b.counters = self._counters

        def ws(i, nbytes):
            if nbytes and self._ws[i].numel() < nbytes:
                self._ws[i] = torch.empty(max(nbytes, 2 * self._ws[i].numel()), dtype=torch.uint8, device=self.dev)
            return self._ws[i] if nbytes else None

        b.tile_ws, b.dec_ws = ws(0, t.tile_workspace_bytes), ws(1, t.dec_workspace_bytes)
        need = t.tile_num_pages * self.Hkv * bs * self.d
        if need and (self._copies is None or self._copies[0].numel() < need):
            self._copies = [torch.empty(max(need, 2 * (self._copies[0].numel() if self._copies else 0)),
                                        dtype=torch.bfloat16, device=self.dev) for _ in range(2)]
        b.copy_k = self._copies[0][:need].view(t.tile_num_pages, self.Hkv, bs, self.d) if need else None
        b.copy_v = self._copies[1][:need].view(t.tile_num_pages, self.Hkv, bs, self.d) if need else None
        b.tile = b.decode = None
        if t.tile_seq_end > t.tile_seq_begin:
            b.tile = dict(seq=(t.tile_seq_begin, t.tile_seq_end), tok=(t.tile_tok_begin, t.tile_tok_end),
                          plan=_Part(dv(t.tile_tasks_off, (t.tile_num_tasks, 8)),
                                     dv(t.tile_merges_off, (t.tile_num_merges, 8)), self.num_ctas, b.tile_ws,
                                     self._counters[0:2]))
        if t.dec_seq_end > t.dec_seq_begin:
            b.decode = dict(seq=(t.dec_seq_begin, t.dec_seq_end), tok=(t.dec_tok_begin, t.dec_tok_end),
                            plan=_Part(dv(t.dec_tasks_off, (t.dec_num_tasks, 8)),
                                       dv(t.dec_merges_off, (t.dec_num_merges, 8)), self.num_ctas, b.dec_ws,
                                       self._counters[2:4]))
        return b


def Fp8SplitBatch(cu_seqlens_q, context_lens, free_list, block_size, max_blocks, num_heads_q, num_heads_kv, head_dim,
                  causal, device="cuda", num_ctas=None):
    """One split step's batch over 8-bit pages (a planner used once; see Fp8SplitPlanner).  The tile
    part computes with K and V rounded to bf16 after dequantization."""
    pl = Fp8SplitPlanner(num_heads_q, num_heads_kv, head_dim, block_size, max_blocks, causal, device=device,
                         num_ctas=num_ctas)
    b = pl.plan(cu_seqlens_q, context_lens, free_list)
    b._planner = pl   # keeps its buffers alive with the batch
    return b


def run_step_fp8_split(batch, q, k_new, v_new, k_pages, v_pages, k_scales, v_scales, scale, out=None, stream=None):
    """One step of a split batch: slot mapping and the quantizing append for the whole batch (one
    launch), then attention_fp8_split."""
    out = torch.empty_like(q) if out is None else out
    xy_kv_append_paged_fp8(k_new, v_new, batch.cu, batch.ctx, batch.block_table, k_pages, v_pages, k_scales, v_scales,
                           batch.err, slot_mapping=batch.slots, stream=stream)
    return attention_fp8_split(batch, q, k_pages, v_pages, k_scales, v_scales, scale, out, stream)


def attention_fp8_split(batch, q, k_pages, v_pages, k_scales, v_scales, scale, out, stream=None):
    """The attention of a split batch: xy_paged_attention_fp8_mixed (page copies and tcgen05 tiles
    for the tile part, the 8-bit decode path for the decode part, each writing its rows of out)."""
    from . import xy_paged_attention_fp8_mixed
    xy_paged_attention_fp8_mixed(q, batch.tables, batch.t, k_pages, v_pages, k_scales, v_scales, len(batch.ctx_host),
                                 batch.MB, scale, batch.causal, batch.num_ctas, batch.copy_k, batch.copy_v,
                                 batch.tile_ws, batch.dec_ws, batch.counters, batch.err, out, stream)
    return out


def check(batch):
    check_err_word(batch.err)
