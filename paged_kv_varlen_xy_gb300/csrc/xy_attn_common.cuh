// Shared pieces of the two attention kernels (mma.sync tiles and tcgen05 tiles): kernel
// parameters, the task prefetch record and the rule that assigns a task to a kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "xy.h"
#include "xy_device.cuh"

namespace xy {

struct AttnParams {
    const __nv_bfloat16 *q;
    const int32_t *cu;
    const int32_t *ctx;
    const int32_t *bt;
    const xy_task *tasks;
    float *ws_o;
    float *ws_lse;
    int32_t *err;
    __nv_bfloat16 *out;
    const float *ksc;  // 8-bit pages: per-row K and V scales [P, Hkv, bs] (null for bf16 pages)
    const float *vsc;
    int *dyn;          // dynamic deal: counter of claimed tasks (null: the static deal)
    unsigned long long *trace;  // per-CTA record {start ns, end ns, tasks run, rows x keys} (null: off)
    int64_t ws_rows;
    int MB, P, S, T, Hq, Hkv, G, bs, causal, num_tasks;
    int kv3d;          // 8-bit pages: K and V codes in one allocation, one 3-D map (kmap) fetches both
    float scale_log2;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A task record plus the per-sequence numbers it needs; fetched one task ahead so that the
// global-load latency overlaps the current task's stages.
struct TaskInfo {
    xy_task t;
    int seq_start, qn, L;
};

__device__ __forceinline__ TaskInfo fetch_info(const xy_task &t, const AttnParams &p) {
    TaskInfo f;
    f.t = t;
    f.seq_start = f.qn = f.L = 0;
    if (t.seq >= 0 && t.seq < p.S) {
        f.seq_start = __ldg(p.cu + t.seq);
        f.qn = __ldg(p.cu + t.seq + 1) - f.seq_start;
        f.L = __ldg(p.ctx + t.seq);
    }
    return f;
}

// Block-table window of a producer warp: lane i holds the physical page of logical page b0 + i of
// sequence `seq` (-1 past the table).
__device__ __forceinline__ int load_window(const AttnParams &p, int seq, int b0, int lane) {
    const int idx = b0 + lane;
    return (idx >= 0 && idx < p.MB) ? __ldg(p.bt + (int64_t)seq * p.MB + idx) : -1;
}

// Dynamic deal: a shared-memory ring of the tasks this CTA has claimed.  A scheduler warp claims
// the next task index of the table with an atomic add on the launch's counter, fetches the record,
// its per-sequence numbers and its first block-table window, and publishes them as entry e in slot
// e % kQueueSlots; every other warp of the CTA reads every entry, in order.  Per slot: full completes when the entry is
// published, empty when all readers have read it, taken when the lead reader (the warp that
// issues the task's first copies) has read it.  Entry e + 1 is claimed once entry e is taken, so a
// CTA holds at most one claimed task beyond the one it is starting.  A lead reader may instead
// defer `taken` until the task it is issuing is nearly done (TaskCursor::defer_taken): the next
// task is then chosen close to the time the CTA needs it, which keeps the deal longest-first
// when a CTA runs only a few tasks.
constexpr int kQueueSlots = 8;
constexpr int kQueueEnd = -2;  // sequence id of the entry that ends the table

struct QueueEntry {
    TaskInfo f;
    int win[32];  // physical pages of logical pages kv_start / bs + 0..31 (-1 past the table)
};

struct TaskQueue {
    QueueEntry *entry;  // [kQueueSlots]
    uint32_t full, empty, taken;  // shared addresses of [kQueueSlots] mbarriers each
    const volatile int *abort;
    static constexpr int kBytes = kQueueSlots * (int)sizeof(QueueEntry) + 3 * kQueueSlots * 8;

    // `at`: kBytes of shared memory, 8-byte aligned (generic pointer and its shared address).
    __device__ void bind(uint8_t *at, uint32_t at_s, const volatile int *abort_flag) {
        full = at_s;
        empty = full + 8 * kQueueSlots;
        taken = empty + 8 * kQueueSlots;
        entry = reinterpret_cast<QueueEntry *>(at + 3 * kQueueSlots * 8);
        abort = abort_flag;
    }
    // one thread, before the CTA's first barrier; `readers`: arrivals that free a slot
    __device__ void init(int readers) const {
        for (int e = 0; e < kQueueSlots; ++e) {
            mbar_init(full + 8 * e, 1);
            mbar_init(empty + 8 * e, readers);
            mbar_init(taken + 8 * e, 1);
        }
    }
    // Scheduler warp: claim a task and publish it as entry e.  Returns 1 (a task), 0 (the end of
    // the table was published) or -1 (a wait gave up; nothing published).
    __device__ int publish(int e, const AttnParams &p, int *counter, int lane) const {
        bool ok = true;
        if (e >= 1)  // the lead reader has started entry e - 1
            ok = mbar_wait(taken + 8 * ((e - 1) % kQueueSlots), ((e - 1) / kQueueSlots) & 1, abort);
        if (ok && e >= kQueueSlots)  // every reader is done with the slot's previous entry
            ok = mbar_wait(empty + 8 * (e % kQueueSlots), ((e / kQueueSlots) - 1) & 1, abort);
        if (!__all_sync(0xffffffffu, ok)) return -1;
        int idx = 0;
        if (lane == 0) idx = atomicAdd(counter, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        QueueEntry &q = entry[e % kQueueSlots];
        const int r = idx < p.num_tasks ? 1 : 0;
        if (r) {
            // lanes 0..7 load one word of the record each
            const int w = lane < 8 ? __ldg(reinterpret_cast<const int32_t *>(p.tasks + idx) + lane) : 0;
            xy_task t;
            t.seq = __shfl_sync(0xffffffffu, w, 0);
            t.kv_head = __shfl_sync(0xffffffffu, w, 1);
            t.q_start = __shfl_sync(0xffffffffu, w, 2);
            t.q_rows = __shfl_sync(0xffffffffu, w, 3);
            t.kv_start = __shfl_sync(0xffffffffu, w, 4);
            t.kv_end = __shfl_sync(0xffffffffu, w, 5);
            t.num_splits = __shfl_sync(0xffffffffu, w, 6);
            t.ws_row = __shfl_sync(0xffffffffu, w, 7);
            const TaskInfo f = fetch_info(t, p);
            const bool seq_ok = t.seq >= 0 && t.seq < p.S && t.kv_start >= 0;
            q.win[lane] = seq_ok ? load_window(p, t.seq, t.kv_start / p.bs, lane) : -1;
            if (lane == 0) q.f = f;
        } else if (lane == 0) {
            q.f.t = xy_task{kQueueEnd, 0, 0, 0, 0, 0, 0, -1};
            q.f.seq_start = q.f.qn = q.f.L = 0;
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(full + 8 * (e % kQueueSlots));  // release: readers see the entry
        return r;
    }
    // Scheduler warp, after its last claim (whatever the reason it stopped): counter[1] counts the
    // CTAs done claiming; the last one returns both words to zero for the next launch.
    __device__ static void finish(int *counter, int lane) {
        if (lane == 0) {
            __threadfence();  // this CTA's claims come before its count
            if (atomicAdd(counter + 1, 1) == (int)gridDim.x - 1) {
                atomicExch(counter, 0);
                atomicExch(counter + 1, 0);
            }
        }
        __syncwarp();
    }
};

// Walks this CTA's tasks.  Static deal: positions blockIdx.x, +gridDim.x, ... of the table, the
// next task's record and per-sequence numbers fetched while the current one runs.  Dynamic deal
// (attach() with a queue): the entries of the CTA's TaskQueue, in order.
struct TaskCursor {
    int ti;
    bool have, have_next, nxt_ready;
    TaskInfo cur, nxt;
    xy_task rec_next;
    // dynamic deal
    const TaskQueue *dq = nullptr;
    int read = 0;
    int win = -1;  // this lane's page of the entry's first block-table window (whole-warp readers)
    bool single = false, lead = false, failed = false;
    bool defer_taken = false;  // lead reader: `taken` waits for release_claim() (or the next read)
    int pend = -1;             // slot whose `taken` arrival is deferred
    volatile int *votes = nullptr;  // [2][vote_n]: a group of warps that agree on every read
    int vote_bar = 0, vote_n = 0, vote_i = 0;

    // q: the queue (null: static deal).  single: only the calling thread reads (else the whole
    // warp).  lead: this reader signals `taken`.  votes/bar/n/i: the reader is warp i of n that
    // pass named barrier `bar` together, so they vote on each read (a read that gave up in one
    // of them stops all of them) and no warp is left waiting at that barrier.
    __device__ void attach(const TaskQueue *q, bool single_thread, bool lead_reader, volatile int *vote_words = nullptr,
                           int bar = 0, int n = 0, int i = 0) {
        dq = q;
        single = single_thread;
        lead = lead_reader;
        votes = vote_words;
        vote_bar = bar;
        vote_n = n;
        vote_i = i;
    }
    // A deferring lead reader lets the scheduler claim the next task.  Idempotent per entry.
    __device__ void release_claim() {
        if (pend >= 0) {
            if (single || (threadIdx.x & 31) == 0) mbar_arrive(dq->taken + 8 * pend);
            pend = -1;
        }
    }
    __device__ void read_entry() {
        release_claim();  // an entry is always taken before the next one is read
        const int s = read % kQueueSlots;
        bool ok = mbar_wait(dq->full + 8 * s, (read / kQueueSlots) & 1, dq->abort);
        if (!single) ok = __all_sync(0xffffffffu, ok);
        int r = -1;
        if (ok) {
            cur = dq->entry[s].f;
            if (!single) {
                win = dq->entry[s].win[threadIdx.x & 31];
                __syncwarp();
            }
            if (single || (threadIdx.x & 31) == 0) {
                mbar_arrive(dq->empty + 8 * s);
                if (lead && !defer_taken) mbar_arrive(dq->taken + 8 * s);
            }
            if (lead && defer_taken) pend = s;
            r = cur.t.seq == kQueueEnd ? 0 : 1;
        }
        ++read;
        if (votes) {
            volatile int *v = votes + (read & 1) * vote_n;
            if ((threadIdx.x & 31) == 0) v[vote_i] = r;
            named_bar_sync(vote_bar, vote_n * 32);
            for (int k = 0; k < vote_n; ++k) r = min(r, v[k]);
        }
        have = r == 1;
        failed = r < 0;
        have_next = nxt_ready = false;
    }
    __device__ void begin(const AttnParams &p) {
        if (dq) {
            read_entry();
            return;
        }
        ti = blockIdx.x;
        have = ti < p.num_tasks;
        if (have) cur = fetch_info(p.tasks[ti], p);
    }
    __device__ void load_next_record(const AttnParams &p) {
        if (dq) return;  // the next entry is not known before it is read
        const int tn = ti + gridDim.x;
        have_next = tn < p.num_tasks;
        if (have_next) rec_next = p.tasks[tn];
        nxt_ready = false;
    }
    __device__ void prefetch_next(const AttnParams &p) {
        if (have_next && !nxt_ready) {
            nxt = fetch_info(rec_next, p);
            nxt_ready = true;
        }
    }
    __device__ void advance(const AttnParams &p) {
        if (dq) {
            read_entry();
            return;
        }
        prefetch_next(p);
        cur = nxt;
        ti += gridDim.x;
        have = have_next;
    }
};

// A hole record of a greedy deal (a position its CTA does not use): every role skips it.
__device__ __forceinline__ bool is_hole(const xy_task &t) { return t.seq == -1 && t.q_rows == 0; }

// Checks every kernel applies to a task before touching memory through it.
__device__ __forceinline__ bool task_common_ok(const TaskInfo &f, const AttnParams &p) {
    const xy_task &t = f.t;
    if (t.seq < 0 || t.seq >= p.S || t.kv_head < 0 || t.kv_head >= p.Hkv) return false;
    if (t.q_rows < 1 || t.q_start < 0) return false;
    if (t.kv_start < 0 || t.kv_start >= t.kv_end) return false;
    if (f.qn < 1 || f.qn > f.L || t.q_start + t.q_rows > f.qn || t.kv_end > f.L) return false;
    if (t.num_splits > 1 && (t.ws_row < 0 || (int64_t)t.ws_row + (int64_t)t.q_rows * p.G > p.ws_rows))
        return false;
    return true;
}

// Tasks with more than this many (token, head) rows run on the tcgen05 tile kernel.
#ifndef XY_TILE_MIN_ROWS
#define XY_TILE_MIN_ROWS 16
#endif

// The tcgen05 tile kernel handles head_dim 128 when G divides 128 (a query box is G heads x
// 128/G tokens); it takes the tasks with more than XY_TILE_MIN_ROWS rows.
__host__ __device__ __forceinline__ bool tile_shape_ok(int G, int head_dim) {
    return head_dim == 128 && (128 % G) == 0;
}
__host__ __device__ __forceinline__ bool is_tile_task(const xy_task &t, int G, int head_dim) {
    return tile_shape_ok(G, head_dim) && t.q_rows * G > XY_TILE_MIN_ROWS;
}

// Per-device "done" marks for once-per-device kernel setup (function attributes are set per
// device): bit d of the word is device d's (devices past 63 set up on every call).
struct PerDeviceOnce {
    unsigned long long bits = 0;
    __host__ bool done(int dev) const {
        return dev >= 0 && dev < 64 && (__atomic_load_n(&bits, __ATOMIC_ACQUIRE) >> dev & 1ull);
    }
    __host__ void mark(int dev) {
        if (dev >= 0 && dev < 64) __atomic_fetch_or(&bits, 1ull << dev, __ATOMIC_RELEASE);
    }
};

// Records a CUDA error for xy_last_error_string() and returns XY_ERR_CUDA.
xy_status cuda_fail(cudaError_t e, const char *what);

// Launches the unified kernel (xy_tile.cu): tcgen05 tiles for tasks of more than
// XY_TILE_MIN_ROWS rows, the decode path for the others, one persistent launch over the task
// table.  kmap_d / vmap_d are the decode path's 3-D page-pool maps.
xy_status launch_meta_attention(const AttnParams &p, const void *k_pages, const void *v_pages, int num_pages,
                                int block_size, int num_ctas, const CUtensorMap &kmap_d, const CUtensorMap &vmap_d,
                                cudaStream_t st);

}  // namespace xy
