// Shared pieces of the two attention kernels (mma.sync tiles and tcgen05 tiles): kernel
// parameters, the task prefetch record and the rule that assigns a task to a kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "xy.h"

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
    int64_t ws_rows;
    int MB, P, S, T, Hq, Hkv, G, bs, causal, num_tasks;
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

// Walks this CTA's tasks (blockIdx.x, +gridDim.x, ...), fetching the next task's record and
// per-sequence numbers while the current one runs.
struct TaskCursor {
    int ti;
    bool have, have_next, nxt_ready;
    TaskInfo cur, nxt;
    xy_task rec_next;

    __device__ void begin(const AttnParams &p) {
        ti = blockIdx.x;
        have = ti < p.num_tasks;
        if (have) cur = fetch_info(p.tasks[ti], p);
    }
    __device__ void load_next_record(const AttnParams &p) {
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
        prefetch_next(p);
        cur = nxt;
        ti += gridDim.x;
        have = have_next;
    }
};

// Block-table window of a producer warp: lane i holds the physical page of logical page b0 + i of
// sequence `seq` (-1 past the table).
__device__ __forceinline__ int load_window(const AttnParams &p, int seq, int b0, int lane) {
    const int idx = b0 + lane;
    return (idx >= 0 && idx < p.MB) ? __ldg(p.bt + (int64_t)seq * p.MB + idx) : -1;
}

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

// Records a CUDA error for xy_last_error_string() and returns XY_ERR_CUDA.
xy_status cuda_fail(cudaError_t e, const char *what);

// Launches the unified kernel (xy_tile.cu): tcgen05 tiles for tasks of more than
// XY_TILE_MIN_ROWS rows, the decode path for the others, one persistent launch over the task
// table.  kmap_d / vmap_d are the decode path's 3-D page-pool maps.
xy_status launch_meta_attention(const AttnParams &p, const void *k_pages, const void *v_pages, int num_pages,
                                int block_size, int num_ctas, const CUtensorMap &kmap_d, const CUtensorMap &vmap_d,
                                cudaStream_t st);

}  // namespace xy
