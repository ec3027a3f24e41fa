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

// A task belongs to the tcgen05 tile kernel when its rows fill a good part of a 128-row MMA
// tile: head_dim 128, G divides 128 (the query box is G heads x 128/G tokens), more than 16 rows.
__host__ __device__ __forceinline__ bool is_tile_task(const xy_task &t, int G, int head_dim) {
    return head_dim == 128 && (128 % G) == 0 && t.q_rows * G > 16;
}

// Records a CUDA error for xy_last_error_string() and returns XY_ERR_CUDA.
xy_status cuda_fail(cudaError_t e, const char *what);

// Launches the tcgen05 tile kernel over the tasks it owns (defined in xy_tile.cu).
xy_status launch_tile_attention(const AttnParams &p, const void *k_pages, const void *v_pages, int num_pages,
                                int block_size, int num_ctas, cudaStream_t st);

}  // namespace xy
