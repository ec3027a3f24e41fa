// a5..a10: paged attention over the task table (QK^T on block-table-gathered pages, virtual +
// causal mask, online softmax, PV, store or split partials) and the split-KV merge.
//
// "XY-Serve 深度实战" (chenxutan.com/d/5031) §2.2 component 3 (Meta-Attention: one
// GEMM-softmax-GEMM kernel driven by a task table, no prefill/decode distinction) and §2.3
// technique 1 (virtual padding: ragged tiles are masked on chip, only valid outputs stored);
// cann-recipes-infer notes (dpshk.com/news/5336026) §3.3 (packed paged_attention with
// cu_seqlens and a page table, is_causal).
//
// Design (GB300): one persistent CTA per SM walks its share of the load-sorted task table
// (tasks blockIdx.x, blockIdx.x + gridDim.x, ...).  A producer warp gathers each 64-key stage
// of K and V with 2-D TMA tiled loads -- one box per (page, 64-column half), rows addressed as
// (physical_page * Hkv + kv_head) * bs + offset -- into a ring of shared-memory stages with
// 128-byte swizzle, so the fragment loads below are bank-conflict free.  Four math warps own
// 16-row slices of the task's (token, head) rows; QK^T and PV run on m16n8k16 tensor-core
// fragments, the softmax on the accumulator registers with quad shuffles.  When a task has
// fewer rows than warps x 16, the warps split the stage's keys instead and merge their
// (max, sum, O) triples through shared memory at the end of the task.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>
#include <vector>

#include "xy.h"
#include "xy_device.cuh"
#include "xy_attn_common.cuh"
#include "xy_decode_path.cuh"

namespace {

using xy::AttnParams;
using xy::ex2;
using xy::TaskCursor;
using xy::TaskInfo;
using xy::dec::kMathWarps;

// Stand-alone decode-path kernel: one persistent CTA per SM, four math warps and two producer
// warps that issue alternate stages (xy_decode_path.cuh).  Issuing a stage -- block-table window
// lookup, eight page boxes, barrier bookkeeping -- costs a producer warp about as long as the math
// warps need to consume one, so two producers keep the ring ahead of the math.  It runs every
// task when the tcgen05 tile kernel cannot (head_dim 64, or G not dividing 128), pure decode
// batches, and every batch over 8-bit pages; tasks then have at most 64 rows.
//
// Page formats (KIND): kBf16; kFp8Narrow, 8-bit pages in pure decode batches with G <= 16 (tasks
// of at most 16 rows); kFp8Wide, 8-bit pages otherwise (up to 64 rows per task, so that a
// prefill or chunk task shares each K/V stage among 64 rows).  8-bit stages hold 128 keys (about
// the bytes of a 64-key bf16 stage); with 16-token pages that is 32 copies per stage (codes and
// scales of 8 pages), so four producer warps, one per ring slot, keep the ring ahead.
enum Kind { kBf16 = 0, kFp8Narrow = 1, kFp8Wide = 2, kFp8Tiny = 3, kBf16Tiny = 4 };

template <int HD, int KIND, bool DYN = false>
struct Cfg {
    using RG = typename std::conditional<
        KIND == kFp8Tiny, xy::dec::RingF8<2, 16, 128, true>,
        typename std::conditional<KIND == kFp8Narrow, xy::dec::RingF8<4, 16>,
        typename std::conditional<KIND == kFp8Wide, xy::dec::RingF8<4, 16 * kMathWarps>,
        typename std::conditional<KIND == kBf16Tiny, xy::dec::Ring<HD, 2, 16>,
                                  xy::dec::Ring<HD, HD == 128 ? 4 : 6, 16 * kMathWarps>>::type>::type>::type>::type;
    static constexpr int kProducers = KIND == kFp8Narrow || KIND == kFp8Wide ? 4 : 2;
    // kFp8Tiny, kBf16Tiny: half-size CTAs (two stages, two producers, tasks of at most 16 rows;
    // over 8-bit pages the transposed products only), two per SM
    static constexpr int kMinBlocks = KIND == kFp8Tiny || KIND == kBf16Tiny ? 2 : 1;
    static_assert(RG::kStages >= kProducers, "every producer owns a ring slot");
    // math warps, producer warps, then (dynamic deal over bf16 pages) the scheduler warp.  Over
    // 8-bit pages a ninth warp would put three warps on one SM sub-partition and cap the registers
    // at 168, so there the first producer warp claims the tasks itself.
    static constexpr bool kSchedWarpUsed = DYN && KIND == kBf16;
    static constexpr bool kInlineClaims = DYN && KIND != kBf16;
    static constexpr int kSchedWarp = kMathWarps + kProducers;
    static constexpr int kThreads = (kSchedWarp + (kSchedWarpUsed ? 1 : 0)) * 32;
    static constexpr int kStagesOff = 0;
    static constexpr int kSlotsOff = RG::kBytes;
    static constexpr int kBarOff = kSlotsOff + RG::kSlotBytes;
    static constexpr int kFlagOff = kBarOff + 2 * RG::kStages * 8;  // abort flag + 2 x 4 vote words
    static constexpr int kQueueVoteOff = kFlagOff + 64;             // 2 x 4 queue-read votes
    static constexpr int kQueueOff = kQueueVoteOff + 32;
    static constexpr int kSmemBytes = kQueueOff + xy::TaskQueue::kBytes + 1024;  // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
};

template <int HD, int KIND, bool DYN>
__global__ void __launch_bounds__(Cfg<HD, KIND, DYN>::kThreads, Cfg<HD, KIND, DYN>::kMinBlocks)
    paged_attention_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const __grid_constant__ CUtensorMap ksmap, const __grid_constant__ CUtensorMap vsmap,
                           const AttnParams p) {
    using C = Cfg<HD, KIND, DYN>;
    using RG = typename C::RG;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = xy::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    xy::dec::Smem sm;
    sm.stages = base + C::kStagesOff;
    sm.stages_gen = gbase + C::kStagesOff;
    sm.slots = reinterpret_cast<float *>(gbase + C::kSlotsOff);
    sm.full_bar = base + C::kBarOff;
    sm.empty_bar = sm.full_bar + RG::kStages * 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::kFlagOff);
    sm.abort_flag = abort_flag;
    sm.vote = abort_flag + 4;  // [2][kMathWarps], indexed by task parity
    sm.bar_id = 1;
    // dynamic deal: every math and producer warp reads every entry of the claim queue
    xy::TaskQueue dq;
    dq.bind(gbase + C::kQueueOff, base + C::kQueueOff, abort_flag);
    const xy::TaskQueue *q = DYN ? &dq : nullptr;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < RG::kStages; ++s) {
            xy::mbar_init(sm.full_bar + 8 * s, 1);
            xy::mbar_init(sm.empty_bar + 8 * s, kMathWarps);
        }
        if (DYN) dq.init(kMathWarps + C::kProducers);
        *abort_flag = 0;
        xy::fence_mbarrier_init();
    }
    __syncthreads();
    // Under a dependent launch this kernel may run while the kernel ahead of it on the stream (the
    // step's KV append) still writes the new tokens' K/V rows: only the producer warps wait for it,
    // each before its first copy of such rows (xy::dec::produce_task); everything else read here
    // is not written by the append.
    if (p.trace && threadIdx.x == 0) p.trace[4 * blockIdx.x] = xy::global_timer_ns();

    if constexpr (C::kSchedWarpUsed) {
        if (warp == C::kSchedWarp) {
            // ---------------------------- scheduler (dynamic deal) ----------------------------
            int r = 1;
            for (int e = 0; r == 1; ++e) r = dq.publish(e, p, p.dyn, lane);
            dq.finish(p.dyn, lane);
            if (r < 0) {
                if (lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            return;
        }
    }
    if (warp >= kMathWarps) {
        // ------------------------------ producer warps ------------------------------
        const int pw = warp - kMathWarps;
        if (lane == 0) {
            xy::prefetch_tensormap(&kmap);
            xy::prefetch_tensormap(&vmap);
        }
        int ctr = 0, pref_win = -1;
        bool ok = true, pref_valid = false, dep_ready = false;
        // inline claims (8-bit pages): producer warp 0 claims task k + 1 once it has issued its
        // first stage of task k (so the claim overlaps the copies), or as it leaves task k
        const bool claims = C::kInlineClaims && pw == 0;
        int published = 0;
        bool claims_done = !claims, claimed = true;
        auto claim_next = [&]() {
            if (claims_done || claimed) return;
            claimed = true;
            const int r = dq.publish(published++, p, p.dyn, lane);
            if (r <= 0) claims_done = true;
            if (r < 0) ok = false;
        };
        if (claims) {
            claimed = false;
            claim_next();   // entry 0
        }
        TaskCursor tc;
        tc.attach(q, false, pw == 0);
        tc.begin(p);
        while (tc.have && ok) {
            tc.load_next_record(p);
            claimed = false;
            if (xy::is_hole(tc.cur.t)) {
                claim_next();
                pref_valid = false;
                tc.advance(p);
                continue;
            }
            if (!xy::dec::task_ok<RG>(tc.cur, p)) {
                if (lane == 0 && pw == 0) xy::set_err(p.err, XY_DEV_BAD_TASK);
                claim_next();
                pref_valid = false;
                tc.advance(p);
                continue;
            }
            const TaskInfo f = tc.cur;
            // the first block-table window: prefetched with the task (static deal) or in its entry
            const bool have_first = DYN || pref_valid;
            const int first_win = DYN ? tc.win : pref_win;
            pref_valid = false;
            ok = xy::dec::produce_task<HD, RG>(
                p, f, &kmap, &vmap, &ksmap, &vsmap, sm, ctr, lane, first_win, have_first, dep_ready,
                [&]() {
                    // the next record has arrived by now: prefetch its numbers and first window
                    tc.prefetch_next(p);
                    if (tc.have_next) {
                        const xy_task &tn = tc.nxt.t;
                        pref_valid = tn.seq >= 0 && tn.seq < p.S && tn.kv_start >= 0;
                        if (pref_valid) pref_win = xy::load_window(p, tn.seq, tn.kv_start / p.bs, lane);
                    }
                    claim_next();
                },
                pw, C::kProducers) && ok;
            claim_next();   // (no stage of the task fell to this warp)
            tc.advance(p);
        }
        if (claims) dq.finish(p.dyn, lane);
        if (!ok || tc.failed) {
            if (lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
            *abort_flag = 1;
        }
        // every stage this warp issued must have landed before the CTA may exit
        xy::dec::drain<RG>(sm, ctr, pw, C::kProducers);
        return;
    }

    // ------------------------------ math warps ------------------------------
    int ctr = 0, iter = 0;
    unsigned long long n_run = 0, work = 0;  // trace: tasks run and their rows x keys
    TaskCursor tc;
    // the math warps pass named barriers together (consume_task), so they vote on each queue read
    tc.attach(q, false, false, reinterpret_cast<volatile int *>(gbase + C::kQueueVoteOff), sm.bar_id, kMathWarps,
              warp);
    tc.begin(p);
    while (tc.have) {
        tc.load_next_record(p);
        if (xy::is_hole(tc.cur.t) || !xy::dec::task_ok<RG>(tc.cur, p)) {
            tc.advance(p);
            continue;
        }
        const TaskInfo f = tc.cur;
        if (!xy::dec::consume_task<HD, RG>(p, f, sm, ctr, iter, warp, lane, [&]() { tc.prefetch_next(p); })) {
            *abort_flag = 1;
            if (warp == 0 && lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
            return;
        }
        ++n_run;
        work += (unsigned long long)(f.t.q_rows * p.G) * (unsigned long long)(f.t.kv_end - f.t.kv_start);
        tc.advance(p);
    }
    if (tc.failed) {
        *abort_flag = 1;
        if (warp == 0 && lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
        return;
    }
    // the math warps finish last: math warp 0 closes the CTA's trace record
    if (p.trace && warp == 0 && lane == 0) {
        unsigned long long *r = p.trace + 4 * blockIdx.x;
        r[1] = xy::global_timer_ns();
        r[2] = n_run;
        r[3] = work;
    }
}

// Split-KV merge: for each split tile, out = sum_c 2^(lse_c - M) O_c / sum_c 2^(lse_c - M).
// Grid (merge records, kCombineY): one warp per (token, head) row, kCombineY x 8 rows of a merge
// in flight, lanes across head_dim.  Lane c of a warp turns split c's lse into its weight, so the
// O rows of all splits load independently (no dependent chain per split).
constexpr int kCombineY = 8;

template <int HD>
__global__ void __launch_bounds__(256) combine_kernel(const xy_merge *__restrict__ merges, const float *__restrict__ ws_o,
                                                      const float *__restrict__ ws_lse, const int32_t *__restrict__ cu,
                                                      int Hq, int G, int64_t ws_rows, int32_t *err,
                                                      __nv_bfloat16 *__restrict__ out) {
    const xy_merge m = merges[blockIdx.x];
    const int R = m.q_rows * G;
    const int ns = m.num_splits;
    if (ns < 2 || m.ws_row < 0 || (int64_t)m.ws_row + (int64_t)ns * R > ws_rows) {
        if (threadIdx.x == 0 && blockIdx.y == 0) xy::set_err(err, XY_DEV_BAD_TASK);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int V = HD / 32;  // floats per lane
    const int seq_start = __ldg(cu + m.seq);
    const int64_t base = m.ws_row;
    for (int r = blockIdx.y * 8 + warp; r < R; r += kCombineY * 8) {
        float M = -INFINITY;
        for (int c = lane; c < ns; c += 32) M = fmaxf(M, __ldg(ws_lse + base + (int64_t)c * R + r));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float U = M == -INFINITY ? 0.f : M;
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
        float W = 0.f;
        for (int c0 = 0; c0 < ns; c0 += 32) {
            const int c = c0 + lane;
            const float wl = c < ns ? ex2(__ldg(ws_lse + base + (int64_t)c * R + r) - U) : 0.f;
            W += wl;
            const int nc = min(32, ns - c0);
#pragma unroll 4
            for (int k = 0; k < nc; ++k) {
                const float w = __shfl_sync(0xffffffffu, wl, k);
                const float *src = ws_o + (base + (int64_t)(c0 + k) * R + r) * HD + lane * V;
                if (V == 4) {
                    const float4 x = __ldg(reinterpret_cast<const float4 *>(src));
                    acc[0] += w * x.x;
                    acc[1] += w * x.y;
                    acc[2] += w * x.z;
                    acc[3] += w * x.w;
                } else {
                    const float2 x = __ldg(reinterpret_cast<const float2 *>(src));
                    acc[0] += w * x.x;
                    acc[1] += w * x.y;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
        const float inv = W > 0.f ? 1.f / W : 0.f;
        const int64_t tok = seq_start + m.q_start + r / G;
        const int h = m.kv_head * G + r % G;
        __nv_bfloat16 *dst = out + (tok * Hq + h) * HD + lane * V;
#pragma unroll
        for (int v = 0; v < V; v += 2)
            *reinterpret_cast<uint32_t *>(dst + v) = xy::pack_bf16x2(acc[v] * inv, acc[v + 1] * inv);
    }
}

// ---------------------------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 3-D map over a page pool viewed as [P * Hkv * bs rows, head_dim] bf16, with the two 64-column
// halves of a row as the outer dimension: dims (64 columns, rows, head_dim / 64 halves), strides
// (head_dim * 2 bytes per row, 128 bytes per half).  A box of (64, box_rows, halves) lands in
// shared memory as [half][box_rows][128 B] with the 128-byte swizzle.
bool make_pool_map(CUtensorMap *map, const void *pool, int64_t rows, int head_dim, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int halves = head_dim / 64;
    cuuint64_t dims[3] = {64u, (cuuint64_t)rows, (cuuint64_t)halves};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, 128u};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, (cuuint32_t)halves};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over an 8-bit page pool viewed as [P * Hkv * bs rows, 128 bytes] (head_dim 128): a box of
// (128, box_rows) lands in shared memory as [box_rows][128 B] with the 128-byte swizzle.
bool make_pool_map_u8(CUtensorMap *map, const void *pool, int64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {128u, (cuuint64_t)rows};
    cuuint64_t strides[1] = {128u};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over K and V 8-bit pools in one allocation, the V pool kv_gap bytes after the K pool:
// (128 bytes, rows, K|V); a box (128, box_rows, 2) lands as [K rows][V rows], each [box_rows][128 B]
// with the 128-byte swizzle.
bool make_pool_map_u8_kv(CUtensorMap *map, const void *k_pool, int64_t rows, int box_rows, uint64_t kv_gap) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {128u, (cuuint64_t)rows, 2u};
    cuuint64_t strides[2] = {128u, (cuuint64_t)kv_gap};
    cuuint32_t box[3] = {128u, (cuuint32_t)box_rows, 2u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(k_pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over an 8-bit pool's scale array viewed as [pages * Hkv rows, bs floats]: a box is one
// (page, head) row of bs scales, one row high, for TMA gathers of four pages' rows at a time.
bool make_scale_map(CUtensorMap *map, const float *scales, int64_t rows, int block_size) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int box = block_size < 256 ? block_size : 256;   // (a box dimension is at most 256)
    cuuint64_t dims[2] = {(cuuint64_t)block_size, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)block_size * 4u};
    cuuint32_t bx[2] = {(cuuint32_t)box, 1u};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(scales), dims, strides, bx, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ksm / vsm: the 8-bit pages' scale maps (any valid map for bf16 pages, which do not read them)
template <int HD, int KIND, bool DYN>
xy_status launch_attention_kernel(const AttnParams &p, const CUtensorMap &km, const CUtensorMap &vm,
                                  const CUtensorMap &ksm, const CUtensorMap &vsm, int num_ctas, cudaStream_t st) {
    using C = Cfg<HD, KIND, DYN>;
    static xy::PerDeviceOnce configured;  // the attribute is per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return XY_ERR_CUDA;
    if (!configured.done(dev)) {
        const cudaError_t e = cudaFuncSetAttribute(paged_attention_kernel<HD, KIND, DYN>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return xy::cuda_fail(e, "paged_attention_kernel smem attribute");
        configured.mark(dev);
    }
    const cudaError_t e = xy::launch_dependent(paged_attention_kernel<HD, KIND, DYN>, dim3(num_ctas),
                                               dim3(C::kThreads), C::kSmemBytes, st, km, vm, ksm, vsm, p);
    return e == cudaSuccess ? XY_OK : xy::cuda_fail(e, "paged_attention_kernel launch");
}

template <int HD, int KIND>
xy_status launch(const AttnParams &p, const CUtensorMap &km, const CUtensorMap &vm, const CUtensorMap &ksm,
                 const CUtensorMap &vsm, int num_ctas, const xy_merge *merges, int num_merges, cudaStream_t st) {
    if (p.num_tasks > 0) {
        const xy_status ks = p.dyn ? launch_attention_kernel<HD, KIND, true>(p, km, vm, ksm, vsm, num_ctas, st)
                                   : launch_attention_kernel<HD, KIND, false>(p, km, vm, ksm, vsm, num_ctas, st);
        if (ks != XY_OK) return ks;
    }
    if (num_merges > 0) {
        combine_kernel<HD><<<dim3(num_merges, kCombineY), 256, 0, st>>>(merges, p.ws_o, p.ws_lse, p.cu, p.Hq, p.G,
                                                                        p.ws_rows, p.err, p.out);
        if (cudaGetLastError() != cudaSuccess) return XY_ERR_CUDA;
    }
    return XY_OK;
}

}  // namespace

namespace xy {
void set_last_error(const char *what, const char *msg);
xy_status cuda_fail(cudaError_t e, const char *what) {
    set_last_error(what, cudaGetErrorString(e));
    return XY_ERR_CUDA;
}
}  // namespace xy

extern "C" int xy_default_num_ctas(int device) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return XY_ERR_CUDA;
    return sms;  // one persistent CTA per SM
}

namespace {

// Argument checks shared by both page formats, and the kernel parameters they give.
xy_status make_params(const void *q, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                      const int32_t *block_table, int max_blocks, const void *k_pages, const void *v_pages,
                      int num_pages, int num_seqs, int num_tokens, int num_heads_q, int num_heads_kv, int head_dim,
                      int block_size, float scale, int causal, const xy_task *tasks, int num_tasks,
                      const xy_merge *merges, int num_merges, int num_ctas, void *workspace, size_t workspace_bytes,
                      int32_t *err_word, void *out, AttnParams *pp) {
    if (!q || !cu_seqlens_q || !context_lens || !block_table || !k_pages || !v_pages || !tasks || !out ||
        !err_word || num_ctas < 1 || max_blocks < 1 || num_pages < 1 || num_seqs < 1 || num_heads_kv < 1 ||
        num_heads_q < num_heads_kv || num_heads_q % num_heads_kv)
        return XY_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out)) return XY_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return XY_ERR_UNSUPPORTED;
    if (block_size < 16 || block_size > 256 || (block_size & (block_size - 1))) return XY_ERR_UNSUPPORTED;
    if (num_merges > 0 && (!merges || !workspace || !aligned16(workspace))) return XY_ERR_WORKSPACE;
    if ((int64_t)num_pages * num_heads_kv * block_size > INT32_MAX) return XY_ERR_UNSUPPORTED;

    AttnParams &p = *pp;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.cu = cu_seqlens_q;
    p.ctx = context_lens;
    p.bt = block_table;
    p.tasks = tasks;
    p.ws_rows = workspace ? (int64_t)(workspace_bytes / ((size_t)(head_dim + 1) * 4)) : 0;
    p.ws_o = static_cast<float *>(workspace);
    p.ws_lse = workspace ? static_cast<float *>(workspace) + p.ws_rows * head_dim : nullptr;
    p.err = err_word;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.ksc = nullptr;
    p.vsc = nullptr;
    p.dyn = nullptr;
    p.trace = nullptr;
    p.kv3d = 0;
    p.MB = max_blocks;
    p.P = num_pages;
    p.S = num_seqs;
    p.T = num_tokens;
    p.Hq = num_heads_q;
    p.Hkv = num_heads_kv;
    p.G = num_heads_q / num_heads_kv;
    p.bs = block_size;
    p.causal = causal ? 1 : 0;
    p.num_tasks = num_tasks;
    p.scale_log2 = scale * 1.4426950408889634f;
    return XY_OK;
}

}  // namespace

namespace {

// xy_paged_attention; the dynamic deal when task_counter is given; the per-CTA trace of
// xy_paged_attention_traced when cta_trace is given.
xy_status attention(const void *q, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                    const int32_t *block_table, int max_blocks, const void *k_pages, const void *v_pages,
                    int num_pages, int num_seqs, int num_tokens, int num_heads_q, int num_heads_kv, int head_dim,
                    int block_size, float scale, int causal, const xy_task *tasks, int num_tasks,
                    const xy_merge *merges, int num_merges, int num_ctas, void *workspace, size_t workspace_bytes,
                    int32_t *task_counter, uint64_t *cta_trace, int32_t *err_word, void *out, void *stream) {
    if (num_tasks < 0 || num_merges < 0 || num_seqs < 0 || num_tokens < 0) return XY_ERR_INVALID_ARG;
    if (num_tasks == 0 && num_merges == 0) return XY_OK;
    if (task_counter && (reinterpret_cast<uintptr_t>(task_counter) & 7)) return XY_ERR_INVALID_ARG;
    if (cta_trace && (reinterpret_cast<uintptr_t>(cta_trace) & 7)) return XY_ERR_INVALID_ARG;
    AttnParams p;
    const xy_status ps = make_params(q, cu_seqlens_q, context_lens, block_table, max_blocks, k_pages, v_pages,
                                     num_pages, num_seqs, num_tokens, num_heads_q, num_heads_kv, head_dim,
                                     block_size, scale, causal, tasks, num_tasks, merges, num_merges, num_ctas,
                                     workspace, workspace_bytes, err_word, out, &p);
    if (ps != XY_OK) return ps;
    p.dyn = reinterpret_cast<int *>(task_counter);
    p.trace = reinterpret_cast<unsigned long long *>(cta_trace);

    const int64_t rows = (int64_t)num_pages * num_heads_kv * block_size;
    const int box_rows = block_size < xy::dec::kStageKeys ? block_size : xy::dec::kStageKeys;
    CUtensorMap km, vm;
    if (!make_pool_map(&km, k_pages, rows, head_dim, box_rows) ||
        !make_pool_map(&vm, v_pages, rows, head_dim, box_rows))
        return XY_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // A batch of one new token per sequence with G <= XY_TILE_MIN_ROWS has only decode-path tasks:
    // the stand-alone decode kernel (more registers, deeper stages) runs it.  Any other batch the
    // tile kernel can take goes to the unified kernel.
    const bool pure_decode = num_tokens == num_seqs && p.G <= XY_TILE_MIN_ROWS;
    if (xy::tile_shape_ok(p.G, head_dim) && !pure_decode) {
        // one launch of the unified kernel runs every task (tcgen05 tiles and decode path) ...
        if (num_tasks > 0) {
            const xy_status ts =
                xy::launch_meta_attention(p, k_pages, v_pages, num_pages, block_size, num_ctas, km, vm, st);
            if (ts != XY_OK) return ts;
        }
        p.num_tasks = 0;  // ... so only the split-KV merge remains
    }
    // pure decode under the dynamic deal: two half-size CTAs per SM slot (a traced launch keeps
    // one CTA per slot, one trace record each)
    if (pure_decode && p.dyn && !p.trace)
        return head_dim == 128 ? launch<128, kBf16Tiny>(p, km, vm, km, vm, 2 * num_ctas, merges, num_merges, st)
                               : launch<64, kBf16Tiny>(p, km, vm, km, vm, 2 * num_ctas, merges, num_merges, st);
    return head_dim == 128 ? launch<128, kBf16>(p, km, vm, km, vm, num_ctas, merges, num_merges, st)
                           : launch<64, kBf16>(p, km, vm, km, vm, num_ctas, merges, num_merges, st);
}

}  // namespace

extern "C" xy_status xy_paged_attention(const void *q, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                        const int32_t *block_table, int max_blocks, const void *k_pages,
                                        const void *v_pages, int num_pages, int num_seqs, int num_tokens,
                                        int num_heads_q, int num_heads_kv, int head_dim, int block_size, float scale,
                                        int causal, const xy_task *tasks, int num_tasks, const xy_merge *merges,
                                        int num_merges, int num_ctas, void *workspace, size_t workspace_bytes,
                                        int32_t *err_word, void *out, void *stream) {
    return attention(q, cu_seqlens_q, context_lens, block_table, max_blocks, k_pages, v_pages, num_pages, num_seqs,
                     num_tokens, num_heads_q, num_heads_kv, head_dim, block_size, scale, causal, tasks, num_tasks, merges,
                     num_merges, num_ctas, workspace, workspace_bytes, nullptr, nullptr, err_word, out, stream);
}

namespace {
// xy_paged_attention_fp8; the dynamic deal when task_counter is given
xy_status attention_fp8(const void *q, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                        const int32_t *block_table, int max_blocks, const void *k_pages, const void *v_pages,
                        const float *k_scales, const float *v_scales, int num_pages, int num_seqs, int num_tokens,
                        int num_heads_q, int num_heads_kv, int head_dim, int block_size, float scale, int causal,
                        const xy_task *tasks, int num_tasks, const xy_merge *merges, int num_merges, int num_ctas,
                        void *workspace, size_t workspace_bytes, int32_t *task_counter, int32_t *err_word, void *out,
                        void *stream) {
    if (num_tasks < 0 || num_merges < 0 || num_seqs < 0 || num_tokens < 0) return XY_ERR_INVALID_ARG;
    if (num_tasks == 0 && num_merges == 0) return XY_OK;
    if (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales)) return XY_ERR_INVALID_ARG;
    AttnParams p;
    const xy_status ps = make_params(q, cu_seqlens_q, context_lens, block_table, max_blocks, k_pages, v_pages,
                                     num_pages, num_seqs, num_tokens, num_heads_q, num_heads_kv, head_dim,
                                     block_size, scale, causal, tasks, num_tasks, merges, num_merges, num_ctas,
                                     workspace, workspace_bytes, err_word, out, &p);
    if (ps != XY_OK) return ps;
    if (head_dim != 128 || p.G > 16 * kMathWarps) return XY_ERR_UNSUPPORTED;
    p.ksc = k_scales;
    p.vsc = v_scales;
    if (task_counter && (reinterpret_cast<uintptr_t>(task_counter) & 7)) return XY_ERR_INVALID_ARG;
    p.dyn = reinterpret_cast<int *>(task_counter);

    const int64_t rows = (int64_t)num_pages * num_heads_kv * block_size;
    const int keys = Cfg<128, kFp8Narrow>::RG::kKeys;  // both 8-bit rings stage 128 keys
    static_assert(Cfg<128, kFp8Wide>::RG::kKeys == Cfg<128, kFp8Narrow>::RG::kKeys, "one box height");
    const int box_rows = block_size < keys ? block_size : keys;
    CUtensorMap km, vm;
    // V codes at a fixed distance after the K codes in one allocation (16-byte multiple, past the K
    // pool): one 3-D map over both, whose box brings a page's K and V codes in one copy
    const uintptr_t kva = reinterpret_cast<uintptr_t>(k_pages), vva = reinterpret_cast<uintptr_t>(v_pages);
    const uint64_t kv_gap = vva > kva ? (uint64_t)(vva - kva) : 0;
    const bool kv3d = kv_gap >= (uint64_t)rows * 128u && kv_gap % 16 == 0 && kv_gap < (1ull << 40);
    if (kv3d) {
        if (!make_pool_map_u8_kv(&km, k_pages, rows, box_rows, kv_gap)) return XY_ERR_CUDA;
        vm = km;
        p.kv3d = 1;
    } else if (!make_pool_map_u8(&km, k_pages, rows, box_rows) || !make_pool_map_u8(&vm, v_pages, rows, box_rows)) {
        return XY_ERR_CUDA;
    }
    CUtensorMap ksm, vsm;
    if (!make_scale_map(&ksm, k_scales, (int64_t)num_pages * num_heads_kv, block_size) ||
        !make_scale_map(&vsm, v_scales, (int64_t)num_pages * num_heads_kv, block_size))
        return XY_ERR_CUDA;
    // every task runs on the decode path (f16 MMAs on converted codes)
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool narrow = num_tokens == num_seqs && p.G <= XY_FP8_NARROW_ROWS;
    // pure decode with G <= 8 under the dynamic deal: two half-size CTAs per SM slot
    if (narrow && p.G <= 8 && p.dyn)
        return launch<128, kFp8Tiny>(p, km, vm, ksm, vsm, 2 * num_ctas, merges, num_merges, st);
    return narrow ? launch<128, kFp8Narrow>(p, km, vm, ksm, vsm, num_ctas, merges, num_merges, st)
                  : launch<128, kFp8Wide>(p, km, vm, ksm, vsm, num_ctas, merges, num_merges, st);
}
}  // namespace

extern "C" xy_status xy_paged_attention_fp8(const void *q, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                            const int32_t *block_table, int max_blocks, const void *k_pages,
                                            const void *v_pages, const float *k_scales, const float *v_scales,
                                            int num_pages, int num_seqs, int num_tokens, int num_heads_q,
                                            int num_heads_kv, int head_dim, int block_size, float scale, int causal,
                                            const xy_task *tasks, int num_tasks, const xy_merge *merges,
                                            int num_merges, int num_ctas, void *workspace, size_t workspace_bytes,
                                            int32_t *err_word, void *out, void *stream) {
    return attention_fp8(q, cu_seqlens_q, context_lens, block_table, max_blocks, k_pages, v_pages, k_scales, v_scales,
                         num_pages, num_seqs, num_tokens, num_heads_q, num_heads_kv, head_dim, block_size, scale,
                         causal, tasks, num_tasks, merges, num_merges, num_ctas, workspace, workspace_bytes, nullptr,
                         err_word, out, stream);
}

// Dynamic deal over 8-bit pages: as xy_paged_attention_fp8, each CTA claiming the next task of the
// table from task_counter (its first producer warp claims, no scheduler warp).
extern "C" xy_status xy_paged_attention_fp8_dynamic(const void *q, const int32_t *cu_seqlens_q,
                                                    const int32_t *context_lens, const int32_t *block_table,
                                                    int max_blocks, const void *k_pages, const void *v_pages,
                                                    const float *k_scales, const float *v_scales, int num_pages,
                                                    int num_seqs, int num_tokens, int num_heads_q, int num_heads_kv,
                                                    int head_dim, int block_size, float scale, int causal,
                                                    const xy_task *tasks, int num_tasks, const xy_merge *merges,
                                                    int num_merges, int num_ctas, void *workspace,
                                                    size_t workspace_bytes, int32_t *task_counter, int32_t *err_word,
                                                    void *out, void *stream) {
    if (!task_counter) return XY_ERR_INVALID_ARG;
    return attention_fp8(q, cu_seqlens_q, context_lens, block_table, max_blocks, k_pages, v_pages, k_scales, v_scales,
                         num_pages, num_seqs, num_tokens, num_heads_q, num_heads_kv, head_dim, block_size, scale,
                         causal, tasks, num_tasks, merges, num_merges, num_ctas, workspace, workspace_bytes,
                         task_counter, err_word, out, stream);
}

// Dynamic deal: the kernels xy_paged_attention would launch, each CTA claiming the next task of
// the table (in table order) from a counter as it starts its current one, instead of walking a
// fixed share.
extern "C" xy_status xy_paged_attention_dynamic(const void *q, const int32_t *cu_seqlens_q,
                                                const int32_t *context_lens, const int32_t *block_table,
                                                int max_blocks, const void *k_pages, const void *v_pages,
                                                int num_pages, int num_seqs, int num_tokens, int num_heads_q,
                                                int num_heads_kv, int head_dim, int block_size, float scale,
                                                int causal, const xy_task *tasks, int num_tasks,
                                                const xy_merge *merges, int num_merges, int num_ctas,
                                                void *workspace, size_t workspace_bytes, int32_t *task_counter,
                                                int32_t *err_word, void *out, void *stream) {
    if (!task_counter) return XY_ERR_INVALID_ARG;
    return attention(q, cu_seqlens_q, context_lens, block_table, max_blocks, k_pages, v_pages, num_pages, num_seqs,
                     num_tokens, num_heads_q, num_heads_kv, head_dim, block_size, scale, causal, tasks, num_tasks, merges,
                     num_merges, num_ctas, workspace, workspace_bytes, task_counter, nullptr, err_word, out, stream);
}

extern "C" xy_status xy_paged_attention_traced(const void *q, const int32_t *cu_seqlens_q,
                                               const int32_t *context_lens, const int32_t *block_table,
                                               int max_blocks, const void *k_pages, const void *v_pages,
                                               int num_pages, int num_seqs, int num_tokens, int num_heads_q,
                                               int num_heads_kv, int head_dim, int block_size, float scale,
                                               int causal, const xy_task *tasks, int num_tasks,
                                               const xy_merge *merges, int num_merges, int num_ctas,
                                               void *workspace, size_t workspace_bytes, int32_t *task_counter,
                                               uint64_t *cta_trace, int32_t *err_word, void *out, void *stream) {
    if (!cta_trace) return XY_ERR_INVALID_ARG;
    return attention(q, cu_seqlens_q, context_lens, block_table, max_blocks, k_pages, v_pages, num_pages, num_seqs,
                     num_tokens, num_heads_q, num_heads_kv, head_dim, block_size, scale, causal, tasks, num_tasks, merges,
                     num_merges, num_ctas, workspace, workspace_bytes, task_counter, cta_trace, err_word, out, stream);
}

// ---------------------------------------------------------------------------------------------
// No-allocation variant: the split-KV scratch is a fixed array in this library instead of a caller
// buffer.  Host code only ever sees a stand-in symbol for the array, never its device address, so
// the address is looked up once per device (with that device current) and cached.

static __device__ __align__(256) unsigned char g_noalloc_scratch[XY_NOALLOC_SCRATCH_BYTES];

namespace {

xy_status noalloc_scratch(void **ptr) {
    static std::mutex mu;
    static std::vector<void *> by_device;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return XY_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)by_device.size() <= dev) by_device.resize(dev + 1, nullptr);
    if (!by_device[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return XY_ERR_CUDA;
        by_device[dev] = p;
    }
    *ptr = by_device[dev];
    return XY_OK;
}

}  // namespace

extern "C" xy_status xy_paged_attention_noalloc(const void *q, const int32_t *cu_seqlens_q,
                                                const int32_t *context_lens, const int32_t *block_table,
                                                int max_blocks, const void *k_pages, const void *v_pages,
                                                int num_pages, int num_seqs, int num_tokens, int num_heads_q,
                                                int num_heads_kv, int head_dim, int block_size, float scale,
                                                int causal, const xy_task *tasks, int num_tasks,
                                                const xy_merge *merges, int num_merges, int num_ctas,
                                                size_t workspace_bytes, int32_t *err_word, void *out,
                                                void *stream) {
    if (workspace_bytes > (size_t)XY_NOALLOC_SCRATCH_BYTES) return XY_ERR_WORKSPACE;
    if (num_tasks == 0 && num_merges == 0) return XY_OK;
    void *scratch = nullptr;
    const xy_status st = noalloc_scratch(&scratch);
    if (st != XY_OK) return st;
    return xy_paged_attention(q, cu_seqlens_q, context_lens, block_table, max_blocks, k_pages, v_pages, num_pages,
                              num_seqs, num_tokens, num_heads_q, num_heads_kv, head_dim, block_size, scale, causal,
                              tasks, num_tasks, merges, num_merges, num_ctas, scratch, workspace_bytes, err_word,
                              out, stream);
}

// ---------------------------------------------------------------------------------------------
// A step over 8-bit pages with decode and multi-token sequences: the tile part on bf16 copies of
// its pages (tcgen05 tiles), the decode part on the codes, both from the tables of
// xy_build_fp8_step_tables.
extern "C" xy_status xy_paged_attention_fp8_mixed(const void *q, const void *tables, const xy_fp8_step_tables *t,
                                                  const void *k_pages, const void *v_pages, const float *k_scales,
                                                  const float *v_scales, int num_pages, int num_seqs, int num_tokens,
                                                  int max_blocks, int num_heads_q, int num_heads_kv, int head_dim,
                                                  int block_size, float scale, int causal, int num_ctas, void *copy_k,
                                                  void *copy_v, int copy_pages, void *tile_ws, size_t tile_ws_bytes,
                                                  void *dec_ws, size_t dec_ws_bytes, int32_t *task_counters,
                                                  int32_t *err_word, void *out, void *stream) {
    if (!q || !tables || !t || !out || !task_counters || !aligned16(tables) ||
        (reinterpret_cast<uintptr_t>(task_counters) & 7) || num_seqs < 0 || num_tokens < 0 || max_blocks < 1 ||
        num_heads_kv < 1 || num_heads_q < num_heads_kv || num_heads_q % num_heads_kv)
        return XY_ERR_INVALID_ARG;
    if (head_dim != 128) return XY_ERR_UNSUPPORTED;
    // the description must fit this batch
    if (t->tile_seq_begin < 0 || t->tile_seq_end < t->tile_seq_begin || t->tile_seq_end > num_seqs ||
        t->dec_seq_begin < 0 || t->dec_seq_end < t->dec_seq_begin || t->dec_seq_end > num_seqs ||
        t->tile_tok_begin < 0 || t->tile_tok_end < t->tile_tok_begin || t->tile_tok_end > num_tokens ||
        t->dec_tok_begin < 0 || t->dec_tok_end < t->dec_tok_begin || t->dec_tok_end > num_tokens ||
        t->tile_num_pages < 0 || t->tile_num_tasks < 0 || t->dec_num_tasks < 0 || t->tile_num_merges < 0 ||
        t->dec_num_merges < 0)
        return XY_ERR_INVALID_ARG;
    const uint8_t *base = static_cast<const uint8_t *>(tables);
    const size_t row_bytes = (size_t)num_heads_q * head_dim * 2;   // one packed token of q / out
    const auto *q8 = static_cast<const uint8_t *>(q);
    auto *o8 = static_cast<uint8_t *>(out);
    const int32_t *ctx = reinterpret_cast<const int32_t *>(base + t->ctx_off);
    const int32_t *bt = reinterpret_cast<const int32_t *>(base + t->bt_off);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int nt = t->tile_seq_end - t->tile_seq_begin, nd = t->dec_seq_end - t->dec_seq_begin;
    if (nt > 0) {
        if (!copy_k || !copy_v || copy_pages < t->tile_num_pages) return XY_ERR_WORKSPACE;
        if (t->tile_workspace_bytes > 0 && (!tile_ws || tile_ws_bytes < t->tile_workspace_bytes))
            return XY_ERR_WORKSPACE;
        xy_status s = xy_dequant_pages_fp8(k_pages, v_pages, k_scales, v_scales, num_pages, num_heads_kv, block_size,
                                           head_dim, reinterpret_cast<const int32_t *>(base + t->tile_pages_off),
                                           t->tile_num_pages, copy_k, copy_v, err_word, stream);
        if (s != XY_OK) return s;
        s = attention(q8 + (size_t)t->tile_tok_begin * row_bytes, reinterpret_cast<const int32_t *>(base + t->tile_cu_off),
                      ctx + t->tile_seq_begin, reinterpret_cast<const int32_t *>(base + t->tile_bt_off), max_blocks,
                      copy_k, copy_v, t->tile_num_pages > 0 ? t->tile_num_pages : 1, nt,
                      t->tile_tok_end - t->tile_tok_begin, num_heads_q, num_heads_kv, head_dim, block_size, scale,
                      causal, reinterpret_cast<const xy_task *>(base + t->tile_tasks_off), t->tile_num_tasks,
                      reinterpret_cast<const xy_merge *>(base + t->tile_merges_off), t->tile_num_merges, num_ctas,
                      tile_ws, tile_ws_bytes, task_counters, nullptr, err_word,
                      o8 + (size_t)t->tile_tok_begin * row_bytes, stream);
        if (s != XY_OK) return s;
    }
    if (nd > 0) {
        if (t->dec_workspace_bytes > 0 && (!dec_ws || dec_ws_bytes < t->dec_workspace_bytes)) return XY_ERR_WORKSPACE;
        const xy_status s = attention_fp8(
            q8 + (size_t)t->dec_tok_begin * row_bytes, reinterpret_cast<const int32_t *>(base + t->dec_cu_off),
            ctx + t->dec_seq_begin, bt + (size_t)t->dec_seq_begin * max_blocks, max_blocks, k_pages, v_pages, k_scales,
            v_scales, num_pages, nd, t->dec_tok_end - t->dec_tok_begin, num_heads_q, num_heads_kv, head_dim,
            block_size, scale, causal, reinterpret_cast<const xy_task *>(base + t->dec_tasks_off), t->dec_num_tasks,
            reinterpret_cast<const xy_merge *>(base + t->dec_merges_off), t->dec_num_merges, num_ctas, dec_ws,
            dec_ws_bytes, task_counters + 2, err_word, o8 + (size_t)t->dec_tok_begin * row_bytes, stream);
        if (s != XY_OK) return s;
    }
    (void)st;
    return XY_OK;
}
