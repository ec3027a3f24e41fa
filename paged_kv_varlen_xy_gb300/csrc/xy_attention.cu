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
#include <vector>

#include "xy.h"
#include "xy_device.cuh"
#include "xy_attn_common.cuh"

namespace {

using xy::AttnParams;
using xy::TaskInfo;
using xy::ex2;
using xy::fetch_info;

constexpr int kStageKeys = 64;
constexpr int kMathWarps = 4;
constexpr int kMaxRows = 16 * kMathWarps;

template <int HD>
struct Cfg {
    static constexpr int kHalves = HD / 64;                     // 128-byte swizzle atoms per row
    static constexpr int kHalfBytes = kStageKeys * 128;         // one half of K or V in a stage
    static constexpr int kTensorBytes = kHalves * kHalfBytes;   // K or V of one stage
    static constexpr int kQBytes = kMaxRows * HD * 2;           // the task's Q rows (first stage only)
    static constexpr int kStageBytes = 2 * kTensorBytes + kQBytes;
    static constexpr int kStages = HD == 128 ? 4 : 6;
    static constexpr int kThreads = (kMathWarps + 1) * 32;
    static constexpr int kSlotFloats = 16 * HD + 32;            // merge slot: O[16][HD], m[16], l[16]
    static constexpr int kStagesOff = 0;
    static constexpr int kSlotsOff = kStages * kStageBytes;
    static constexpr int kBarOff = kSlotsOff + kMathWarps * kSlotFloats * 4;
    static constexpr int kFlagOff = kBarOff + 2 * kStages * 8;  // abort flag + 2 x 4 vote words
    static constexpr int kSmemBytes = kFlagOff + 64 + 1024;     // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
};

// Tasks of the CUDA-core/mma.sync path: the ones the tcgen05 tile kernel does not own.
template <int HD>
__device__ __forceinline__ bool mine(const TaskInfo &f, const AttnParams &p) {
    return !xy::is_tile_task(f.t, p.G, HD);
}

__device__ __forceinline__ bool info_ok(const TaskInfo &f, const AttnParams &p) {
    const xy_task &t = f.t;
    if (!xy::task_common_ok(f, p)) return false;
    if (t.q_rows * p.G > kMaxRows || (t.kv_start % kStageKeys) != 0) return false;
    return true;
}

// Byte offset of element (key, col) of a stage tensor.  The stage holds 64 keys in boxes of BR =
// 2^sh keys (one box per page, or per 64 keys of a larger page); a box is [half][BR][128 B] with
// the TMA 128-byte swizzle, i.e. the 16-byte chunk index is XOR-ed with (key & 7), so eight
// consecutive keys of one half hit eight different bank groups.
template <int HD>
__device__ __forceinline__ uint32_t swz(int key, int col, int sh) {
    const int half = col >> 6, chunk = (col & 63) >> 3;
    const int r = key & ((1 << sh) - 1);
    return (uint32_t)((key - r) * Cfg<HD>::kHalves * 128 + ((half * 128) << sh) + r * 128 +
                      ((chunk ^ (key & 7)) << 4) + (col & 7) * 2);
}

template <int HD>
__global__ void __launch_bounds__(Cfg<HD>::kThreads, 1)
    paged_attention_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const AttnParams p) {
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = xy::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t stages = base + C::kStagesOff;
    float *slots = reinterpret_cast<float *>(gbase + C::kSlotsOff);
    const uint32_t full_bar = base + C::kBarOff;
    const uint32_t empty_bar = full_bar + C::kStages * 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::kFlagOff);
    volatile int *vote = abort_flag + 4;  // [2][kMathWarps], indexed by task parity

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            xy::mbar_init(full_bar + 8 * s, 1);
            xy::mbar_init(empty_bar + 8 * s, kMathWarps);
        }
        *abort_flag = 0;
        xy::fence_mbarrier_init();
    }
    __syncthreads();

    const int BR = p.bs < kStageKeys ? p.bs : kStageKeys;  // keys per TMA box
    const int br_sh = 31 - __clz(BR);

    if (warp == kMathWarps) {
        // ------------------------------ producer warp ------------------------------
        if (lane == 0) {
            xy::prefetch_tensormap(&kmap);
            xy::prefetch_tensormap(&vmap);
        }
        // Block-table entries are read 32 logical pages at a time (one per lane) and the next
        // window is loaded before it is needed, so no stage waits on a dependent global load.
        auto load_win = [&](const int32_t *row, int base) -> int {
            const int idx = base + lane;
            return (idx >= 0 && idx < p.MB) ? __ldg(row + idx) : -1;
        };
        int ctr = 0;
        bool ok = true;
        int ti = blockIdx.x;
        bool have = ti < p.num_tasks;
        TaskInfo cur;
        if (have) cur = fetch_info(p.tasks[ti], p);
        int pref_win = -1;
        bool pref_valid = false;
        while (have && ok) {
            const int tn = ti + gridDim.x;
            const bool have_next = tn < p.num_tasks;
            xy_task rec_next;
            if (have_next) rec_next = p.tasks[tn];
            TaskInfo nxt;
            bool nxt_fetched = false;
            if (!mine<HD>(cur, p)) {
                // a tcgen05 tile task: the tile kernel runs it
            } else if (!info_ok(cur, p)) {
                if (lane == 0) xy::set_err(p.err, XY_DEV_BAD_TASK);
            } else {
                const xy_task &t = cur.t;
                const int32_t *bt_row = p.bt + (int64_t)t.seq * p.MB;
                int win0 = t.kv_start / p.bs;
                int pg_win = pref_valid ? pref_win : load_win(bt_row, win0);
                int pg_nxt = load_win(bt_row, win0 + 32);
                bool first_stage = true;
                for (int kv0 = t.kv_start; kv0 < t.kv_end; kv0 += kStageKeys, ++ctr) {
                    const int s = ctr % C::kStages;
                    if (ctr >= C::kStages &&
                        !xy::mbar_wait(empty_bar + 8 * s, ((ctr / C::kStages) - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int nkeys = min(kStageKeys, t.kv_end - kv0);
                    const int nbox = (nkeys + BR - 1) / BR;
                    if ((kv0 + nkeys - 1) / p.bs - win0 >= 32) {  // stage reaches into the next window
                        win0 += 32;
                        pg_win = pg_nxt;
                        pg_nxt = load_win(bt_row, win0 + 32);
                    }
                    const int n_copies = nbox * 2;  // one box per (page, tensor), both column halves
                    const int b = lane % nbox;
                    int my_pg = __shfl_sync(0xffffffffu, pg_win, (kv0 + b * BR) / p.bs - win0);
                    if (lane < n_copies && (my_pg < 0 || my_pg >= p.P)) {
                        xy::set_err(p.err, XY_DEV_PAGE_OOB);
                        my_pg = 0;
                    }
                    const uint32_t row_bytes = (uint32_t)p.G * HD * 2;  // one token's G query rows
                    const uint32_t q_bytes = first_stage ? (uint32_t)t.q_rows * row_bytes : 0u;
                    const uint32_t stage = stages + s * C::kStageBytes;
                    if (lane == 0)
                        xy::mbar_arrive_expect_tx(full_bar + 8 * s,
                                                  (uint32_t)(n_copies * C::kHalves * BR * 128) + q_bytes);
                    __syncwarp();
                    if (lane < n_copies) {
                        const int tensor = lane / nbox;
                        const int key = kv0 + b * BR;
                        const int y = (my_pg * p.Hkv + t.kv_head) * p.bs + (key % p.bs);
                        const uint32_t dst = stage + tensor * C::kTensorBytes + b * C::kHalves * BR * 128;
                        xy::tma_load_3d(dst, tensor ? &vmap : &kmap, 0, y, 0, full_bar + 8 * s);
                    }
                    if (first_stage) {
                        // the task's query rows: token j's G heads are one contiguous run of q
                        for (int j = lane; j < t.q_rows; j += 32) {
                            const int64_t tok = (int64_t)cur.seq_start + t.q_start + j;
                            const __nv_bfloat16 *src = p.q + (tok * p.Hq + (int64_t)t.kv_head * p.G) * HD;
                            xy::bulk_load(stage + 2 * C::kTensorBytes + j * row_bytes, src, row_bytes,
                                          full_bar + 8 * s);
                        }
                        first_stage = false;
                        if (have_next) {  // the next record has arrived by now: prefetch its numbers
                            nxt = fetch_info(rec_next, p);
                            nxt_fetched = true;
                            pref_valid = rec_next.seq >= 0 && rec_next.seq < p.S && rec_next.kv_start >= 0;
                            if (pref_valid)
                                pref_win = load_win(p.bt + (int64_t)rec_next.seq * p.MB, rec_next.kv_start / p.bs);
                        }
                    }
                    __syncwarp();
                }
            }
            if (!nxt_fetched) {
                pref_valid = false;
                if (have_next) nxt = fetch_info(rec_next, p);
            }
            cur = nxt;
            ti = tn;
            have = have_next;
        }
        if (!ok) {
            if (lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
            *abort_flag = 1;
        }
        // Drain: every issued stage must have landed before the CTA may exit.
        for (int k = ctr - 1; k >= 0 && k >= ctr - C::kStages; --k)
            xy::mbar_wait(full_bar + 8 * (k % C::kStages), (k / C::kStages) & 1);
        return;
    }

    // ------------------------------ math warps ------------------------------
    const int g4 = lane >> 2, c4 = lane & 3;
    int ctr = 0, iter = 0;
    int ti = blockIdx.x;
    bool have = ti < p.num_tasks;
    TaskInfo cur;
    if (have) cur = fetch_info(p.tasks[ti], p);
    while (have) {
        const int tn = ti + gridDim.x;
        const bool have_next = tn < p.num_tasks;
        xy_task rec_next;
        if (have_next) rec_next = p.tasks[tn];
        TaskInfo nxt;
        bool nxt_fetched = false;
        if (!mine<HD>(cur, p) || !info_ok(cur, p)) {
            if (have_next) nxt = fetch_info(rec_next, p);
            cur = nxt;
            ti = tn;
            have = have_next;
            continue;
        }
        const xy_task t = cur.t;
        const int R = t.q_rows * p.G;
        int nrg = (R + 15) >> 4;
        if (nrg == 3) nrg = 4;
        const int wpg = kMathWarps / nrg;      // warps sharing one 16-row slice
        const int rg = warp % nrg, ks = warp / nrg;
        const int row_a = rg * 16 + g4, row_b = row_a + 8;
        const int seq_start = cur.seq_start;
        const int qn = cur.qn;
        const int L = cur.L;

        auto row_limit = [&](int r) -> int {
            if (r >= R) return t.kv_end;    // padding rows: never stored, kept finite
            const int lim = p.causal ? (L - qn + t.q_start + r / p.G + 1) : L;
            return min(lim, t.kv_end);
        };
        const int lim_a = row_limit(row_a), lim_b = row_limit(row_b);
        int lim_max = max(lim_a, lim_b);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lim_max = max(lim_max, __shfl_xor_sync(0xffffffffu, lim_max, o));

        // Q fragments (A operand, row-major 16 x HD) come from the first stage of the task, where
        // the producer placed the task's rows in (token, head) order; rows past R are zero.
        uint32_t qa[HD / 16][4];

        float o_acc[HD / 8][4];
#pragma unroll
        for (int n = 0; n < HD / 8; ++n) o_acc[n][0] = o_acc[n][1] = o_acc[n][2] = o_acc[n][3] = 0.f;
        float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

        const int sub = kStageKeys / wpg;
        bool ok = true;
        for (int kv0 = t.kv_start; kv0 < t.kv_end; kv0 += kStageKeys, ++ctr) {
            const int s = ctr % C::kStages;
            if (!xy::mbar_wait(full_bar + 8 * s, (ctr / C::kStages) & 1, abort_flag)) {
                ok = false;
                break;
            }
            const uint32_t kst = stages + s * C::kStageBytes;
            const uint32_t vst = kst + C::kTensorBytes;
            if (kv0 == t.kv_start) {
                const uint8_t *qs = gbase + C::kStagesOff + s * C::kStageBytes + 2 * C::kTensorBytes;
                const uint32_t *qa_ptr = row_a < R ? reinterpret_cast<const uint32_t *>(qs + row_a * HD * 2) : nullptr;
                const uint32_t *qb_ptr = row_b < R ? reinterpret_cast<const uint32_t *>(qs + row_b * HD * 2) : nullptr;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const int w0 = kk * 8 + c4, w1 = w0 + 4;  // 32-bit words: cols 16kk+2c and +8
                    qa[kk][0] = qa_ptr ? qa_ptr[w0] : 0u;
                    qa[kk][1] = qb_ptr ? qb_ptr[w0] : 0u;
                    qa[kk][2] = qa_ptr ? qa_ptr[w1] : 0u;
                    qa[kk][3] = qb_ptr ? qb_ptr[w1] : 0u;
                }
                if (have_next) {  // prefetch the next task's numbers while this one runs
                    nxt = fetch_info(rec_next, p);
                    nxt_fetched = true;
                }
            }

            const int k_lo = kv0 + ks * sub;
            const int k_hi = min(min(k_lo + sub, t.kv_end), lim_max);
            for (int kc = k_lo; kc < k_hi; kc += 16) {
                const int kr = kc - kv0;
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                {
                    const int mi = lane >> 3;
                    const int krow = kr + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        uint32_t b0, b1, b2, b3;
                        xy::ldsm_x4(kst + swz<HD>(krow, kk * 16 + ((mi & 1) << 3), br_sh), b0, b1, b2, b3);
                        xy::mma_bf16_16816(sc[0], qa[kk], b0, b1);
                        xy::mma_bf16_16816(sc[1], qa[kk], b2, b3);
                    }
                }
                // virtual + causal mask, then online softmax in the log2 domain
                float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = kc + 8 * j + 2 * c4 + e;
                        sc[j][e] = key < lim_a ? sc[j][e] * p.scale_log2 : -INFINITY;
                        sc[j][2 + e] = key < lim_b ? sc[j][2 + e] * p.scale_log2 : -INFINITY;
                        mx_a = fmaxf(mx_a, sc[j][e]);
                        mx_b = fmaxf(mx_b, sc[j][2 + e]);
                    }
                }
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
                const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
                const float mu_a = mn_a == -INFINITY ? 0.f : mn_a;
                const float mu_b = mn_b == -INFINITY ? 0.f : mn_b;
                const float al_a = ex2(m_a - mu_a), al_b = ex2(m_b - mu_b);
                m_a = mn_a;
                m_b = mn_b;
                float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    sc[j][0] = ex2(sc[j][0] - mu_a);
                    sc[j][1] = ex2(sc[j][1] - mu_a);
                    sc[j][2] = ex2(sc[j][2] - mu_b);
                    sc[j][3] = ex2(sc[j][3] - mu_b);
                    ps_a += sc[j][0] + sc[j][1];
                    ps_b += sc[j][2] + sc[j][3];
                }
                l_a = l_a * al_a + ps_a;
                l_b = l_b * al_b + ps_b;
#pragma unroll
                for (int n = 0; n < HD / 8; ++n) {
                    o_acc[n][0] *= al_a;
                    o_acc[n][1] *= al_a;
                    o_acc[n][2] *= al_b;
                    o_acc[n][3] *= al_b;
                }
                uint32_t pa[4];
                pa[0] = xy::pack_bf16x2(sc[0][0], sc[0][1]);
                pa[1] = xy::pack_bf16x2(sc[0][2], sc[0][3]);
                pa[2] = xy::pack_bf16x2(sc[1][0], sc[1][1]);
                pa[3] = xy::pack_bf16x2(sc[1][2], sc[1][3]);
                // keys at or past kv_end may hold anything (unused slots, stale stage data):
                // their weights are 0, and their V entries are zeroed so 0 * NaN cannot occur.
                const bool tail = kc + 16 > t.kv_end;
                const int key_lo = kc + 2 * c4;
                const uint32_t keep0 = (key_lo < t.kv_end ? 0x0000ffffu : 0u) | (key_lo + 1 < t.kv_end ? 0xffff0000u : 0u);
                const uint32_t keep1 = (key_lo + 8 < t.kv_end ? 0x0000ffffu : 0u) | (key_lo + 9 < t.kv_end ? 0xffff0000u : 0u);
                {
                    const int mi = lane >> 3;
                    const int vrow = kr + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                    for (int jd = 0; jd < HD / 16; ++jd) {
                        uint32_t b0, b1, b2, b3;
                        xy::ldsm_x4_t(vst + swz<HD>(vrow, 8 * (2 * jd + (mi >> 1)), br_sh), b0, b1, b2, b3);
                        if (tail) {
                            b0 &= keep0;
                            b1 &= keep1;
                            b2 &= keep0;
                            b3 &= keep1;
                        }
                        xy::mma_bf16_16816(o_acc[2 * jd], pa, b0, b1);
                        xy::mma_bf16_16816(o_acc[2 * jd + 1], pa, b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) xy::mbar_arrive(empty_bar + 8 * s);
        }

        l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

        if (wpg > 1) {
            float *my = slots + warp * C::kSlotFloats;
#pragma unroll
            for (int n = 0; n < HD / 8; ++n) {
                const int col = 8 * n + 2 * c4;
                *reinterpret_cast<float2 *>(my + g4 * HD + col) = make_float2(o_acc[n][0], o_acc[n][1]);
                *reinterpret_cast<float2 *>(my + (g4 + 8) * HD + col) = make_float2(o_acc[n][2], o_acc[n][3]);
            }
            if (c4 == 0) {
                my[16 * HD + g4] = m_a;
                my[16 * HD + g4 + 8] = m_b;
                my[16 * HD + 16 + g4] = l_a;
                my[16 * HD + 16 + g4 + 8] = l_b;
            }
        }
        // Every math warp reaches this barrier (all waits above are bounded), so the vote makes
        // the decision to stop uniform and no warp is left waiting at a named barrier.
        if (lane == 0) vote[(iter & 1) * kMathWarps + warp] = (!ok || *abort_flag) ? 1 : 0;
        xy::named_bar_sync(1, kMathWarps * 32);
        {
            int bad = 0;
            for (int w = 0; w < kMathWarps; ++w) bad |= vote[(iter & 1) * kMathWarps + w];
            ++iter;
            if (bad) {
                *abort_flag = 1;
                if (warp == 0 && lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
                return;
            }
        }
        if (wpg > 1) {
            if (ks == 0) {
                float M_a = m_a, M_b = m_b;
                for (int k = 1; k < wpg; ++k) {
                    const float *ot = slots + (rg + k * nrg) * C::kSlotFloats;
                    M_a = fmaxf(M_a, ot[16 * HD + g4]);
                    M_b = fmaxf(M_b, ot[16 * HD + g4 + 8]);
                }
                const float U_a = M_a == -INFINITY ? 0.f : M_a, U_b = M_b == -INFINITY ? 0.f : M_b;
                float f_a = ex2(m_a - U_a), f_b = ex2(m_b - U_b);
                l_a *= f_a;
                l_b *= f_b;
#pragma unroll
                for (int n = 0; n < HD / 8; ++n) {
                    o_acc[n][0] *= f_a;
                    o_acc[n][1] *= f_a;
                    o_acc[n][2] *= f_b;
                    o_acc[n][3] *= f_b;
                }
                for (int k = 1; k < wpg; ++k) {
                    const float *ot = slots + (rg + k * nrg) * C::kSlotFloats;
                    const float ga = ex2(ot[16 * HD + g4] - U_a), gb = ex2(ot[16 * HD + g4 + 8] - U_b);
                    l_a += ga * ot[16 * HD + 16 + g4];
                    l_b += gb * ot[16 * HD + 16 + g4 + 8];
#pragma unroll
                    for (int n = 0; n < HD / 8; ++n) {
                        const int col = 8 * n + 2 * c4;
                        const float2 xa = *reinterpret_cast<const float2 *>(ot + g4 * HD + col);
                        const float2 xb = *reinterpret_cast<const float2 *>(ot + (g4 + 8) * HD + col);
                        o_acc[n][0] += ga * xa.x;
                        o_acc[n][1] += ga * xa.y;
                        o_acc[n][2] += gb * xb.x;
                        o_acc[n][3] += gb * xb.y;
                    }
                }
                m_a = M_a;
                m_b = M_b;
            }
            xy::named_bar_sync(1, kMathWarps * 32);
        }
        if (!nxt_fetched && have_next) nxt = fetch_info(rec_next, p);
        cur = nxt;
        ti = tn;
        have = have_next;
        if (ks != 0) continue;

        // store: the final bf16 rows, or this chunk's normalised partial + log2-sum-exp
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = half ? row_b : row_a;
            if (r >= R) continue;
            const float l = half ? l_b : l_a, m = half ? m_b : m_a;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            if (t.num_splits == 1) {
                const int64_t tok = seq_start + t.q_start + r / p.G;
                const int h = t.kv_head * p.G + r % p.G;
                __nv_bfloat16 *dst = p.out + (tok * p.Hq + h) * HD;
#pragma unroll
                for (int n = 0; n < HD / 8; ++n) {
                    const float x0 = o_acc[n][2 * half] * inv, x1 = o_acc[n][2 * half + 1] * inv;
                    *reinterpret_cast<uint32_t *>(dst + 8 * n + 2 * c4) = xy::pack_bf16x2(x0, x1);
                }
            } else {
                const int64_t wr = (int64_t)t.ws_row + r;
                float *dst = p.ws_o + wr * HD;
#pragma unroll
                for (int n = 0; n < HD / 8; ++n)
                    *reinterpret_cast<float2 *>(dst + 8 * n + 2 * c4) =
                        make_float2(o_acc[n][2 * half] * inv, o_acc[n][2 * half + 1] * inv);
                if (c4 == 0) p.ws_lse[wr] = l > 0.f ? m + __log2f(l) : -INFINITY;
            }
        }
    }
}

// Split-KV merge: for each split tile, out = sum_c 2^(lse_c - M) O_c / sum_c 2^(lse_c - M).
// One CTA per merge record, one warp per (token, head) row, lanes across head_dim.
template <int HD>
__global__ void __launch_bounds__(128) combine_kernel(const xy_merge *__restrict__ merges, const float *__restrict__ ws_o,
                                                      const float *__restrict__ ws_lse, const int32_t *__restrict__ cu,
                                                      int Hq, int G, int64_t ws_rows, int32_t *err,
                                                      __nv_bfloat16 *__restrict__ out) {
    const xy_merge m = merges[blockIdx.x];
    const int R = m.q_rows * G;
    if (m.num_splits < 2 || m.ws_row < 0 || (int64_t)m.ws_row + (int64_t)m.num_splits * R > ws_rows) {
        if (threadIdx.x == 0) xy::set_err(err, XY_DEV_BAD_TASK);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int V = HD / 32;  // floats per lane
    const int seq_start = __ldg(cu + m.seq);
    for (int r = warp; r < R; r += blockDim.x >> 5) {
        float M = -INFINITY;
        for (int c = 0; c < m.num_splits; ++c) M = fmaxf(M, __ldg(ws_lse + m.ws_row + (int64_t)c * R + r));
        const float U = M == -INFINITY ? 0.f : M;
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
        float W = 0.f;
        for (int c = 0; c < m.num_splits; ++c) {
            const int64_t row = m.ws_row + (int64_t)c * R + r;
            const float w = ex2(__ldg(ws_lse + row) - U);
            W += w;
            const float *src = ws_o + row * HD + lane * V;
            if (V == 4) {
                const float4 x = __ldg(reinterpret_cast<const float4 *>(src));
                acc[0] += w * x.x;
                acc[1] += w * x.y;
                acc[2] += w * x.z;
                acc[3] += w * x.w;
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) acc[v] += w * __ldg(src + v);
            }
        }
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

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int HD>
xy_status launch(const AttnParams &p, const CUtensorMap &km, const CUtensorMap &vm, int num_ctas,
                 const xy_merge *merges, int num_merges, cudaStream_t st) {
    using C = Cfg<HD>;
    static int configured_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return XY_ERR_CUDA;
    if (configured_device != dev) {  // the attribute is per device
        if (cudaFuncSetAttribute(paged_attention_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess)
            return XY_ERR_CUDA;
        configured_device = dev;
    }
    if (p.num_tasks > 0) {
        paged_attention_kernel<HD><<<num_ctas, C::kThreads, C::kSmemBytes, st>>>(km, vm, p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return xy::cuda_fail(e, "paged_attention_kernel launch");
    }
    if (num_merges > 0) {
        combine_kernel<HD><<<num_merges, 128, 0, st>>>(merges, p.ws_o, p.ws_lse, p.cu, p.Hq, p.G, p.ws_rows, p.err,
                                                       p.out);
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

extern "C" xy_status xy_paged_attention(const void *q, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                        const int32_t *block_table, int max_blocks, const void *k_pages,
                                        const void *v_pages, int num_pages, int num_seqs, int num_tokens,
                                        int num_heads_q, int num_heads_kv, int head_dim, int block_size, float scale,
                                        int causal, const xy_task *tasks, int num_tasks, const xy_merge *merges,
                                        int num_merges, int num_ctas, void *workspace, size_t workspace_bytes,
                                        int32_t *err_word, void *out, void *stream) {
    if (num_tasks < 0 || num_merges < 0 || num_seqs < 0 || num_tokens < 0) return XY_ERR_INVALID_ARG;
    if (num_tasks == 0 && num_merges == 0) return XY_OK;
    if (!q || !cu_seqlens_q || !context_lens || !block_table || !k_pages || !v_pages || !tasks || !out ||
        !err_word || num_ctas < 1 || max_blocks < 1 || num_pages < 1 || num_seqs < 1 || num_heads_kv < 1 ||
        num_heads_q < num_heads_kv || num_heads_q % num_heads_kv)
        return XY_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out)) return XY_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return XY_ERR_UNSUPPORTED;
    if (block_size < 16 || block_size > 256 || (block_size & (block_size - 1))) return XY_ERR_UNSUPPORTED;
    if (num_merges > 0 && (!merges || !workspace || !aligned16(workspace))) return XY_ERR_WORKSPACE;

    const int64_t rows = (int64_t)num_pages * num_heads_kv * block_size;
    if (rows > INT32_MAX) return XY_ERR_UNSUPPORTED;
    const int box_rows = block_size < kStageKeys ? block_size : kStageKeys;
    CUtensorMap km, vm;
    if (!make_pool_map(&km, k_pages, rows, head_dim, box_rows) ||
        !make_pool_map(&vm, v_pages, rows, head_dim, box_rows))
        return XY_ERR_CUDA;

    AttnParams p;
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
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Prefill/chunk tiles (more than 16 rows) run on the tcgen05 kernel first; a batch with one
    // query token per sequence and G <= 16 has none.
    if (num_tasks > 0 && head_dim == 128 && (128 % p.G) == 0 && (num_tokens > num_seqs || p.G > 16)) {
        const xy_status ts = xy::launch_tile_attention(p, k_pages, v_pages, num_pages, block_size, num_ctas, st);
        if (ts != XY_OK) return ts;
    }
    return head_dim == 128 ? launch<128>(p, km, vm, num_ctas, merges, num_merges, st)
                           : launch<64>(p, km, vm, num_ctas, merges, num_merges, st);
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
