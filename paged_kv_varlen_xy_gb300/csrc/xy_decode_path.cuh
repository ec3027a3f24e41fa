// The decode path of the paged attention: tasks with few (token, head) rows, which are
// HBM-bound.  Used by the stand-alone kernel in xy_attention.cu and by the unified kernel in
// xy_tile.cu, which host it with their own warp layout and shared-memory map.
//
// "XY-Serve 深度实战" (chenxutan.com/d/5031) §2.2 component 3 (one GEMM-softmax-GEMM per task of
// the task table) and §2.3 technique 1 (virtual padding: masked on chip, valid rows stored).
//
// A producer warp gathers each 64-key stage of K and V with 3-D TMA boxes -- one box per page
// (both 64-column halves), rows addressed as (physical_page * Hkv + kv_head) * bs + offset --
// into a ring of shared-memory stages with 128-byte swizzle; the task's query rows travel with
// its first stage as bulk copies.  Four math warps own 16-row slices of the task's rows; QK^T and
// PV run on m16n8k16 tensor-core fragments, the online softmax on the accumulator registers with
// quad shuffles.  When a task has fewer rows than warps x 16 the warps split each stage's keys
// and merge their (max, sum, O) triples through shared memory at the end of the task.
//
// 8-bit pages (E4M3 codes with one fp32 scale per stored (token, KV head) row, head_dim 128):
// the stage holds the codes (a 128-byte row per key) and the stage keys' K and V scales.  The
// math warps turn codes into f16 in registers (exact) right after the fragment loads and run f16
// MMAs; the query rows are converted bf16 -> f16 once per task.  K scales multiply the fp32
// scores; V scales multiply the softmax weights before they are rounded to f16, relative to the
// largest V scale seen so far (so the packed weights stay in [0, 1]), and that largest scale
// multiplies O once at the end of the task.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "xy.h"
#include "xy_attn_common.cuh"
#include "xy_device.cuh"

namespace xy {
namespace dec {

constexpr int kStageKeys = 64;
constexpr int kMathWarps = 4;

// Geometry of a decode stage ring: NS stages of K, V (64 keys x HD) and room for QR query rows.
template <int HD, int NS, int QR>
struct Ring {
    static constexpr bool kFp8 = false;
    static constexpr int kKeys = kStageKeys;                       // keys per stage
    static constexpr int kHalves = HD / 64;                        // 128-byte swizzle atoms per row
    static constexpr int kTensorBytes = kHalves * kStageKeys * 128;  // K or V of one stage
    static constexpr int kQOff = 2 * kTensorBytes;                 // query rows
    static constexpr int kScaleOff = 0;                            // (no scales)
    static constexpr int kQBytes = QR * HD * 2;                    // the task's rows (first stage only)
    static constexpr int kStageBytes = 2 * kTensorBytes + kQBytes;
    static constexpr int kStages = NS;
    static constexpr int kMaxRows = QR;
    static constexpr int kBytes = NS * kStageBytes;
    static constexpr int kSlotFloats = 16 * HD + 32;               // merge slot: O[16][HD], m[16], l[16]
    static constexpr int kSlotBytes = (kMathWarps - 1) * kSlotFloats * 4;  // warps ks >= 1
    static_assert(QR % 16 == 0 && QR <= 16 * kMathWarps, "rows per decode task");
};

// Geometry of an 8-bit decode stage ring (head_dim 128): NS stages, each holding the K and V codes
// of KEYS keys (one 128-byte row per key, 128-byte swizzle), their K scales then V scales (fp32),
// and room for QR bf16 query rows.  A stage of 128 keys carries about as many bytes as a 64-key
// bf16 stage, and gives each of four key-splitting math warps 32 keys.
template <int NS, int QR, int KEYS = 128, bool ONLY_T = false>
struct RingF8 {
    static constexpr bool kFp8 = true;
    // every task runs the transposed products (tasks of at most 8 rows; consume_task_f8t)
    static constexpr bool kOnlyT = ONLY_T;
    static constexpr int kKeys = KEYS;
    static constexpr int kHalves = 1;
    static constexpr int kTensorBytes = KEYS * 128;
    static constexpr int kScaleOff = 2 * kTensorBytes;
    static constexpr int kQOff = kScaleOff + 2 * KEYS * 4;
    static constexpr int kQBytes = QR * 128 * 2;
    static constexpr int kStageBytes = (kQOff + kQBytes + 1023) / 1024 * 1024;  // stages stay 1024-aligned
    static constexpr int kStages = NS;
    static constexpr int kMaxRows = ONLY_T ? 8 : QR;
    static constexpr int kBytes = NS * kStageBytes;
    static constexpr int kSlotFloats = 16 * 128 + 32;
    static constexpr int kSlotBytes = (kMathWarps - 1) * kSlotFloats * 4;
    static_assert(QR % 16 == 0 && QR <= 16 * kMathWarps, "rows per decode task");
    static_assert(KEYS % (32 * kMathWarps) == 0, "32 keys per math warp and step");
};

// Byte offset, from the stage start, of 16-byte chunk `chunk` of key `key`'s K (kv = 0) or V
// (kv = 1) codes in an 8-bit stage.  The stage holds its keys in boxes of BR = 2^br_sh keys (one
// per page, or per 128 keys of a longer page), each box as [K rows][V rows] of [BR][128 B] with the
// 128-byte swizzle: so one copy can bring a page's K and V codes when the two pools share one
// allocation (a 3-D tensor map), and two copies land in the same places when they do not.
__device__ __forceinline__ uint32_t swz8kv(int kv, int key, int chunk, int br_sh) {
    return (uint32_t)(((((key >> br_sh) << 1) | kv) << (br_sh + 7)) + ((key & ((1 << br_sh) - 1)) << 7) +
                      ((chunk ^ (key & 7)) << 4));
}

// Shared-memory handles of the decode path, set up by the hosting kernel.
struct Smem {
    uint32_t stages;             // shared address of the stage ring (1024-aligned)
    uint8_t *stages_gen;         // generic pointer to the same ring
    float *slots;                // merge slots
    uint32_t full_bar;           // kStages mbarriers, count 1 (+ transaction bytes)
    uint32_t empty_bar;          // kStages mbarriers, count kMathWarps
    volatile int *abort_flag;    // CTA-wide
    volatile int *vote;          // [2][kMathWarps]
    uint32_t bar_id;             // named barrier shared by the four math warps
};

// Byte offset of element (key, col) of a stage tensor.  The stage holds 64 keys in boxes of BR =
// 2^sh keys (one box per page, or per 64 keys of a larger page); a box is [half][BR][128 B] with
// the TMA 128-byte swizzle, i.e. the 16-byte chunk index is XOR-ed with (key & 7), so eight
// consecutive keys of one half hit eight different bank groups.
template <int HD>
__device__ __forceinline__ uint32_t swz(int key, int col, int sh) {
    const int half = col >> 6, chunk = (col & 63) >> 3;
    const int r = key & ((1 << sh) - 1);
    return (uint32_t)((key - r) * (HD / 64) * 128 + ((half * 128) << sh) + r * 128 + ((chunk ^ (key & 7)) << 4) +
                      (col & 7) * 2);
}

// Checks of a decode-path task beyond task_common_ok.
template <class RG>
__device__ __forceinline__ bool task_ok(const TaskInfo &f, const AttnParams &p) {
    return task_common_ok(f, p) && f.t.q_rows * p.G <= RG::kMaxRows && (f.t.kv_start % RG::kKeys) == 0;
}

// Producer warp `pw` of `npw`: issue the stages of decode task `f` that land in ring slots
// s = pw, pw + npw, ... (a slot always has the same producer, which issues its uses in order, so
// each producer waits only on its own slots' empty barriers).  `ctr` counts all of the stages.
// `pg_first` is the task's first block-table window if it was prefetched (else -1 with
// have_first false).  `first_stage_done()` runs once, right after this warp's first stage of the
// task is issued (the caller prefetches the next task there), and `stage_done(keys_left)` after
// each of this warp's stages with the task's keys beyond that stage.  Returns false if a wait
// gave up.
// `dep_ready`: whether this warp has waited for the kernel ahead on the stream (the step's KV
// append, whose dependent launch lets this kernel start while it runs).  The warp waits before its
// first stage that holds one of a task's new tokens (keys >= L - qn, the rows the append writes);
// stages of older keys -- and the query rows, tables and block-table windows, which the append
// does not write -- go out before it.
// 8-bit pages: ksmap / vsmap view the K and V scale arrays as [pages * Hkv rows, bs floats] with a
// one-row box; with pages of at most 32 tokens a stage's scales come four pages per copy (TMA
// gather4) instead of one bulk copy per page and tensor (null for bf16 pages).
struct NoStageHook {
    __device__ void operator()(int) const {}
};
template <int HD, class RG, class F, class H = NoStageHook>
__device__ bool produce_task(const AttnParams &p, const TaskInfo &f, const CUtensorMap *kmap, const CUtensorMap *vmap,
                             const CUtensorMap *ksmap, const CUtensorMap *vsmap, const Smem &sm, int &ctr, int lane,
                             int pg_first, bool have_first, bool &dep_ready, F first_stage_done, int pw = 0,
                             int npw = 1, H stage_done = H()) {
    const xy_task &t = f.t;
    const int bs_sh = 31 - __clz(p.bs);                   // page size is a power of two
    const int BR = p.bs < RG::kKeys ? p.bs : RG::kKeys;  // keys per TMA box
    const int br_sh = 31 - __clz(BR);
    const uint32_t row_bytes = (uint32_t)p.G * HD * 2;     // one token's G query rows
    // block-table entries are read 32 logical pages at a time (one per lane), the next window
    // loaded before it is needed, so no stage waits on a dependent global load
    int win0 = t.kv_start >> bs_sh;
    int pg_win = have_first ? pg_first : load_window(p, t.seq, win0, lane);
    int pg_nxt = load_window(p, t.seq, win0 + 32, lane);
    bool first_mine = true;
    for (int kv0 = t.kv_start; kv0 < t.kv_end; kv0 += RG::kKeys, ++ctr) {
        if ((ctr % RG::kStages) % npw != pw) continue;  // another producer's slot
        const int s = ctr % RG::kStages;
        if (ctr >= RG::kStages &&
            !__all_sync(0xffffffffu, mbar_wait(sm.empty_bar + 8 * s, ((ctr / RG::kStages) - 1) & 1, sm.abort_flag)))
            return false;
        const int nkeys = min(RG::kKeys, t.kv_end - kv0);
        const int nbox = (nkeys + BR - 1) >> br_sh;
        while (((kv0 + nkeys - 1) >> bs_sh) - win0 >= 32) {  // the stage reaches into the next window
            win0 += 32;
            pg_win = pg_nxt;
            pg_nxt = load_window(p, t.seq, win0 + 32, lane);
        }
        // one box per (page, tensor), both column halves; 8-bit pages add each box's K and V scales
        // (one bulk copy per page and tensor, or for pages of at most 32 tokens one gather of four
        // pages' scale rows per tensor)
        const bool gather = RG::kFp8 && BR <= 32;
        const int ngather = (nbox + 3) >> 2;
        // 8-bit pools in one allocation (p.kv3d): one 3-D box brings a page's K and V codes
        const int n_code = RG::kFp8 && p.kv3d ? nbox : 2 * nbox;
        const int n_copies = RG::kFp8 ? n_code + (gather ? 0 : 2 * nbox) : 2 * nbox;
        const int b = lane % nbox;
        int my_pg = __shfl_sync(0xffffffffu, pg_win, ((kv0 + (b << br_sh)) >> bs_sh) - win0);
        if (lane < n_copies && (my_pg < 0 || my_pg >= p.P)) {
            set_err(p.err, XY_DEV_PAGE_OOB);
            my_pg = 0;
        }
        if (!dep_ready && kv0 + nkeys > f.L - f.qn) {
            grid_dep_wait();
            dep_ready = true;
        }
        // the task's first stage also carries its query rows
        const bool q_here = kv0 == t.kv_start;
        const uint32_t q_bytes = q_here ? (uint32_t)t.q_rows * row_bytes : 0u;
        const uint32_t stage = sm.stages + s * RG::kStageBytes;
        const uint32_t kv_bytes =
            RG::kFp8 ? (uint32_t)(nbox * BR * 2 * 128 + (gather ? ngather * 4 : nbox) * BR * 2 * 4)
                     : (uint32_t)(n_copies * RG::kHalves * BR * 128);
        if (lane == 0) mbar_arrive_expect_tx(sm.full_bar + 8 * s, kv_bytes + q_bytes);
        __syncwarp();
        if (lane < n_copies) {
            const int tensor = lane / nbox;
            const int key = kv0 + (b << br_sh);
            const int y = ((my_pg * p.Hkv + t.kv_head) << bs_sh) + (key & (p.bs - 1));
            if constexpr (RG::kFp8) {
                // lane groups of nbox: the codes (one 3-D box per page, or a K box and a V box),
                // then the scales (K, V) when they are not gathered; box b's codes land as
                // [K rows][V rows] (swz8kv)
                const int code_groups = p.kv3d ? 1 : 2;
                if (tensor < code_groups) {
                    if (p.kv3d)
                        tma_load_3d(stage + (b << (br_sh + 8)), kmap, 0, y, 0, sm.full_bar + 8 * s);
                    else
                        tma_load_2d(stage + (((b << 1) | tensor) << (br_sh + 7)), tensor ? vmap : kmap, 0, y,
                                    sm.full_bar + 8 * s);
                } else {
                    const int st = tensor - code_groups;                    // 0: K scales, 1: V scales
                    const float *src = (st ? p.vsc : p.ksc) + y;           // the box's BR scales
                    bulk_load(stage + RG::kScaleOff + st * RG::kKeys * 4 + b * BR * 4, src, (uint32_t)BR * 4,
                              sm.full_bar + 8 * s);
                }
            } else {
                const uint32_t dst = stage + tensor * RG::kTensorBytes + b * RG::kHalves * BR * 128;
                tma_load_3d(dst, tensor ? vmap : kmap, 0, y, 0, sm.full_bar + 8 * s);
            }
        }
        if constexpr (RG::kFp8) {
            if (gather) {
                // scale rows (page * Hkv + head) of boxes 4g .. 4g + 3; a group past the stage's last
                // page repeats that page's row (the extra rows land in unused scale slots of the stage)
                const int srow = my_pg * p.Hkv + t.kv_head;   // box `lane % nbox`'s row
                for (int g = 0; g < ngather; ++g) {
                    int r[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) r[i] = __shfl_sync(0xffffffffu, srow, min(4 * g + i, nbox - 1));
                    if (lane < 2) {
                        const uint32_t dst = stage + RG::kScaleOff + lane * RG::kKeys * 4 + g * 4 * BR * 4;
                        tma_gather4(dst, lane ? vsmap : ksmap, 0, r[0], r[1], r[2], r[3], sm.full_bar + 8 * s);
                    }
                }
            }
        }
        if (q_here) {
            // token j's G heads are one contiguous run of q
            for (int j = lane; j < t.q_rows; j += 32) {
                const int64_t tok = (int64_t)f.seq_start + t.q_start + j;
                const __nv_bfloat16 *src = p.q + (tok * p.Hq + (int64_t)t.kv_head * p.G) * HD;
                bulk_load(stage + RG::kQOff + j * row_bytes, src, row_bytes, sm.full_bar + 8 * s);
            }
        }
        if (first_mine) {
            first_mine = false;
            first_stage_done();
        }
        stage_done(t.kv_end - (kv0 + nkeys));
        __syncwarp();
    }
    return true;
}

// Producer `pw` of `npw`, before exiting: every stage it issued (`ctr` stages issued in all) has
// landed.
template <class RG>
__device__ __forceinline__ void drain(const Smem &sm, int ctr, int pw = 0, int npw = 1) {
    for (int k = ctr - 1; k >= 0 && k >= ctr - RG::kStages; --k)
        if ((k % RG::kStages) % npw == pw) mbar_wait(sm.full_bar + 8 * (k % RG::kStages), (k / RG::kStages) & 1);
}

// 8-bit pages, tasks of at most 8 (token, head) rows: the products transposed, S^T = K Q^T and
// O^T = V^T P^T, so that keys and head-dim columns fill the 16-row side of the m16n8k16 fragments
// and the (at most 8) query rows its 8-column side.  Per 32 keys a warp then issues 16 + 16 MMAs
// instead of 32 + 32 and holds 8 scores instead of 16 (a decode row no longer pads 15 of 16 MMA
// rows).  The packed weights reach the second product's B fragments through an in-register 8x8
// transpose.  Accumulator tile (cc, e): its row g holds column 32cc + 2g + e and its row g + 8
// column 32cc + 16 + 2g + e; its columns are the query rows.  Otherwise as consume_task: each math
// warp takes 32 keys of every stage, and the four merge their (max, sum, O) at the end.
// ONE: the task has a single (token, head) row (G = 1 decode).  Each lane then holds no second
// real row, and the softmax work of the second accumulator column (masking, maxima, exp2, sums,
// rescales) is left out; that column's weights are 0, so its accumulators stay 0.
template <class RG, bool ONE, class F>
__device__ bool consume_task_f8t(const AttnParams &p, const TaskInfo &f, const Smem &sm, int &ctr, int &iter, int w,
                                 int lane, F first_stage_seen) {
    constexpr int HD = 128;
    static_assert(RG::kKeys == 32 * kMathWarps, "32 keys per math warp and stage");
    const int g4 = lane >> 2, c4 = lane & 3;
    const int br_sh = 31 - __clz(p.bs < RG::kKeys ? p.bs : RG::kKeys);   // keys per stage box
    const xy_task t = f.t;
    const int R = t.q_rows * p.G;  // at most 8
    const int qn = f.qn, L = f.L;
    auto row_limit = [&](int r) -> int {
        if (r >= R) return t.kv_end;  // padding rows: never stored, kept finite
        const int lim = p.causal ? (L - qn + t.q_start + r / p.G + 1) : L;
        return min(lim, t.kv_end);
    };
    const int r0 = 2 * c4, r1 = r0 + 1;  // this lane's query rows (accumulator columns)
    const int lim0 = row_limit(r0), lim1 = ONE ? 0 : row_limit(r1);
    int lim_max = max(lim0, lim1);
    lim_max = max(lim_max, __shfl_xor_sync(0xffffffffu, lim_max, 1));
    lim_max = max(lim_max, __shfl_xor_sync(0xffffffffu, lim_max, 2));

    uint32_t qb[HD / 16][2];  // Q^T B fragments, f16, in the k-order of the K code fragments
    float o[HD / 32][2][4];
#pragma unroll
    for (int cc = 0; cc < HD / 32; ++cc)
#pragma unroll
        for (int e = 0; e < 2; ++e) o[cc][e][0] = o[cc][e][1] = o[cc][e][2] = o[cc][e][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // l: this lane's keys only
    float s_max = 0.f, s_inv = 0.f;  // largest V scale seen, and its reciprocal

    auto keys32 = [&](uint32_t kst, uint32_t vst, const float *scl, int kc, int kr) {
        const int mi = lane >> 3;
        // S^T of 16-key blocks b = 0, 1: C fragment rows are keys kc + 16b + g (0, 1) and + 8
        // (2, 3), columns the query rows r0, r1; even and odd 16-column k-steps accumulate apart
        float sp[2][2][4];
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int h = 0; h < 2; ++h) sp[b][h][0] = sp[b][h][1] = sp[b][h][2] = sp[b][h][3] = 0.f;
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                // matrix i: keys 8(i&1).. of chunk 2cc + (i>>1); lane (g, c) gets cols 4c..4c+3 of
                // its key, i.e. the A fragment (rows = keys) of one k-step in Q's k-order
                const int krow = kr + 16 * b + ((mi & 1) << 3) + (lane & 7);
                uint32_t r[4], lo[4], hi[4];
                ldsm_x4(kst + swz8kv(0, krow, 2 * cc + (mi >> 1), br_sh), r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(r[i], lo[i], hi[i]);
                const uint32_t a0[4] = {lo[0], lo[1], hi[0], hi[1]};
                const uint32_t a1[4] = {lo[2], lo[3], hi[2], hi[3]};
                mma_f16_16816(sp[b][0], a0, qb[2 * cc][0], qb[2 * cc][1]);
                mma_f16_16816(sp[b][1], a1, qb[2 * cc + 1][0], qb[2 * cc + 1][1]);
            }
        }
        float sc[2][4];
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int j = 0; j < 4; ++j) sc[b][j] = sp[b][0][j] + sp[b][1][j];
        // scales of keys kc + 16b + 8h + g (V scales of keys at or past kv_end, which may hold
        // anything, read as 0); virtual + causal mask; online softmax (log2 domain)
        float vs[2][2];
        float mx0 = -INFINITY, mx1 = -INFINITY, vmax = 0.f;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int o_ = kr + 16 * b + 8 * h + g4;
                const int key = kc + 16 * b + 8 * h + g4;
                const float kx = scl[o_], vx = scl[RG::kKeys + o_];
                vs[b][h] = key < t.kv_end ? vx : 0.f;
                vmax = fmaxf(vmax, vs[b][h]);
                const float fk = p.scale_log2 * kx;
                sc[b][2 * h] = key < lim0 ? sc[b][2 * h] * fk : -INFINITY;
                mx0 = fmaxf(mx0, sc[b][2 * h]);
                if constexpr (!ONE) {
                    sc[b][2 * h + 1] = key < lim1 ? sc[b][2 * h + 1] * fk : -INFINITY;
                    mx1 = fmaxf(mx1, sc[b][2 * h + 1]);
                }
            }
        }
        // lazy reference max, as in consume_task; a row's keys lie across the lanes of one column c
        float al0 = 1.f, al1 = 1.f;
        if (__any_sync(0xffffffffu, mx0 > m0 + 8.f || (!ONE && mx1 > m1 + 8.f))) {
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
                if constexpr (!ONE) mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
            }
            const float mn0 = mx0 > m0 + 8.f ? mx0 : m0;
            al0 = ex2(m0 - (mn0 == -INFINITY ? 0.f : mn0));
            m0 = mn0;
            if constexpr (!ONE) {
                const float mn1 = mx1 > m1 + 8.f ? mx1 : m1;
                al1 = ex2(m1 - (mn1 == -INFINITY ? 0.f : mn1));
                m1 = mn1;
            }
        }
        const float mu0 = m0 == -INFINITY ? 0.f : m0, mu1 = m1 == -INFINITY ? 0.f : m1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                sc[b][2 * h] = ex2(sc[b][2 * h] - mu0);
                ps0 += sc[b][2 * h];
                if constexpr (ONE) {
                    sc[b][2 * h + 1] = 0.f;
                } else {
                    sc[b][2 * h + 1] = ex2(sc[b][2 * h + 1] - mu1);
                    ps1 += sc[b][2 * h + 1];
                }
            }
        }
        l0 = l0 * al0 + ps0;
        if constexpr (!ONE) l1 = l1 * al1 + ps1;
        bool rescale = al0 != 1.f || al1 != 1.f;
        if (__any_sync(0xffffffffu, vmax > s_max)) {
            // every column c holds the same keys, so the maximum over g is warp-uniform
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, x));
            const float gs = s_max / vmax;
            al0 *= gs;
            if constexpr (!ONE) al1 *= gs;
            s_max = vmax;
            s_inv = 1.f / vmax;
            rescale = true;
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int cc = 0; cc < HD / 32; ++cc)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    o[cc][e][0] *= al0;
                    o[cc][e][1] *= al1;
                    o[cc][e][2] *= al0;
                    o[cc][e][3] *= al1;
                }
        }
        // P^T B fragments: (key g | g + 8, rows r0, r1) packed, then transposed to (row g, keys
        // 2c, 2c+1 | 8 + 2c, 9 + 2c)
        uint32_t pb[2][2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const float w0 = vs[b][0] * s_inv, w1 = vs[b][1] * s_inv;
            pb[b][0] = movm_t(pack_f16x2(sc[b][0] * w0, sc[b][1] * w0));
            pb[b][1] = movm_t(pack_f16x2(sc[b][2] * w1, sc[b][3] * w1));
        }
        // V^T A fragments from ldmatrix.trans over the code rows (as in consume_task: lane (g, c)
        // gets cols 2g, 2g+1 of keys 2c, 2c+1 of matrix i = keys 8(i&1).. of chunk 2cc + (i>>1));
        // even columns feed tile (cc, 0), odd ones tile (cc, 1).  Keys at or past kv_end get zero
        // V entries, so 0 * NaN cannot occur.
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int key_lo = kc + 16 * b + 2 * c4;
            const bool tail = kc + 16 * b + 16 > t.kv_end;
            const uint32_t keep0 =
                (key_lo < t.kv_end ? 0x0000ffffu : 0u) | (key_lo + 1 < t.kv_end ? 0xffff0000u : 0u);
            const uint32_t keep1 =
                (key_lo + 8 < t.kv_end ? 0x0000ffffu : 0u) | (key_lo + 9 < t.kv_end ? 0xffff0000u : 0u);
            const int vrow = kr + 16 * b + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
            for (int cc = 0; cc < HD / 32; ++cc) {
                uint32_t r[4], ev[4], od[4];
                ldsm_x4_t(kst + swz8kv(1, vrow, 2 * cc + (mi >> 1), br_sh), r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // bytes (k0 c0, k0 c1, k1 c0, k1 c1) regrouped as (k0 c0, k1 c0, k0 c1, k1 c1)
                    e4m3x4_to_f16x2x2(__byte_perm(r[i], 0u, 0x3120), ev[i], od[i]);
                    if (tail) {
                        const uint32_t keep = (i & 1) ? keep1 : keep0;
                        ev[i] &= keep;
                        od[i] &= keep;
                    }
                }
                const uint32_t ae[4] = {ev[0], ev[2], ev[1], ev[3]};
                const uint32_t ao[4] = {od[0], od[2], od[1], od[3]};
                mma_f16_16816(o[cc][0], ae, pb[b][0], pb[b][1]);
                mma_f16_16816(o[cc][1], ao, pb[b][0], pb[b][1]);
            }
        }
    };

    const int sub = RG::kKeys / kMathWarps;  // 32
    bool ok = true;
    for (int kv0 = t.kv_start; kv0 < t.kv_end; kv0 += RG::kKeys, ++ctr) {
        const int s = ctr % RG::kStages;
        if (!mbar_wait(sm.full_bar + 8 * s, (ctr / RG::kStages) & 1, sm.abort_flag)) {
            ok = false;
            break;
        }
        const uint32_t kst = sm.stages + s * RG::kStageBytes;
        const uint32_t vst = kst + RG::kTensorBytes;
        if (kv0 == t.kv_start) {
            // f16 query rows in the k-order of the K fragments: k 2c, 2c+1 hold cols 16kk+4c, +1
            // and k 2c+8, 2c+9 cols 16kk+4c+2, +3; rows past R are zero
            const uint8_t *qs = sm.stages_gen + s * RG::kStageBytes + RG::kQOff;
            const uint32_t *qp = g4 < R ? reinterpret_cast<const uint32_t *>(qs + g4 * HD * 2) : nullptr;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const int w0 = kk * 8 + 2 * c4;
                qb[kk][0] = qp ? bf16x2_to_f16x2(qp[w0]) : 0u;
                qb[kk][1] = qp ? bf16x2_to_f16x2(qp[w0 + 1]) : 0u;
            }
            first_stage_seen();
        }
        const int k_lo = kv0 + w * sub;
        const int k_hi = min(min(k_lo + sub, t.kv_end), lim_max);
        const float *scl = reinterpret_cast<const float *>(sm.stages_gen + s * RG::kStageBytes + RG::kScaleOff);
        if (k_lo < k_hi) keys32(kst, vst, scl, k_lo, k_lo - kv0);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty_bar + 8 * s);
    }

    // back from units of s_max; row sums over the lanes of a column
#pragma unroll
    for (int cc = 0; cc < HD / 32; ++cc)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int j = 0; j < 4; ++j) o[cc][e][j] *= s_max;
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, x);
        l1 += __shfl_xor_sync(0xffffffffu, l1, x);
    }
    // lane (g, c) holds columns 32cc + 16h + 2g, +1 of rows r0 (j = 0) and r1 (j = 1)
    auto col_of = [&](int cc, int h) -> int { return 32 * cc + 16 * h + 2 * g4; };
    if (w > 0) {  // warps 1..3 hand their triples to warp 0
        float *my = sm.slots + (w - 1) * RG::kSlotFloats;
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                *reinterpret_cast<float2 *>(my + r0 * HD + col_of(cc, h)) = make_float2(o[cc][0][2 * h], o[cc][1][2 * h]);
                *reinterpret_cast<float2 *>(my + r1 * HD + col_of(cc, h)) =
                    make_float2(o[cc][0][2 * h + 1], o[cc][1][2 * h + 1]);
            }
        if (g4 == 0) {
            my[16 * HD + r0] = m0;
            my[16 * HD + r1] = m1;
            my[16 * HD + 16 + r0] = l0;
            my[16 * HD + 16 + r1] = l1;
        }
    }
    // Every math warp reaches this barrier (all waits above are bounded), so the vote makes the
    // decision to stop uniform and no warp is left waiting at a named barrier.
    if (lane == 0) sm.vote[(iter & 1) * kMathWarps + w] = (!ok || *sm.abort_flag) ? 1 : 0;
    named_bar_sync(sm.bar_id, kMathWarps * 32);
    {
        int bad = 0;
        for (int v = 0; v < kMathWarps; ++v) bad |= sm.vote[(iter & 1) * kMathWarps + v];
        ++iter;
        if (bad) return false;
    }
    if (w == 0) {
        float M0 = m0, M1 = m1;
        for (int k = 1; k < kMathWarps; ++k) {
            const float *ot = sm.slots + (k - 1) * RG::kSlotFloats;
            M0 = fmaxf(M0, ot[16 * HD + r0]);
            M1 = fmaxf(M1, ot[16 * HD + r1]);
        }
        const float U0 = M0 == -INFINITY ? 0.f : M0, U1 = M1 == -INFINITY ? 0.f : M1;
        const float f0 = ex2(m0 - U0), f1 = ex2(m1 - U1);
        l0 *= f0;
        l1 *= f1;
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                o[cc][e][0] *= f0;
                o[cc][e][1] *= f1;
                o[cc][e][2] *= f0;
                o[cc][e][3] *= f1;
            }
        for (int k = 1; k < kMathWarps; ++k) {
            const float *ot = sm.slots + (k - 1) * RG::kSlotFloats;
            const float ga = ex2(ot[16 * HD + r0] - U0), gb = ex2(ot[16 * HD + r1] - U1);
            l0 += ga * ot[16 * HD + 16 + r0];
            l1 += gb * ot[16 * HD + 16 + r1];
#pragma unroll
            for (int cc = 0; cc < HD / 32; ++cc)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 xa = *reinterpret_cast<const float2 *>(ot + r0 * HD + col_of(cc, h));
                    const float2 xb = *reinterpret_cast<const float2 *>(ot + r1 * HD + col_of(cc, h));
                    o[cc][0][2 * h] += ga * xa.x;
                    o[cc][1][2 * h] += ga * xa.y;
                    o[cc][0][2 * h + 1] += gb * xb.x;
                    o[cc][1][2 * h + 1] += gb * xb.y;
                }
        }
        m0 = M0;
        m1 = M1;
    }
    named_bar_sync(sm.bar_id, kMathWarps * 32);
    if (w != 0) return true;

    // store: the final bf16 rows, or this chunk's normalised partial + log2-sum-exp
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int r = r0 + j;
        if (r >= R) continue;
        const float l = j ? l1 : l0, m = j ? m1 : m0;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        if (t.num_splits == 1) {
            const int64_t tok = f.seq_start + t.q_start + r / p.G;
            const int hq = t.kv_head * p.G + r % p.G;
            __nv_bfloat16 *dst = p.out + (tok * p.Hq + hq) * HD;
#pragma unroll
            for (int cc = 0; cc < HD / 32; ++cc)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    *reinterpret_cast<uint32_t *>(dst + col_of(cc, h)) =
                        pack_bf16x2(o[cc][0][2 * h + j] * inv, o[cc][1][2 * h + j] * inv);
        } else {
            const int64_t wr = (int64_t)t.ws_row + r;
            float *dst = p.ws_o + wr * HD;
#pragma unroll
            for (int cc = 0; cc < HD / 32; ++cc)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    *reinterpret_cast<float2 *>(dst + col_of(cc, h)) =
                        make_float2(o[cc][0][2 * h + j] * inv, o[cc][1][2 * h + j] * inv);
            if (g4 == 0) p.ws_lse[wr] = l > 0.f ? m + __log2f(l) : -INFINITY;
        }
    }
    return true;
}

// Math warp w (0..3) runs decode task `f`.  `ctr` counts stages consumed on the ring, `iter` the
// tasks run (vote parity).  `first_stage_seen()` runs once, after the first stage has landed.
// Returns false when the math warps voted to stop (a wait gave up); every math warp returns the
// same value, and all of them pass the same named barriers.
template <int HD, class RG, class F>
__device__ bool consume_task(const AttnParams &p, const TaskInfo &f, const Smem &sm, int &ctr, int &iter, int w,
                             int lane, F first_stage_seen) {
    if constexpr (RG::kFp8) {
        if (f.t.q_rows * p.G == 1)
            return consume_task_f8t<RG, true>(p, f, sm, ctr, iter, w, lane, first_stage_seen);
        if (RG::kOnlyT || f.t.q_rows * p.G <= 8)
            return consume_task_f8t<RG, false>(p, f, sm, ctr, iter, w, lane, first_stage_seen);
    }
    const int g4 = lane >> 2, c4 = lane & 3;
    const int BR = p.bs < RG::kKeys ? p.bs : RG::kKeys;
    const int br_sh = 31 - __clz(BR);
    const xy_task t = f.t;
    const int R = t.q_rows * p.G;
    int nrg = (R + 15) >> 4;
    if (nrg == 3) nrg = 4;
    const int wpg = kMathWarps / nrg;  // warps sharing one 16-row slice
    const int rg = w % nrg, ks = w / nrg;
    const int row_a = rg * 16 + g4, row_b = row_a + 8;
    const int qn = f.qn, L = f.L;

    auto row_limit = [&](int r) -> int {
        if (r >= R) return t.kv_end;  // padding rows: never stored, kept finite
        const int lim = p.causal ? (L - qn + t.q_start + r / p.G + 1) : L;
        return min(lim, t.kv_end);
    };
    const int lim_a = row_limit(row_a), lim_b = row_limit(row_b);
    static_assert(!RG::kFp8 || HD == 128, "8-bit pages: head_dim 128");
    // output columns of accumulator pair n: 8n + 2c, +1; over 8-bit pages 16(n/2) + 4c + 2(n%2), +1
    // (see the V fragments of fp8_keys32)
    auto ocol = [&](int n) -> int { return RG::kFp8 ? 16 * (n >> 1) + 4 * c4 + 2 * (n & 1) : 8 * n + 2 * c4; };
    float s_max = 0.f, s_inv = 0.f;  // 8-bit pages: largest V scale seen, and its reciprocal
    int lim_max = max(lim_a, lim_b);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lim_max = max(lim_max, __shfl_xor_sync(0xffffffffu, lim_max, o));

    // Q fragments (A operand, row-major 16 x HD) come from the first stage of the task, where the
    // producer placed the task's rows in (token, head) order; rows past R are zero.
    uint32_t qa[HD / 16][4];
    float o_acc[HD / 8][4];
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) o_acc[n][0] = o_acc[n][1] = o_acc[n][2] = o_acc[n][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    // 8-bit pages: 32 keys of one stage, as two 16-key blocks b = 0, 1 whose QK^T chains are
    // independent and which share one max / rescale step.  K scales multiply the fp32 scores;
    // V scales the weights, relative to s_max (the largest V scale so far, so the packed f16
    // weights stay in [0, 1]); O is kept in units of s_max and rescaled when s_max grows.
    auto fp8_keys32 = [&](uint32_t kst, uint32_t vst, const float *scl, int kc, int kr) {
        const int mi = lane >> 3;
        float sc[2][2][4];  // [block][n-tile: keys 8j..8j+7 of the block][C fragment]
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int j = 0; j < 2; ++j) sc[b][j][0] = sc[b][j][1] = sc[b][j][2] = sc[b][j][3] = 0.f;
        // ldmatrix over the code rows: matrix i holds keys 8(i&1).. of 16-byte chunk 2cc+(i>>1);
        // lane (g, c) gets the codes of cols 4c..4c+3 of key g, i.e. the B fragment of one k-step
        // in the k-order of the query fragments
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int krow = kr + 16 * b + ((mi & 1) << 3) + (lane & 7);
                uint32_t r[4];
                ldsm_x4(kst + swz8kv(0, krow, 2 * cc + (mi >> 1), br_sh), r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t b0, b1;
                    e4m3x4_to_f16x2x2(r[i], b0, b1);
                    mma_f16_16816(sc[b][i & 1], qa[2 * cc + (i >> 1)], b0, b1);
                }
            }
        }
        // scales of this lane's keys kc + 16b + 8j + 2c + e (V scales of keys at or past kv_end,
        // which may hold anything, read as 0); virtual + causal mask; online softmax (log2 domain)
        float vsc[2][2][2];
        float mx_a = -INFINITY, mx_b = -INFINITY, vmax = 0.f;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int o = kr + 16 * b + 8 * j + 2 * c4;
                const float2 kx = *reinterpret_cast<const float2 *>(scl + o);
                const float2 vx = *reinterpret_cast<const float2 *>(scl + RG::kKeys + o);
                const int key = kc + 16 * b + 8 * j + 2 * c4;
                vsc[b][j][0] = key < t.kv_end ? vx.x : 0.f;
                vsc[b][j][1] = key + 1 < t.kv_end ? vx.y : 0.f;
                vmax = fmaxf(vmax, fmaxf(vsc[b][j][0], vsc[b][j][1]));
                const float f0 = p.scale_log2 * kx.x, f1 = p.scale_log2 * kx.y;
                sc[b][j][0] = key < lim_a ? sc[b][j][0] * f0 : -INFINITY;
                sc[b][j][1] = key + 1 < lim_a ? sc[b][j][1] * f1 : -INFINITY;
                sc[b][j][2] = key < lim_b ? sc[b][j][2] * f0 : -INFINITY;
                sc[b][j][3] = key + 1 < lim_b ? sc[b][j][3] * f1 : -INFINITY;
                mx_a = fmaxf(mx_a, fmaxf(sc[b][j][0], sc[b][j][1]));
                mx_b = fmaxf(mx_b, fmaxf(sc[b][j][2], sc[b][j][3]));
            }
        }
        // The reference max m is raised only when a row's max exceeds it by more than 8 (weights
        // then stay <= 2^8, fine in f16 and fp32); the stale reference cancels in O / l.  Each
        // lane tests its own scores, so the row maxima (quad shuffles) are formed only when some
        // reference has to grow -- in a task's first step and rarely after it.
        float al_a = 1.f, al_b = 1.f;
        if (__any_sync(0xffffffffu, mx_a > m_a + 8.f || mx_b > m_b + 8.f)) {
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
            const bool grow_a = mx_a > m_a + 8.f, grow_b = mx_b > m_b + 8.f;  // the same in a row's quad
            const float mn_a = grow_a ? mx_a : m_a, mn_b = grow_b ? mx_b : m_b;
            al_a = ex2(m_a - (mn_a == -INFINITY ? 0.f : mn_a));
            al_b = ex2(m_b - (mn_b == -INFINITY ? 0.f : mn_b));
            m_a = mn_a;
            m_b = mn_b;
        }
        const float mu_a = m_a == -INFINITY ? 0.f : m_a;
        const float mu_b = m_b == -INFINITY ? 0.f : m_b;
        float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                sc[b][j][0] = ex2(sc[b][j][0] - mu_a);
                sc[b][j][1] = ex2(sc[b][j][1] - mu_a);
                sc[b][j][2] = ex2(sc[b][j][2] - mu_b);
                sc[b][j][3] = ex2(sc[b][j][3] - mu_b);
                ps_a += sc[b][j][0] + sc[b][j][1];
                ps_b += sc[b][j][2] + sc[b][j][3];
            }
        }
        l_a = l_a * al_a + ps_a;
        l_b = l_b * al_b + ps_b;
        bool rescale = al_a != 1.f || al_b != 1.f;
        if (__any_sync(0xffffffffu, vmax > s_max)) {
            // a larger V scale: the step's largest (every quad holds the same keys, so the quad
            // maximum is the same in every quad and the branch below is warp-uniform)
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
            const float g = s_max / vmax;
            al_a *= g;
            al_b *= g;
            s_max = vmax;
            s_inv = 1.f / vmax;
            rescale = true;
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int n = 0; n < HD / 8; ++n) {
                o_acc[n][0] *= al_a;
                o_acc[n][1] *= al_a;
                o_acc[n][2] *= al_b;
                o_acc[n][3] *= al_b;
            }
        }
        uint32_t pa[2][4];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float w0 = vsc[b][j][0] * s_inv, w1 = vsc[b][j][1] * s_inv;
                pa[b][2 * j] = pack_f16x2(sc[b][j][0] * w0, sc[b][j][1] * w1);
                pa[b][2 * j + 1] = pack_f16x2(sc[b][j][2] * w0, sc[b][j][3] * w1);
            }
        }
        // ldmatrix.trans over the code rows: matrix i holds keys 8(i&1).. of chunk 2cc+(i>>1);
        // lane (g, c) gets the code pairs (cols 2g, 2g+1) of keys 2c and 2c+1 (+8).  Regrouped by
        // column they are the B fragments of two n-tiles: even columns 2g and odd columns 2g+1 of
        // the chunk, so the C fragments of pair 2ch + {0, 1} hold columns 16ch + 4c + {0, 2} and
        // {1, 3}.  Keys at or past kv_end get zero V entries, so 0 * NaN cannot occur.
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int key_lo = kc + 16 * b + 2 * c4;
            const bool tail = kc + 16 * b + 16 > t.kv_end;
            const uint32_t keep0 =
                (key_lo < t.kv_end ? 0x0000ffffu : 0u) | (key_lo + 1 < t.kv_end ? 0xffff0000u : 0u);
            const uint32_t keep1 =
                (key_lo + 8 < t.kv_end ? 0x0000ffffu : 0u) | (key_lo + 9 < t.kv_end ? 0xffff0000u : 0u);
            const int vrow = kr + 16 * b + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
            for (int cc = 0; cc < HD / 32; ++cc) {
                uint32_t r[4];
                ldsm_x4_t(kst + swz8kv(1, vrow, 2 * cc + (mi >> 1), br_sh), r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // bytes (k0 c0, k0 c1, k1 c0, k1 c1) regrouped as (k0 c0, k1 c0, k0 c1, k1 c1)
                    uint32_t ea0, eb0, ea1, eb1;
                    e4m3x4_to_f16x2x2(__byte_perm(r[2 * h], 0u, 0x3120), ea0, eb0);
                    e4m3x4_to_f16x2x2(__byte_perm(r[2 * h + 1], 0u, 0x3120), ea1, eb1);
                    if (tail) {
                        ea0 &= keep0;
                        eb0 &= keep0;
                        ea1 &= keep1;
                        eb1 &= keep1;
                    }
                    const int ch = 2 * cc + h;
                    mma_f16_16816(o_acc[2 * ch], pa[b], ea0, ea1);
                    mma_f16_16816(o_acc[2 * ch + 1], pa[b], eb0, eb1);
                }
            }
        }
    };

    const int sub = RG::kKeys / wpg;
    bool ok = true;
    for (int kv0 = t.kv_start; kv0 < t.kv_end; kv0 += RG::kKeys, ++ctr) {
        const int s = ctr % RG::kStages;
        if (!mbar_wait(sm.full_bar + 8 * s, (ctr / RG::kStages) & 1, sm.abort_flag)) {
            ok = false;
            break;
        }
        const uint32_t kst = sm.stages + s * RG::kStageBytes;
        const uint32_t vst = kst + RG::kTensorBytes;
        if (kv0 == t.kv_start) {
            const uint8_t *qs = sm.stages_gen + s * RG::kStageBytes + RG::kQOff;
            const uint32_t *qa_ptr = row_a < R ? reinterpret_cast<const uint32_t *>(qs + row_a * HD * 2) : nullptr;
            const uint32_t *qb_ptr = row_b < R ? reinterpret_cast<const uint32_t *>(qs + row_b * HD * 2) : nullptr;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                if constexpr (RG::kFp8) {
                    // f16, in the k-order of the 8-bit K fragments: k 2c, 2c+1 hold cols 16kk+4c,
                    // +1 and k 2c+8, 2c+9 cols 16kk+4c+2, +3 (a dot product may sum in any order)
                    const int w0 = kk * 8 + 2 * c4, w1 = w0 + 1;
                    qa[kk][0] = qa_ptr ? bf16x2_to_f16x2(qa_ptr[w0]) : 0u;
                    qa[kk][1] = qb_ptr ? bf16x2_to_f16x2(qb_ptr[w0]) : 0u;
                    qa[kk][2] = qa_ptr ? bf16x2_to_f16x2(qa_ptr[w1]) : 0u;
                    qa[kk][3] = qb_ptr ? bf16x2_to_f16x2(qb_ptr[w1]) : 0u;
                } else {
                    const int w0 = kk * 8 + c4, w1 = w0 + 4;  // 32-bit words: cols 16kk+2c and +8
                    qa[kk][0] = qa_ptr ? qa_ptr[w0] : 0u;
                    qa[kk][1] = qb_ptr ? qb_ptr[w0] : 0u;
                    qa[kk][2] = qa_ptr ? qa_ptr[w1] : 0u;
                    qa[kk][3] = qb_ptr ? qb_ptr[w1] : 0u;
                }
            }
            first_stage_seen();
        }

        const int k_lo = kv0 + ks * sub;
        const int k_hi = min(min(k_lo + sub, t.kv_end), lim_max);
        if constexpr (RG::kFp8) {
            const float *scl = reinterpret_cast<const float *>(sm.stages_gen + s * RG::kStageBytes + RG::kScaleOff);
            for (int kc = k_lo; kc < k_hi; kc += 32) fp8_keys32(kst, vst, scl, kc, kc - kv0);
        } else {
            for (int kc = k_lo; kc < k_hi; kc += 16) {
                const int kr = kc - kv0;
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                {
                    const int mi = lane >> 3;
                    const int krow = kr + ((mi >> 1) << 3) + (lane & 7);
    #pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(kst + swz<HD>(krow, kk * 16 + ((mi & 1) << 3), br_sh), b0, b1, b2, b3);
                        mma_bf16_16816(sc[0], qa[kk], b0, b1);
                        mma_bf16_16816(sc[1], qa[kk], b2, b3);
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
                pa[0] = pack_bf16x2(sc[0][0], sc[0][1]);
                pa[1] = pack_bf16x2(sc[0][2], sc[0][3]);
                pa[2] = pack_bf16x2(sc[1][0], sc[1][1]);
                pa[3] = pack_bf16x2(sc[1][2], sc[1][3]);
                // keys at or past kv_end may hold anything (unused slots, stale stage data): their
                // weights are 0, and their V entries are zeroed so 0 * NaN cannot occur
                const bool tail = kc + 16 > t.kv_end;
                const int key_lo = kc + 2 * c4;
                const uint32_t keep0 =
                    (key_lo < t.kv_end ? 0x0000ffffu : 0u) | (key_lo + 1 < t.kv_end ? 0xffff0000u : 0u);
                const uint32_t keep1 =
                    (key_lo + 8 < t.kv_end ? 0x0000ffffu : 0u) | (key_lo + 9 < t.kv_end ? 0xffff0000u : 0u);
                {
                    const int mi = lane >> 3;
                    const int vrow = kr + ((mi & 1) << 3) + (lane & 7);
    #pragma unroll
                    for (int jd = 0; jd < HD / 16; ++jd) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(vst + swz<HD>(vrow, 8 * (2 * jd + (mi >> 1)), br_sh), b0, b1, b2, b3);
                        if (tail) {
                            b0 &= keep0;
                            b1 &= keep1;
                            b2 &= keep0;
                            b3 &= keep1;
                        }
                        mma_bf16_16816(o_acc[2 * jd], pa, b0, b1);
                        mma_bf16_16816(o_acc[2 * jd + 1], pa, b2, b3);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty_bar + 8 * s);
    }

    if constexpr (RG::kFp8) {
        // back from units of s_max; interleave the even- and odd-column tiles so that pair n holds
        // columns ocol(n), ocol(n) + 1 (register renaming only)
#pragma unroll
        for (int ch = 0; ch < HD / 16; ++ch) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float a0 = o_acc[2 * ch][2 * h] * s_max, a1 = o_acc[2 * ch][2 * h + 1] * s_max;
                const float b0 = o_acc[2 * ch + 1][2 * h] * s_max, b1 = o_acc[2 * ch + 1][2 * h + 1] * s_max;
                o_acc[2 * ch][2 * h] = a0;
                o_acc[2 * ch][2 * h + 1] = b0;
                o_acc[2 * ch + 1][2 * h] = a1;
                o_acc[2 * ch + 1][2 * h + 1] = b1;
            }
        }
    }
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

    if (wpg > 1 && ks > 0) {  // warps ks >= 1 hand their triples to warp ks = 0 of their slice
        float *my = sm.slots + (w - nrg) * RG::kSlotFloats;
#pragma unroll
        for (int n = 0; n < HD / 8; ++n) {
            const int col = ocol(n);
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
    // Every math warp reaches this barrier (all waits above are bounded), so the vote makes the
    // decision to stop uniform and no warp is left waiting at a named barrier.
    if (lane == 0) sm.vote[(iter & 1) * kMathWarps + w] = (!ok || *sm.abort_flag) ? 1 : 0;
    named_bar_sync(sm.bar_id, kMathWarps * 32);
    {
        int bad = 0;
        for (int v = 0; v < kMathWarps; ++v) bad |= sm.vote[(iter & 1) * kMathWarps + v];
        ++iter;
        if (bad) return false;
    }
    if (wpg > 1) {
        if (ks == 0) {
            float M_a = m_a, M_b = m_b;
            for (int k = 1; k < wpg; ++k) {
                const float *ot = sm.slots + (rg + (k - 1) * nrg) * RG::kSlotFloats;
                M_a = fmaxf(M_a, ot[16 * HD + g4]);
                M_b = fmaxf(M_b, ot[16 * HD + g4 + 8]);
            }
            const float U_a = M_a == -INFINITY ? 0.f : M_a, U_b = M_b == -INFINITY ? 0.f : M_b;
            const float f_a = ex2(m_a - U_a), f_b = ex2(m_b - U_b);
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
                const float *ot = sm.slots + (rg + (k - 1) * nrg) * RG::kSlotFloats;
                const float ga = ex2(ot[16 * HD + g4] - U_a), gb = ex2(ot[16 * HD + g4 + 8] - U_b);
                l_a += ga * ot[16 * HD + 16 + g4];
                l_b += gb * ot[16 * HD + 16 + g4 + 8];
#pragma unroll
                for (int n = 0; n < HD / 8; ++n) {
                    const int col = ocol(n);
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
        named_bar_sync(sm.bar_id, kMathWarps * 32);
    }
    if (ks != 0) return true;

    // store: the final bf16 rows, or this chunk's normalised partial + log2-sum-exp
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = half ? row_b : row_a;
        if (r >= R) continue;
        const float l = half ? l_b : l_a, m = half ? m_b : m_a;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        if (t.num_splits == 1) {
            const int64_t tok = f.seq_start + t.q_start + r / p.G;
            const int h = t.kv_head * p.G + r % p.G;
            __nv_bfloat16 *dst = p.out + (tok * p.Hq + h) * HD;
#pragma unroll
            for (int n = 0; n < HD / 8; ++n) {
                const float x0 = o_acc[n][2 * half] * inv, x1 = o_acc[n][2 * half + 1] * inv;
                *reinterpret_cast<uint32_t *>(dst + ocol(n)) = pack_bf16x2(x0, x1);
            }
        } else {
            const int64_t wr = (int64_t)t.ws_row + r;
            float *dst = p.ws_o + wr * HD;
#pragma unroll
            for (int n = 0; n < HD / 8; ++n)
                *reinterpret_cast<float2 *>(dst + ocol(n)) =
                    make_float2(o_acc[n][2 * half] * inv, o_acc[n][2 * half + 1] * inv);
            if (c4 == 0) p.ws_lse[wr] = l > 0.f ? m + __log2f(l) : -INFINITY;
        }
    }
    return true;
}

}  // namespace dec
}  // namespace xy
