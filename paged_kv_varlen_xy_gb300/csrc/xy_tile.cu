// Tensor-core (tcgen05 / TMEM) tiles of the paged attention: the prefill and chunk tasks, whose
// (token, head) rows fill a 128-row MMA tile.  The decode-sized tasks run in xy_attention.cu.
//
// "XY-Serve 深度实战" (chenxutan.com/d/5031) §2.2 component 3: Meta-Attention is one fused
// GEMM-softmax-GEMM over a task's (query block x KV block) tiles; §2.3 technique 1: ragged tiles
// are masked on chip and only valid rows are stored.
//
// One persistent CTA per SM, six warps:
//   warp 4      producer: TMA loads of the task's 128 query rows (G heads x 128/G tokens, one 3-D
//               box per 64-column half) and of 128-key K/V tiles gathered page by page through
//               the block table (2-D boxes, 128-byte swizzle) into a 3-stage ring;
//   warp 5      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM buffers, then
//               O += P_{j-1} V_{j-1} with P read from TMEM (it overwrites the first 64 columns of
//               its S buffer as packed bf16);
//   warps 0..3  softmax, one query row per thread (TMEM lane = row): masked row max, exp2,
//               row sum, P back to TMEM; O is rescaled in TMEM only when a row's running max grows
//               by more than 2^8 (the stale max is otherwise kept, which is exact because O and
//               the row sum share it); epilogue O / l straight from TMEM to global memory.
// TMEM: S0 = columns [0,128), S1 = [128,256), O = [256,384) of a 512-column allocation.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "xy.h"
#include "xy_attn_common.cuh"
#include "xy_device.cuh"

namespace {

using xy::AttnParams;
using xy::ex2;
using xy::fetch_info;
using xy::TaskInfo;

constexpr int HD = 128;
constexpr int kTileKeys = 128;
constexpr int kStages = 3;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr int kHalfBytes = 128 * 128;           // 128 rows x 64 bf16 columns
constexpr int kTileBytes = 2 * kHalfBytes;      // Q, K or V tile: [half][128 rows][128 B]
constexpr int kQOff = 0;
constexpr int kStageOff = kTileBytes;
constexpr int kStageBytes = 2 * kTileBytes;     // K then V
enum {
    B_QFULL = 0,
    B_QEMPTY,
    B_KVFULL0,
    B_KVEMPTY0 = B_KVFULL0 + kStages,
    B_SFULL0 = B_KVEMPTY0 + kStages,
    B_SFREE0 = B_SFULL0 + 2,
    B_PFULL0 = B_SFREE0 + 2,
    B_OBAR = B_PFULL0 + 2,
    B_DONE,
    B_COUNT
};
constexpr int kBarOff = kStageOff + kStages * kStageBytes;
constexpr int kMiscOff = kBarOff + B_COUNT * 8;  // TMEM base address, abort flag
constexpr int kSmemBytes = kMiscOff + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ bool mine(const TaskInfo &f, const AttnParams &p) {
    return xy::is_tile_task(f.t, p.G, HD);
}

__device__ __forceinline__ bool tile_ok(const TaskInfo &f, const AttnParams &p) {
    return xy::task_common_ok(f, p) && f.t.q_rows * p.G <= 128 && (f.t.kv_start % kTileKeys) == 0;
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

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

__global__ void __launch_bounds__(kThreads, 1)
    tile_attention_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const __grid_constant__ CUtensorMap qmap, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = xy::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    auto bar = [&](int i) -> uint32_t { return base + kBarOff + 8 * i; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kMiscOff + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        xy::mbar_init(bar(B_QFULL), 1);
        xy::mbar_init(bar(B_QEMPTY), 1);
        for (int s = 0; s < kStages; ++s) {
            xy::mbar_init(bar(B_KVFULL0 + s), 1);
            xy::mbar_init(bar(B_KVEMPTY0 + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            xy::mbar_init(bar(B_SFULL0 + b), 1);
            xy::mbar_init(bar(B_SFREE0 + b), 1);
            xy::mbar_init(bar(B_PFULL0 + b), 4);  // one arrival per softmax warp
        }
        xy::mbar_init(bar(B_OBAR), 1);
        xy::mbar_init(bar(B_DONE), 1);
        *abort_flag = 0;
        xy::fence_mbarrier_init();
    }
    if (warp == kMmaWarp) {
        xy::tmem_alloc(base + kMiscOff, kTmemCols);
        xy::tmem_relinquish();
    }
    xy::tc_fence_before();
    __syncthreads();
    xy::tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const int BRt = p.bs < kTileKeys ? p.bs : kTileKeys;  // keys per K/V box

    if (warp == kProducerWarp) {
        // ---------------------------------- producer ----------------------------------
        if (lane == 0) {
            xy::prefetch_tensormap(&kmap);
            xy::prefetch_tensormap(&vmap);
            xy::prefetch_tensormap(&qmap);
        }
        auto load_win = [&](const int32_t *row, int b0) -> int {
            const int idx = b0 + lane;
            return (idx >= 0 && idx < p.MB) ? __ldg(row + idx) : -1;
        };
        int ctr = 0, qk = 0;
        bool ok = true;
        int pref_win = -1;
        bool pref_valid = false;
        TaskCursor tc;
        tc.begin(p);
        while (tc.have && ok) {
            tc.load_next_record(p);
            bool run = mine(tc.cur, p);
            if (run && !tile_ok(tc.cur, p)) {
                if (lane == 0) xy::set_err(p.err, XY_DEV_BAD_TASK);
                run = false;
            }
            if (!run) {
                pref_valid = false;
                tc.advance(p);
                continue;
            }
            const TaskInfo f = tc.cur;
            const xy_task &t = f.t;
            if (qk > 0 && !warp_all(xy::mbar_wait(bar(B_QEMPTY), (qk - 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            if (lane == 0) {
                xy::mbar_arrive_expect_tx(bar(B_QFULL), kTileBytes);
                const int y = t.kv_head * p.G, z = f.seq_start + t.q_start;
                xy::tma_load_3d(base + kQOff, &qmap, 0, y, z, bar(B_QFULL));
                xy::tma_load_3d(base + kQOff + kHalfBytes, &qmap, 64, y, z, bar(B_QFULL));
            }
            ++qk;
            const int32_t *bt_row = p.bt + (int64_t)t.seq * p.MB;
            int win0 = t.kv_start / p.bs;
            int pg_win = pref_valid ? pref_win : load_win(bt_row, win0);
            int pg_nxt = load_win(bt_row, win0 + 32);
            pref_valid = false;
            bool first = true;
            for (int kv0 = t.kv_start; kv0 < t.kv_end; kv0 += kTileKeys, ++ctr) {
                const int s = ctr % kStages;
                if (ctr >= kStages &&
                    !warp_all(xy::mbar_wait(bar(B_KVEMPTY0 + s), ((ctr / kStages) - 1) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                const int nkeys = min(kTileKeys, t.kv_end - kv0);
                const int nbox = (nkeys + BRt - 1) / BRt;
                if ((kv0 + nkeys - 1) / p.bs - win0 >= 32) {
                    win0 += 32;
                    pg_win = pg_nxt;
                    pg_nxt = load_win(bt_row, win0 + 32);
                }
                const int n_copies = nbox * 4;  // (page box) x (2 halves) x (K, V)
                const int b = lane % nbox;
                int my_pg = __shfl_sync(0xffffffffu, pg_win, (kv0 + b * BRt) / p.bs - win0);
                if (lane < n_copies && (my_pg < 0 || my_pg >= p.P)) {
                    xy::set_err(p.err, XY_DEV_PAGE_OOB);
                    my_pg = 0;
                }
                if (lane == 0) xy::mbar_arrive_expect_tx(bar(B_KVFULL0 + s), (uint32_t)(n_copies * BRt * 128));
                __syncwarp();
                if (lane < n_copies) {
                    const int rest = lane / nbox;
                    const int half = rest & 1, tensor = rest >> 1;
                    const int key = kv0 + b * BRt;
                    const int y = (my_pg * p.Hkv + t.kv_head) * p.bs + (key % p.bs);
                    const uint32_t dst =
                        base + kStageOff + s * kStageBytes + tensor * kTileBytes + half * kHalfBytes + b * BRt * 128;
                    xy::tma_load_2d(dst, tensor ? &vmap : &kmap, half * 64, y, bar(B_KVFULL0 + s));
                }
                __syncwarp();
                if (first) {
                    first = false;
                    tc.prefetch_next(p);
                    if (tc.have_next) {
                        const xy_task &tn = tc.nxt.t;
                        pref_valid = tn.seq >= 0 && tn.seq < p.S && tn.kv_start >= 0;
                        if (pref_valid) pref_win = load_win(p.bt + (int64_t)tn.seq * p.MB, tn.kv_start / p.bs);
                    }
                }
            }
            tc.advance(p);
        }
        if (!ok) {
            if (lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
            *abort_flag = 1;
        }
        // every issued copy must land before the CTA may exit
        for (int k = ctr - 1; k >= 0 && k >= ctr - kStages; --k)
            xy::mbar_wait(bar(B_KVFULL0 + k % kStages), (k / kStages) & 1);
        if (qk > 0) xy::mbar_wait(bar(B_QFULL), (qk - 1) & 1);
    } else if (warp == kMmaWarp) {
        // ---------------------------------- MMA issuer ----------------------------------
        if (lane == 0) {
            const uint32_t id_s = xy::idesc_bf16(128, 128, 0, 0);   // Q (K-major) x K tile (K-major)
            const uint32_t id_o = xy::idesc_bf16(128, 128, 0, 1);   // P (TMEM) x V tile (MN-major)
            int ctr = 0, g = 0, qk = 0;
            bool ok = true, issued = false;
            auto issue_pv = [&](int jj) -> bool {
                const int gb = g + jj, b = gb & 1;
                if (!xy::mbar_wait(bar(B_PFULL0 + b), (gb >> 1) & 1, abort_flag)) return false;
                xy::tc_fence_after();
                const int s = (ctr + jj) % kStages;
                const uint32_t vst = base + kStageOff + s * kStageBytes + kTileBytes;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    xy::umma_ts(tbase + kTmemO, tbase + b * 128 + k * 8, xy::smem_desc_sw128(vst + k * 2048, kHalfBytes, 1024),
                                id_o, (jj > 0 || k > 0) ? 1u : 0u);
                xy::umma_commit(bar(B_KVEMPTY0 + s));
                xy::umma_commit(bar(B_SFREE0 + b));
                xy::umma_commit(bar(B_OBAR));
                return true;
            };
            TaskCursor tc;
            tc.begin(p);
            while (tc.have && ok) {
                tc.load_next_record(p);
                if (!mine(tc.cur, p) || !tile_ok(tc.cur, p)) {
                    tc.advance(p);
                    continue;
                }
                const xy_task t = tc.cur.t;
                const int n = (t.kv_end - t.kv_start + kTileKeys - 1) / kTileKeys;
                if (!xy::mbar_wait(bar(B_QFULL), qk & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                xy::tc_fence_after();
                tc.prefetch_next(p);
                for (int j = 0; j < n && ok; ++j) {
                    const int s = (ctr + j) % kStages;
                    if (!xy::mbar_wait(bar(B_KVFULL0 + s), ((ctr + j) / kStages) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int gb = g + j, b = gb & 1;
                    if (gb >= 2 && !xy::mbar_wait(bar(B_SFREE0 + b), ((gb >> 1) - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    xy::tc_fence_after();
                    issued = true;
                    const uint32_t kst = base + kStageOff + s * kStageBytes;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t koff = (k >> 2) * kHalfBytes + (k & 3) * 32;
                        xy::umma_ss(tbase + b * 128, xy::smem_desc_sw128(base + kQOff + koff, 16, 1024),
                                    xy::smem_desc_sw128(kst + koff, 16, 1024), id_s, k > 0 ? 1u : 0u);
                    }
                    xy::umma_commit(bar(B_SFULL0 + b));
                    if (j >= 1) ok = issue_pv(j - 1);
                }
                if (ok) ok = issue_pv(n - 1);
                xy::umma_commit(bar(B_QEMPTY));
                g += n;
                ctr += n;
                ++qk;
                tc.advance(p);
            }
            if (!ok) {
                xy::set_err(p.err, XY_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            if (issued) {  // everything issued has completed before TMEM is freed
                xy::umma_commit(bar(B_DONE));
                xy::mbar_wait(bar(B_DONE), 0);
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---------------------------------- softmax ----------------------------------
        const int row = warp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        int ctr = 0, g = 0;
        bool ok = true;
        TaskCursor tc;
        tc.begin(p);
        while (tc.have && ok) {
            tc.load_next_record(p);
            if (!mine(tc.cur, p) || !tile_ok(tc.cur, p)) {
                tc.advance(p);
                continue;
            }
            const TaskInfo f = tc.cur;
            const xy_task t = f.t;
            const int R = t.q_rows * p.G;
            const int n = (t.kv_end - t.kv_start + kTileKeys - 1) / kTileKeys;
            const bool valid = row < R;
            const int lim = valid ? min(t.kv_end, p.causal ? f.L - f.qn + t.q_start + row / p.G + 1 : f.L) : t.kv_end;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                const int gb = g + j, b = gb & 1;
                if (!warp_all(xy::mbar_wait(bar(B_SFULL0 + b), (gb >> 1) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                xy::tc_fence_after();
                if (j == 0) tc.prefetch_next(p);
                const int kt0 = t.kv_start + j * kTileKeys;
                uint32_t sr[128];
                xy::tmem_ld128(tbase + lane_off + b * 128, sr);
                // masked row max (keys at or past this row's limit are -inf), eight independent chains
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
                if (kt0 + kTileKeys <= lim) {
#pragma unroll
                    for (int i = 0; i < 128; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[i]));
                } else {
#pragma unroll
                    for (int i = 0; i < 128; ++i) {
                        if (kt0 + i >= lim) sr[i] = __float_as_uint(-INFINITY);
                        mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[i]));
                    }
                }
                const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                const float m_new = fmaxf(m, mx * p.scale_log2);  // the scale is positive
                if (__any_sync(0xffffffffu, m_new > m + kRescaleThreshold)) {
                    const float alpha = m_new == -INFINITY ? 1.f : ex2(m - m_new);
                    m = m_new;
                    l *= alpha;
                    if (j > 0) {  // O has PV_0..PV_{j-1}; rescale it once the last of them is done
                        if (!warp_all(xy::mbar_wait(bar(B_OBAR), (g + j - 1) & 1, abort_flag))) {
                            ok = false;
                            break;
                        }
                        xy::tc_fence_after();
#pragma unroll 1
                        for (int h = 0; h < 4; ++h) {
                            uint32_t orow[32];
                            xy::tmem_ld32(tbase + lane_off + kTmemO + h * 32, orow);
#pragma unroll
                            for (int i = 0; i < 32; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * alpha);
                            xy::tmem_st32(tbase + lane_off + kTmemO + h * 32, orow);
                        }
                    }
                }
                // p = 2^(s * scale_log2 - m), packed to bf16 pairs, written over the S columns
                const float neg_mu = m == -INFINITY ? 0.f : -m;
                float ls4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float p0 = ex2(fmaf(__uint_as_float(sr[64 * h + 2 * i]), p.scale_log2, neg_mu));
                        const float p1 = ex2(fmaf(__uint_as_float(sr[64 * h + 2 * i + 1]), p.scale_log2, neg_mu));
                        ls4[i & 3] += p0 + p1;
                        pk[i] = xy::pack_bf16x2(p0, p1);
                    }
                    xy::tmem_st32(tbase + lane_off + b * 128 + 32 * h, pk);
                }
                const float ls = (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
                l += ls;
                if (kt0 + kTileKeys > t.kv_end) {
                    // keys at or past kv_end: unused page slots or stale stage data; their P is 0 and
                    // their V rows are zeroed so that 0 * NaN cannot reach O
                    if (kt0 + row >= t.kv_end) {
                        const int s = (ctr + j) % kStages;
                        uint8_t *vrow = gbase + kStageOff + s * kStageBytes + kTileBytes + row * 128;
                        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            reinterpret_cast<uint4 *>(vrow)[i] = z;
                            reinterpret_cast<uint4 *>(vrow + kHalfBytes)[i] = z;
                        }
                    }
                    xy::fence_async_smem();
                }
                xy::tc_fence_before();
                __syncwarp();
                if (lane == 0) xy::mbar_arrive(bar(B_PFULL0 + b));
            }
            if (!ok) break;
            if (!warp_all(xy::mbar_wait(bar(B_OBAR), (g + n - 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            xy::tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            if (t.num_splits == 1) {
                const int64_t tok = f.seq_start + t.q_start + row / p.G;
                const int h = t.kv_head * p.G + row % p.G;
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + (tok * p.Hq + h) * HD);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    xy::tmem_ld32(tbase + lane_off + kTmemO + c * 32, r);
                    if (valid) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 w;
                            w.x = xy::pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv, __uint_as_float(r[8 * v + 1]) * inv);
                            w.y = xy::pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv);
                            w.z = xy::pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv);
                            w.w = xy::pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv);
                            dst[c * 4 + v] = w;
                        }
                    }
                }
            } else {
                const int64_t wr = (int64_t)t.ws_row + row;
                float4 *dst = reinterpret_cast<float4 *>(p.ws_o + wr * HD);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    xy::tmem_ld32(tbase + lane_off + kTmemO + c * 32, r);
                    if (valid) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            dst[c * 8 + v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                                         __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
                    }
                }
                if (valid) p.ws_lse[wr] = l > 0.f ? m + __log2f(l) : -INFINITY;
            }
            g += n;
            ctr += n;
            tc.advance(p);
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
        }
    }

    xy::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        xy::tc_fence_after();
        xy::tmem_dealloc(tbase, kTmemCols);
    }
}

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

}  // namespace

namespace xy {

xy_status launch_tile_attention(const AttnParams &p, const void *k_pages, const void *v_pages, int num_pages,
                                int block_size, int num_ctas, cudaStream_t st) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return XY_ERR_CUDA;
    const int64_t rows = (int64_t)num_pages * p.Hkv * block_size;
    const int br = block_size < kTileKeys ? block_size : kTileKeys;
    // K/V pools as [rows, 128] bf16; a box is 64 columns x br rows (one page, or half of a 256-key page)
    CUtensorMap km, vm, qm;
    cuuint64_t kdims[2] = {(cuuint64_t)HD, (cuuint64_t)rows};
    cuuint64_t kstr[1] = {(cuuint64_t)HD * 2};
    cuuint32_t kbox[2] = {64u, (cuuint32_t)br};
    cuuint32_t e2[2] = {1u, 1u};
    if (fn(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(k_pages), kdims, kstr, kbox, e2,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return XY_ERR_CUDA;
    if (fn(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(v_pages), kdims, kstr, kbox, e2,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return XY_ERR_CUDA;
    // queries as (128 columns, Hq heads, T tokens); a box is one 64-column half of G heads x 128/G tokens,
    // i.e. the task's 128 rows in (token, head) order; tokens past T read as zero
    cuuint64_t qdims[3] = {(cuuint64_t)HD, (cuuint64_t)p.Hq, (cuuint64_t)p.T};
    cuuint64_t qstr[2] = {(cuuint64_t)HD * 2, (cuuint64_t)p.Hq * HD * 2};
    cuuint32_t qbox[3] = {64u, (cuuint32_t)p.G, (cuuint32_t)(128 / p.G)};
    cuuint32_t e3[3] = {1u, 1u, 1u};
    if (fn(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16 *>(p.q), qdims, qstr, qbox, e3,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return XY_ERR_CUDA;
    static int configured_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return XY_ERR_CUDA;
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(tile_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
            cudaSuccess)
            return XY_ERR_CUDA;
        configured_device = dev;
    }
    tile_attention_kernel<<<num_ctas, kThreads, kSmemBytes, st>>>(km, vm, qm, p);
    return cudaGetLastError() == cudaSuccess ? XY_OK : XY_ERR_CUDA;
}

}  // namespace xy
