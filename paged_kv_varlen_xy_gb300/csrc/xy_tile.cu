// Tensor-core (tcgen05 / TMEM) tiles of the paged attention: the prefill and chunk tasks, whose
// (token, head) rows fill a 128-row MMA tile.  The decode-sized tasks run in xy_attention.cu.
//
// "XY-Serve 深度实战" (chenxutan.com/d/5031) §2.2 component 3: Meta-Attention is one fused
// GEMM-softmax-GEMM over a task's (query block x KV block) tiles; §2.3 technique 1: ragged tiles
// are masked on chip and only valid rows are stored.
//
// One persistent CTA per SM, eighteen warps:
//   warp 16     producer: TMA loads of the task's 128 query rows (G heads x 128/G tokens, one 3-D
//               box per 64-column half) into one of two Q buffers, and of 128-key K and V tiles,
//               gathered page by page through the block table (2-D boxes, 128-byte swizzle), into
//               a 4-slot ring (K_j and V_j take separate slots, so K runs ahead of V);
//   warp 17     MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM buffers, then
//               O += P_{j-1} V_{j-1} with P read from TMEM (packed bf16, two buffers of its own,
//               so the next S never waits for a PV);
//   warps 0..15 softmax, four threads per query row (TMEM lane = row; warps 4q..4q+3 take key
//               columns 32q..32q+31), the row max exchanged through shared memory:
//               masked max, exp2, row sum, P back to TMEM.  O is rescaled in TMEM only when a row's
//               running max grows by more than 2^8 (otherwise the stale max is kept, which is exact
//               because O and the row sum share it).  Epilogue: O / l from TMEM to global memory.
// TMEM: S0 = columns [0,128), S1 = [128,256), P0 = [256,320), P1 = [320,384), O = [384,512).
// The softmax warps release an S buffer as soon as they have loaded it, so S_{j+2} overlaps the
// softmax and PV of tile j.

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
constexpr int kSlots = 4;                       // K/V ring slots (one K or V tile each)
constexpr int kSoftmaxWarps = 16;               // kQ threads per query row
constexpr int kQ = kSoftmaxWarps / 4;
constexpr int kCols = 128 / kQ;                 // S / O columns per softmax thread
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
static_assert(kCols == 32, "the softmax code moves 32 TMEM columns per thread");
constexpr int kHalfBytes = 128 * 128;           // 128 rows x 64 bf16 columns
constexpr int kTileBytes = 2 * kHalfBytes;      // Q, K or V tile: [half][128 rows][128 B]
constexpr int kQOff = 0;                        // Q0, Q1
constexpr int kSlotOff = 2 * kTileBytes;
enum {
    B_QFULL0 = 0,
    B_QEMPTY0 = B_QFULL0 + 2,
    B_FULL0 = B_QEMPTY0 + 2,
    B_EMPTY0 = B_FULL0 + kSlots,
    B_SFULL0 = B_EMPTY0 + kSlots,
    B_SFREE0 = B_SFULL0 + 2,
    B_PFULL0 = B_SFREE0 + 2,
    B_PFREE0 = B_PFULL0 + 2,
    B_OFREE = B_PFREE0 + 2,
    B_OBAR,
    B_DONE,
    B_COUNT
};
constexpr int kBarOff = kSlotOff + kSlots * kTileBytes;
constexpr int kMiscOff = kBarOff + B_COUNT * 8;     // TMEM base address, abort flag
constexpr int kVoteOff = kMiscOff + 16;              // one vote per softmax warp
constexpr int kRedOff = kVoteOff + 4 * kSoftmaxWarps; // row-max exchange [2 parity][kQ][128]
constexpr int kSumOff = kRedOff + 2 * kQ * 128 * 4;  // row-sum exchange [kQ][128]
constexpr int kSmemBytes = kSumOff + kQ * 128 * 4 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemP = 256;
constexpr uint32_t kTmemO = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kSoftmaxBar = 1;        // named barrier id of the softmax warps

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
    volatile int *vote = reinterpret_cast<volatile int *>(gbase + kVoteOff);
    float *red = reinterpret_cast<float *>(gbase + kRedOff);
    float *sums = reinterpret_cast<float *>(gbase + kSumOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            xy::mbar_init(bar(B_QFULL0 + i), 1);
            xy::mbar_init(bar(B_QEMPTY0 + i), 1);
            xy::mbar_init(bar(B_SFULL0 + i), 1);
            xy::mbar_init(bar(B_SFREE0 + i), kSoftmaxWarps);
            xy::mbar_init(bar(B_PFULL0 + i), kSoftmaxWarps);
            xy::mbar_init(bar(B_PFREE0 + i), 1);
        }
        xy::mbar_init(bar(B_OFREE), kSoftmaxWarps);
        for (int s = 0; s < kSlots; ++s) {
            xy::mbar_init(bar(B_FULL0 + s), 1);
            xy::mbar_init(bar(B_EMPTY0 + s), 1);
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
        int c = 0, qk = 0;
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
            const int qb = qk & 1;
            if (qk >= 2 && !warp_all(xy::mbar_wait(bar(B_QEMPTY0 + qb), ((qk >> 1) - 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            if (lane == 0) {
                xy::mbar_arrive_expect_tx(bar(B_QFULL0 + qb), kTileBytes);
                const int y = t.kv_head * p.G, z = f.seq_start + t.q_start;
                const uint32_t qdst = base + kQOff + qb * kTileBytes;
                xy::tma_load_3d(qdst, &qmap, 0, y, z, bar(B_QFULL0 + qb));
                xy::tma_load_3d(qdst + kHalfBytes, &qmap, 64, y, z, bar(B_QFULL0 + qb));
            }
            ++qk;
            const int32_t *bt_row = p.bt + (int64_t)t.seq * p.MB;
            int win0 = t.kv_start / p.bs;
            int pg_win = pref_valid ? pref_win : load_win(bt_row, win0);
            int pg_nxt = load_win(bt_row, win0 + 32);
            pref_valid = false;
            bool first = true;
            for (int kv0 = t.kv_start; kv0 < t.kv_end && ok; kv0 += kTileKeys) {
                const int nkeys = min(kTileKeys, t.kv_end - kv0);
                const int nbox = (nkeys + BRt - 1) / BRt;
                if ((kv0 + nkeys - 1) / p.bs - win0 >= 32) {
                    win0 += 32;
                    pg_win = pg_nxt;
                    pg_nxt = load_win(bt_row, win0 + 32);
                }
                const int b = lane % nbox;
                int my_pg = __shfl_sync(0xffffffffu, pg_win, (kv0 + b * BRt) / p.bs - win0);
                const int n_copies = nbox * 2;  // (page box) x (2 halves), per tensor
                if (lane < n_copies && (my_pg < 0 || my_pg >= p.P)) {
                    xy::set_err(p.err, XY_DEV_PAGE_OOB);
                    my_pg = 0;
                }
                const int y = (my_pg * p.Hkv + t.kv_head) * p.bs + ((kv0 + b * BRt) % p.bs);
                const int half = lane / nbox;
#pragma unroll
                for (int tensor = 0; tensor < 2; ++tensor, ++c) {
                    const int s = c % kSlots;
                    if (c >= kSlots &&
                        !warp_all(xy::mbar_wait(bar(B_EMPTY0 + s), ((c / kSlots) - 1) & 1, abort_flag))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) xy::mbar_arrive_expect_tx(bar(B_FULL0 + s), (uint32_t)(n_copies * BRt * 128));
                    __syncwarp();
                    if (lane < n_copies) {
                        const uint32_t dst = base + kSlotOff + s * kTileBytes + half * kHalfBytes + b * BRt * 128;
                        xy::tma_load_2d(dst, tensor ? &vmap : &kmap, half * 64, y, bar(B_FULL0 + s));
                    }
                    __syncwarp();
                }
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
        for (int k = c - 1; k >= 0 && k >= c - kSlots; --k)
            xy::mbar_wait(bar(B_FULL0 + k % kSlots), (k / kSlots) & 1);
        for (int k = qk - 1; k >= 0 && k >= qk - 2; --k) xy::mbar_wait(bar(B_QFULL0 + (k & 1)), (k >> 1) & 1);
    } else if (warp == kMmaWarp) {
        // ---------------------------------- MMA issuer ----------------------------------
        if (lane == 0) {
            const uint32_t id_s = xy::idesc_bf16(128, 128, 0, 0);   // Q (K-major) x K tile (K-major)
            const uint32_t id_o = xy::idesc_bf16(128, 128, 0, 1);   // P (TMEM) x V tile (MN-major)
            int c = 0, g = 0, qk = 0;
            bool ok = true, issued = false;
            // Descriptors are built once; a k-step or a buffer only adds a constant to the 14-bit
            // address field (addresses stay below 256 KB), so the issue loop is a few adds per MMA
            // and the single issuing thread keeps up with the tensor core.
            const uint64_t q_desc0 = xy::smem_desc_sw128(base + kQOff, 16, 1024);
            const uint64_t k_desc0 = xy::smem_desc_sw128(base + kSlotOff, 16, 1024);
            const uint64_t v_desc0 = xy::smem_desc_sw128(base + kSlotOff, kHalfBytes, 1024);
            constexpr uint32_t kTileDesc = kTileBytes >> 4;  // one Q buffer or ring slot
            auto issue_pv = [&](int jj, uint32_t o_addr) -> bool {
                const int gb = g + jj, b = gb & 1;
                if (jj == 0 && qk >= 1 && !xy::mbar_wait(bar(B_OFREE), (qk - 1) & 1, abort_flag))
                    return false;  // the previous task's epilogue has read O
                if (!xy::mbar_wait(bar(B_PFULL0 + b), (gb >> 1) & 1, abort_flag)) return false;
                const int cv = c + 2 * jj + 1, s = cv % kSlots;
                if (!xy::mbar_wait(bar(B_FULL0 + s), (cv / kSlots) & 1, abort_flag)) return false;
                xy::tc_fence_after();
                const uint64_t vd = v_desc0 + (uint64_t)(s * kTileDesc);
                const uint32_t pa = tbase + kTmemP + b * 64;
                xy::umma_ts(o_addr, pa, vd, id_o, jj > 0 ? 1u : 0u);
#pragma unroll
                for (int k = 1; k < 8; ++k) xy::umma_ts(o_addr, pa + k * 8, vd + (uint64_t)(k * (2048 >> 4)), id_o, 1u);
                xy::umma_commit(bar(B_EMPTY0 + s));
                xy::umma_commit(bar(B_PFREE0 + b));
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
                const int qb = qk & 1;
                const uint32_t o_addr = tbase + kTmemO;
                if (!xy::mbar_wait(bar(B_QFULL0 + qb), (qk >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                xy::tc_fence_after();
                tc.prefetch_next(p);
                for (int j = 0; j < n && ok; ++j) {
                    const int ck = c + 2 * j, s = ck % kSlots;
                    if (!xy::mbar_wait(bar(B_FULL0 + s), (ck / kSlots) & 1, abort_flag)) {
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
                    const uint64_t qd = q_desc0 + (uint64_t)(qb * kTileDesc);
                    const uint64_t kd = k_desc0 + (uint64_t)(s * kTileDesc);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint64_t koff = (uint64_t)(((k >> 2) * kHalfBytes + (k & 3) * 32) >> 4);
                        xy::umma_ss(tbase + b * 128, qd + koff, kd + koff, id_s, k > 0 ? 1u : 0u);
                    }
                    xy::umma_commit(bar(B_EMPTY0 + s));
                    xy::umma_commit(bar(B_SFULL0 + b));
                    if (j == n - 1) xy::umma_commit(bar(B_QEMPTY0 + qb));
                    if (j >= 1) ok = issue_pv(j - 1, o_addr);
                }
                if (ok) ok = issue_pv(n - 1, o_addr);
                g += n;
                c += 2 * n;
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
    } else {
        // ---------------------------------- softmax ----------------------------------
        const int q4 = warp >> 2;                   // key columns [kCols*q4, kCols*q4 + kCols)
        const int row = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const int col0 = kCols * q4;
        int c = 0, g = 0, qk = 0;
        bool ok = true;
        TaskCursor tc;
        tc.begin(p);
        while (tc.have) {
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
            const uint32_t o_addr = tbase + lane_off + kTmemO + col0;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                const int gb = g + j, b = gb & 1;
                // a failed wait (timeout or abort) is recorded, not acted on: every softmax warp
                // keeps executing the same named barriers and the decision to stop is voted below
                ok = warp_all(xy::mbar_wait(bar(B_SFULL0 + b), (gb >> 1) & 1, abort_flag)) && ok;
                xy::tc_fence_after();
                if (j == 0) tc.prefetch_next(p);
                const int kt0 = t.kv_start + j * kTileKeys + col0;
                uint32_t sr[kCols];
                xy::tmem_ld32(tbase + lane_off + b * 128 + col0, sr);
                xy::tc_fence_before();
                __syncwarp();
                if (lane == 0) xy::mbar_arrive(bar(B_SFREE0 + b));  // S_b may be overwritten now
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (kt0 + kCols <= lim) {
#pragma unroll
                    for (int i = 0; i < kCols; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(sr[i]));
                } else {
#pragma unroll
                    for (int i = 0; i < kCols; ++i) {
                        if (kt0 + i >= lim) sr[i] = __float_as_uint(-INFINITY);
                        mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(sr[i]));
                    }
                }
                float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                // exchange the partial row maxima of the kQ threads of a row
                float *rd = red + (gb & 1) * (kQ * 128);
                rd[q4 * 128 + row] = mx;
                xy::named_bar_sync(kSoftmaxBar, kSoftmaxWarps * 32);
#pragma unroll
                for (int o = 1; o < kQ; ++o) mx = fmaxf(mx, rd[((q4 + o) % kQ) * 128 + row]);
                const float m_new = fmaxf(m, mx * p.scale_log2);  // the scale is positive
                if (__any_sync(0xffffffffu, m_new > m + kRescaleThreshold)) {
                    const float alpha = m_new == -INFINITY ? 1.f : ex2(m - m_new);
                    m = m_new;
                    l *= alpha;
                    if (j > 0) {  // O has PV_0..PV_{j-1}; rescale these columns once the last one is done
                        ok = warp_all(xy::mbar_wait(bar(B_OBAR), (gb - 1) & 1, abort_flag)) && ok;
                        xy::tc_fence_after();
                        uint32_t orow[kCols];
                        xy::tmem_ld32(o_addr, orow);
#pragma unroll
                        for (int i = 0; i < kCols; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * alpha);
                        xy::tmem_st32(o_addr, orow);
                    }
                }
                // p = 2^(s * scale_log2 - m), packed to bf16 pairs, into this thread's P columns
                const float neg_mu = m == -INFINITY ? 0.f : -m;
                float ls4[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[kCols / 2];
#pragma unroll
                for (int i = 0; i < kCols / 2; ++i) {
                    const float p0 = ex2(fmaf(__uint_as_float(sr[2 * i]), p.scale_log2, neg_mu));
                    const float p1 = ex2(fmaf(__uint_as_float(sr[2 * i + 1]), p.scale_log2, neg_mu));
                    ls4[i & 3] += p0 + p1;
                    pk[i] = xy::pack_bf16x2(p0, p1);
                }
                if (gb >= 2) {  // P_b is free once PV of tile gb-2 has read it
                    ok = warp_all(xy::mbar_wait(bar(B_PFREE0 + b), ((gb >> 1) - 1) & 1, abort_flag)) && ok;
                    xy::tc_fence_after();
                }
                xy::tmem_st16(tbase + lane_off + kTmemP + b * 64 + (kCols / 2) * q4, pk);
                l += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
                if (t.kv_start + (j + 1) * kTileKeys > t.kv_end) {
                    // keys at or past kv_end: unused page slots or stale data; their P is 0 and their V
                    // rows are zeroed so that 0 * NaN cannot occur.  The V tile has its own slot: wait
                    // for its copy to land first.  This thread zeroes its row's kCols columns, which in
                    // the 128-byte swizzle are 16-byte chunks (q4 % 2) * 4 .. +3 XOR (row & 7).
                    const int cv = c + 2 * j + 1, s = cv % kSlots;
                    ok = warp_all(xy::mbar_wait(bar(B_FULL0 + s), (cv / kSlots) & 1, abort_flag)) && ok;
                    if (t.kv_start + j * kTileKeys + row >= t.kv_end) {
                        uint4 *vrow = reinterpret_cast<uint4 *>(gbase + kSlotOff + s * kTileBytes +
                                                                (col0 >> 6) * kHalfBytes + row * 128);
                        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int i = 0; i < kCols / 8; ++i) vrow[(((col0 & 63) >> 3) + i) ^ (row & 7)] = z;
                    }
                    xy::fence_async_smem();
                }
                xy::tc_fence_before();
                __syncwarp();
                if (lane == 0) xy::mbar_arrive(bar(B_PFULL0 + b));
            }
            ok = warp_all(xy::mbar_wait(bar(B_OBAR), (g + n - 1) & 1, abort_flag)) && ok;
            xy::tc_fence_after();
            // row sums of the kQ threads of a row, and the vote on whether to go on
            sums[q4 * 128 + row] = l;
            if (lane == 0) vote[warp] = ok ? 0 : 1;
            xy::named_bar_sync(kSoftmaxBar, kSoftmaxWarps * 32);
            float L = l;
#pragma unroll
            for (int o = 1; o < kQ; ++o) L += sums[((q4 + o) % kQ) * 128 + row];
            int bad = 0;
#pragma unroll
            for (int w = 0; w < kSoftmaxWarps; ++w) bad |= vote[w];
            const float inv = L > 0.f ? 1.f / L : 0.f;
            uint32_t r[kCols];
            xy::tmem_ld32(o_addr, r);
            if (valid && !bad) {
                if (t.num_splits == 1) {
                    const int64_t tok = f.seq_start + t.q_start + row / p.G;
                    const int h = t.kv_head * p.G + row % p.G;
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (tok * p.Hq + h) * HD + col0);
#pragma unroll
                    for (int v = 0; v < kCols / 8; ++v) {
                        uint4 w;
                        w.x = xy::pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv, __uint_as_float(r[8 * v + 1]) * inv);
                        w.y = xy::pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv);
                        w.z = xy::pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv);
                        w.w = xy::pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv);
                        dst[v] = w;
                    }
                } else {
                    const int64_t wr = (int64_t)t.ws_row + row;
                    float4 *dst = reinterpret_cast<float4 *>(p.ws_o + wr * HD + col0);
#pragma unroll
                    for (int v = 0; v < kCols / 4; ++v)
                        dst[v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                             __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
                    if (q4 == 0) p.ws_lse[wr] = L > 0.f ? m + __log2f(L) : -INFINITY;
                }
            }
            xy::tc_fence_before();
            __syncwarp();
            if (lane == 0) xy::mbar_arrive(bar(B_OFREE));
            g += n;
            c += 2 * n;
            ++qk;
            if (bad) {
                *abort_flag = 1;
                if (warp == 0 && lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
                break;
            }
            tc.advance(p);
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

void set_last_error(const char *what, const char *msg);

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
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail(cudaGetLastError(), "cudaGetDevice");
    if (configured_device != dev) {
        const cudaError_t e =
            cudaFuncSetAttribute(tile_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return cuda_fail(e, "tile_attention_kernel smem attribute");
        configured_device = dev;
    }
    tile_attention_kernel<<<num_ctas, kThreads, kSmemBytes, st>>>(km, vm, qm, p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? XY_OK : cuda_fail(e, "tile_attention_kernel launch");
}

}  // namespace xy
