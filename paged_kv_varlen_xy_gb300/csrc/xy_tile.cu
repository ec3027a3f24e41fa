// Tensor-core (tcgen05 / TMEM) tiles of the paged attention: the prefill and chunk tasks, whose
// (token, head) rows fill 128-row MMA tiles.  The decode-sized tasks run in xy_attention.cu.
//
// "XY-Serve 深度实战" (chenxutan.com/d/5031) §2.2 component 3: Meta-Attention is one fused
// GEMM-softmax-GEMM over a task's (query block x KV block) tiles; §2.3 technique 1: ragged tiles
// are masked on chip and only valid rows are stored.
//
// A task holds up to 256 (token, head) rows: query tile A (rows 0..127) and tile B (rows
// 128..255), both against the same 128-key K/V tiles, so each K/V tile loaded serves two MMA
// tiles.  One persistent CTA per SM, twelve warps in three warpgroups:
//   warp 8      producer: TMA loads of the task's query rows (G heads x 128/G tokens per tile,
//               one 3-D box per 64-column half) and of 128-key K and V tiles gathered page by
//               page through the block table (2-D boxes, 128-byte swizzle) into a 4-slot ring
//               (K_j and V_j take separate slots, so K runs ahead of V);
//   warp 9      MMA issuer (one thread), per K/V tile j:
//                 PV_A(j-1), S_A(j), PV_B(j-1), S_B(j)
//               with S_X = Q_X K^T into TMEM and O_X += P_X V, P_X read from TMEM where the
//               softmax wrote it over the first 64 columns of S_X (the MMAs of one thread run in
//               issue order, so PV_X(j-1) has read P_X before S_X(j) overwrites it);
//   warps 0..3  softmax of tile A, warps 4..7 softmax of tile B: one query row per thread (TMEM
//               lane = row), masked row max, exp2, row sum, P back to TMEM.  While one group
//               works, the tensor core runs the other tile's MMAs.  O_X is rescaled in TMEM only
//               when a row's running max grows by more than 2^8 (otherwise the stale max is kept,
//               which is exact because O and the row sum share it).  Epilogue: O / l from TMEM,
//               staged in shared memory and written by TMA stores for whole query tiles.
//               Warps 0..3 are also the math warps of decode-path tasks;
//   warp 10     second producer of the decode ring; warp 11 claims tasks under the dynamic deal.
// Registers: the CTA is launched with 168 per thread; the softmax warpgroups raise theirs to 200
// and the producer / MMA / scheduler warpgroup lowers its own to 104 (setmaxnreg), so that the
// softmax and decode-path code runs without spills.
// TMEM: S_A = columns [0,128), S_B = [128,256), O_A = [256,384), O_B = [384,512).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "xy.h"
#include "xy_attn_common.cuh"
#include "xy_decode_path.cuh"
#include "xy_device.cuh"

namespace {

using xy::AttnParams;
using xy::ex2;
using xy::fetch_info;
using xy::TaskCursor;
using xy::TaskInfo;

constexpr int HD = 128;
constexpr int kTileKeys = 128;
constexpr int kClaimAheadKeys = 512;            // dynamic deal: see the producer's claim release
constexpr int kSlots = 4;                       // K/V ring slots (one K or V tile each)
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kDecProducerWarp = 10;   // second producer of the decode ring (odd stages)
constexpr int kSchedWarp = 11;         // dynamic deal only: claims tasks into the CTA's queue
constexpr int kThreads = 12 * 32;      // (the scheduler warp idles under the static deals)
// Registers per thread: launched with kLaunchRegs each, the softmax warpgroups (warps 0..7) raise
// theirs to kRegsSoftmax and the producer / MMA / scheduler warpgroup (8..11) lowers its own to
// kRegsControl; the budgets must fit in what the CTA was launched with.
constexpr int kLaunchRegs = (65536 / kThreads) & ~7;
constexpr uint32_t kRegsSoftmax = 200, kRegsControl = 104;
static_assert(2 * kRegsSoftmax + kRegsControl <= 3 * kLaunchRegs, "register split");
constexpr int kQueueReaders = 11;      // every warp but the scheduler reads every queue entry
constexpr int kHalfBytes = 128 * 128;           // 128 rows x 64 bf16 columns
constexpr int kTileBytes = 2 * kHalfBytes;      // one Q, K or V tile: [half][128 rows][128 B]
constexpr int kQOff = 0;                        // Q_A, Q_B
constexpr int kSlotOff = 2 * kTileBytes;
enum {
    B_QFULL = 0,
    B_QEMPTY,
    B_FULL0,
    B_EMPTY0 = B_FULL0 + kSlots,
    B_SFULL0 = B_EMPTY0 + kSlots,   // per query tile X
    B_PFULL0 = B_SFULL0 + 2,
    B_OBAR0 = B_PFULL0 + 2,
    B_OFREE0 = B_OBAR0 + 2,
    B_DONE = B_OFREE0 + 2,
    B_COUNT
};
// The decode path (tasks of at most XY_TILE_MIN_ROWS rows, xy_decode_path.cuh) uses the same
// bytes: its stage ring from offset 0 and its merge slots after it.  A switch of task kind waits
// until the other kind's consumers are done with shared memory.
using DecRing = xy::dec::Ring<HD, 4, (XY_TILE_MIN_ROWS + 15) / 16 * 16>;
static_assert(XY_TILE_MIN_ROWS <= DecRing::kMaxRows, "decode-path tasks of the unified kernel fit the ring");
constexpr int kDecStagesOff = 0;
constexpr int kDecSlotsOff = DecRing::kBytes;
// the epilogue's staging of bf16 output rows for the TMA store: one 64-column half of one query
// tile per softmax group (128 rows x 128 bytes, 128-byte swizzle), outside the decode path's bytes
constexpr int kStageOff = kSlotOff + kSlots * kTileBytes;
constexpr int kBarOff = kStageOff + 2 * kHalfBytes;
static_assert(kDecSlotsOff + DecRing::kSlotBytes <= kStageOff, "decode path fits below the output staging");
constexpr int kDecBarOff = kBarOff + B_COUNT * 8;    // decode ring full[4], empty[4], task-done[2]
constexpr int kMiscOff = kDecBarOff + (2 * DecRing::kStages + 2) * 8;  // TMEM base, abort flag, decode go
constexpr int kVoteOff = kMiscOff + 16;             // one vote per softmax warp, then 2 x 4 decode votes
constexpr int kQueueVoteOff = kVoteOff + 96;        // queue-read votes: [softmax group][2][4]
constexpr int kQueueOff = kQueueVoteOff + 64;       // the dynamic deal's claim queue
constexpr int kSmemBytes = kQueueOff + xy::TaskQueue::kBytes + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ bool mine(const TaskInfo &f, const AttnParams &p) {
    return xy::is_tile_task(f.t, p.G, HD);
}

__device__ __forceinline__ bool tile_ok(const TaskInfo &f, const AttnParams &p) {
    return xy::task_common_ok(f, p) && f.t.q_rows * p.G <= 256 && (f.t.kv_start % kTileKeys) == 0;
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

template <bool DYN>
__global__ void __launch_bounds__(kThreads, 1)
    meta_attention_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                          const __grid_constant__ CUtensorMap kmap_d,
                          const __grid_constant__ CUtensorMap vmap_d, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = xy::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    auto bar = [&](int i) -> uint32_t { return base + kBarOff + 8 * i; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kMiscOff + 4);
    // decode tasks 0 .. *dec_go - 1 may write the decode ring: the producer warp raises it once the
    // tile work before a decode task no longer reads shared memory (a count, so no phase aliasing)
    volatile int *dec_go = reinterpret_cast<volatile int *>(gbase + kMiscOff + 8);
    volatile int *vote = reinterpret_cast<volatile int *>(gbase + kVoteOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    xy::dec::Smem dsm;
    dsm.stages = base + kDecStagesOff;
    dsm.stages_gen = gbase + kDecStagesOff;
    dsm.slots = reinterpret_cast<float *>(gbase + kDecSlotsOff);
    dsm.full_bar = base + kDecBarOff;
    dsm.empty_bar = dsm.full_bar + DecRing::kStages * 8;
    dsm.abort_flag = abort_flag;
    dsm.vote = vote + 16;
    dsm.bar_id = 3;
    // decode task j done (math warps past its last shared-memory access): dec_done + 8 * (j & 1),
    // phase j >> 1.  Two barriers, and the producer confirms task j - 2 before issuing task j, so
    // every wait below is on the latest phase issued on its barrier and parity cannot alias.
    const uint32_t dec_done = base + kDecBarOff + 8 * (2 * DecRing::kStages);
    // dynamic deal: the claim queue every warp but the scheduler reads
    xy::TaskQueue dq;
    dq.bind(gbase + kQueueOff, base + kQueueOff, abort_flag);
    const xy::TaskQueue *q = DYN ? &dq : nullptr;

    if (threadIdx.x == 0) {
        xy::mbar_init(bar(B_QFULL), 1);
        xy::mbar_init(bar(B_QEMPTY), 1);
        for (int s = 0; s < kSlots; ++s) {
            xy::mbar_init(bar(B_FULL0 + s), 1);
            xy::mbar_init(bar(B_EMPTY0 + s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            xy::mbar_init(bar(B_SFULL0 + x), 1);
            xy::mbar_init(bar(B_PFULL0 + x), 4);   // the four warps of softmax group x
            xy::mbar_init(bar(B_OBAR0 + x), 1);
            xy::mbar_init(bar(B_OFREE0 + x), 4);
        }
        xy::mbar_init(bar(B_DONE), 1);
        for (int st = 0; st < DecRing::kStages; ++st) {
            xy::mbar_init(base + kDecBarOff + 8 * st, 1);
            xy::mbar_init(base + kDecBarOff + 8 * (DecRing::kStages + st), xy::dec::kMathWarps);
        }
        xy::mbar_init(dec_done, xy::dec::kMathWarps);
        xy::mbar_init(dec_done + 8, xy::dec::kMathWarps);
        if (DYN) dq.init(kQueueReaders);
        *abort_flag = 0;
        *dec_go = 0;
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
    // Under a dependent launch this kernel may run while the kernel ahead of it on the stream (the
    // step's KV append) still writes the new tokens' K/V rows: only the producer warps wait for it,
    // each before its first copy of such rows; everything else read here is not written by the
    // append.
    if (p.trace && threadIdx.x == 0) p.trace[4 * blockIdx.x] = xy::global_timer_ns();
    const int BRt = p.bs < kTileKeys ? p.bs : kTileKeys;  // keys per K/V box
    const int qt_tokens = 128 / p.G;                      // tokens per query tile

    // Each warpgroup sets its register budget once, at the head of its roles' code.
    if (warp >= kProducerWarp) {
    xy::setmaxnreg_dec<kRegsControl>();
    if (warp == kProducerWarp) {
        // ---------------------------------- producer ----------------------------------
        if (lane == 0) {
            xy::prefetch_tensormap(&kmap);
            xy::prefetch_tensormap(&vmap);
            xy::prefetch_tensormap(&qmap);
            xy::prefetch_tensormap(&omap);
            xy::prefetch_tensormap(&kmap_d);
            xy::prefetch_tensormap(&vmap_d);
        }
        auto load_win = [&](const int32_t *row, int b0) -> int {
            const int idx = b0 + lane;
            return (idx >= 0 && idx < p.MB) ? __ldg(row + idx) : -1;
        };
        int c = 0, qk = 0;          // tile path: ring slot uses, tasks
        int dctr = 0, nd = 0;       // decode path: stages issued, tasks
        int last_kind = 0;          // 1 tile, 2 decode
        bool ok = true, dep_ready = false;  // dep_ready: waited for the kernel ahead (the KV append)
        int pref_win = -1;
        bool pref_valid = false;
        unsigned long long n_run = 0, work = 0;  // trace: tasks issued and their rows x keys
        TaskCursor tc;
        tc.attach(q, false, true);  // the lead reader: its reads pace the claims
        // the next task is claimed once the current one has at most kClaimAheadKeys keys left to
        // issue: early enough for the claim's global reads to land before the ring drains
        tc.defer_taken = true;
        tc.begin(p);
        while (tc.have && ok) {
            tc.load_next_record(p);
            if (xy::is_hole(tc.cur.t)) {
                pref_valid = false;
                tc.advance(p);
                continue;
            }
            const bool tile = mine(tc.cur, p);
            if (!(tile ? tile_ok(tc.cur, p) : xy::dec::task_ok<DecRing>(tc.cur, p))) {
                if (lane == 0) xy::set_err(p.err, XY_DEV_BAD_TASK);
                pref_valid = false;
                tc.advance(p);
                continue;
            }
            ++n_run;
            work += (unsigned long long)(tc.cur.t.q_rows * p.G) *
                    (unsigned long long)(tc.cur.t.kv_end - tc.cur.t.kv_start);
            const int kind = tile ? 1 : 2;
            if (last_kind != 0 && kind != last_kind) {
                // The two paths share shared memory: before writing it for the other kind, wait
                // until the consumers of the previous kind are done with it.
                bool w = true;
                if (last_kind == 1) {  // the last tile task's MMAs have read Q and every slot
                    w = xy::mbar_wait(bar(B_QEMPTY), (qk - 1) & 1, abort_flag);
                    for (int k = c - 1; w && k >= 0 && k >= c - kSlots; --k)
                        w = xy::mbar_wait(bar(B_EMPTY0 + k % kSlots), (k / kSlots) & 1, abort_flag);
                } else {  // the math warps have finished the last decode task (merge slots included)
                    w = xy::mbar_wait(dec_done + 8 * ((nd - 1) & 1), ((nd - 1) >> 1) & 1, abort_flag);
                }
                if (!warp_all(w)) {
                    ok = false;
                    break;
                }
            }
            last_kind = kind;
            if (!tile) {
                if (nd >= 2 &&
                    !warp_all(xy::mbar_wait(dec_done + 8 * (nd & 1), ((nd - 2) >> 1) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                __threadfence_block();
                if (lane == 0) *dec_go = nd + 1;  // the second decode producer may write task nd
                const TaskInfo f = tc.cur;
                // the first block-table window: prefetched (static deal) or in the entry
                const bool have_first = DYN || pref_valid;
                const int first_win = DYN ? tc.win : pref_win;
                pref_valid = false;
                ok = xy::dec::produce_task<HD, DecRing>(p, f, &kmap_d, &vmap_d, nullptr, nullptr, dsm, dctr, lane, first_win, have_first, dep_ready,
                                                        [&]() {
                                                            tc.prefetch_next(p);
                                                            if (tc.have_next) {
                                                                const xy_task &tn = tc.nxt.t;
                                                                pref_valid = tn.seq >= 0 && tn.seq < p.S && tn.kv_start >= 0;
                                                                if (pref_valid)
                                                                    pref_win = xy::load_window(p, tn.seq, tn.kv_start / p.bs, lane);
                                                            }
                                                        },
                                                        0, 2, [&](int keys_left) {
                                                            if (keys_left <= kClaimAheadKeys) tc.release_claim();
                                                        });
                ++nd;
                tc.advance(p);
                continue;
            }
            const TaskInfo f = tc.cur;
            const xy_task &t = f.t;
            const bool has_b = t.q_rows * p.G > 128;
            // while the previous task's last S still reads the Q buffer, bring this task's query
            // rows into L2 (one prefetch per 64-column half of each query tile)
            if (qk >= 1 && lane < (has_b ? 4 : 2))
                xy::tma_prefetch_3d(&qmap, (lane & 1) * 64, t.kv_head * p.G, f.seq_start + t.q_start + (lane >> 1) * qt_tokens);
            if (qk >= 1 && !warp_all(xy::mbar_wait(bar(B_QEMPTY), (qk - 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            if (lane == 0) {
                xy::mbar_arrive_expect_tx(bar(B_QFULL), (has_b ? 2 : 1) * kTileBytes);
                const int y = t.kv_head * p.G, z = f.seq_start + t.q_start;
                for (int x = 0; x < (has_b ? 2 : 1); ++x) {
                    const uint32_t qdst = base + kQOff + x * kTileBytes;
                    xy::tma_load_3d(qdst, &qmap, 0, y, z + x * qt_tokens, bar(B_QFULL));
                    xy::tma_load_3d(qdst + kHalfBytes, &qmap, 64, y, z + x * qt_tokens, bar(B_QFULL));
                }
            }
            ++qk;
            const int32_t *bt_row = p.bt + (int64_t)t.seq * p.MB;
            int win0 = t.kv_start / p.bs;
            int pg_win = DYN ? tc.win : pref_valid ? pref_win : load_win(bt_row, win0);
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
                if (!dep_ready && kv0 + nkeys > f.L - f.qn) {  // the tile holds new tokens' rows
                    xy::grid_dep_wait();
                    dep_ready = true;
                }
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
                if (t.kv_end - (kv0 + nkeys) <= kClaimAheadKeys) tc.release_claim();
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
        tc.release_claim();  // (a loop left early may still hold one)
        if (!ok || tc.failed) {
            if (lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
            *abort_flag = 1;
        } else if (p.trace && lane == 0) {
            p.trace[4 * blockIdx.x + 2] = n_run;
            p.trace[4 * blockIdx.x + 3] = work;
        }
        // every issued copy must land before the CTA may exit
        for (int k = c - 1; k >= 0 && k >= c - kSlots; --k)
            xy::mbar_wait(bar(B_FULL0 + k % kSlots), (k / kSlots) & 1);
        if (qk > 0) xy::mbar_wait(bar(B_QFULL), (qk - 1) & 1);
        xy::dec::drain<DecRing>(dsm, dctr, 0, 2);
    } else if (warp == kMmaWarp) {
        // ---------------------------------- MMA issuer ----------------------------------
        if (lane == 0) {
            const uint32_t id_s = xy::idesc_bf16(128, 128, 0, 0);   // Q (K-major) x K tile (K-major)
            const uint32_t id_o = xy::idesc_bf16(128, 128, 0, 1);   // P (TMEM) x V tile (MN-major)
            // Descriptors are built once; a k-step or buffer only adds a constant to the 14-bit
            // address field (addresses stay below 256 KB), keeping the single issuing thread cheap.
            const uint64_t q_desc0 = xy::smem_desc_sw128(base + kQOff, 16, 1024);
            const uint64_t k_desc0 = xy::smem_desc_sw128(base + kSlotOff, 16, 1024);
            const uint64_t v_desc0 = xy::smem_desc_sw128(base + kSlotOff, kHalfBytes, 1024);
            constexpr uint32_t kTileDesc = kTileBytes >> 4;
            int c = 0, qk = 0;
            int ns[2] = {0, 0};   // S_X issued so far (= PV_X issued, = tiles of group X)
            int nt[2] = {0, 0};   // tasks in which query tile X was active (= its O_X epilogues)
            bool ok = true, issued = false;
            auto wait = [&](uint32_t b, uint32_t parity) -> bool {
                if (!xy::mbar_wait(b, parity, abort_flag)) {
                    ok = false;
                    return false;
                }
                return true;
            };
            auto issue_s = [&](int x, int j) {
                const int s = (c + 2 * j) % kSlots;
                const uint64_t qd = q_desc0 + (uint64_t)(x * kTileDesc);
                const uint64_t kd = k_desc0 + (uint64_t)(s * kTileDesc);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t koff = (uint64_t)(((k >> 2) * kHalfBytes + (k & 3) * 32) >> 4);
                    xy::umma_ss(tbase + x * 128, qd + koff, kd + koff, id_s, k > 0 ? 1u : 0u);
                }
                xy::umma_commit(bar(B_SFULL0 + x));
                ++ns[x];
            };
            auto issue_pv = [&](int x, int j) {
                const int s = (c + 2 * j + 1) % kSlots;
                const uint64_t vd = v_desc0 + (uint64_t)(s * kTileDesc);
                const uint32_t pa = tbase + x * 128, od = tbase + kTmemO + x * 128;
                xy::umma_ts(od, pa, vd, id_o, j > 0 ? 1u : 0u);
#pragma unroll
                for (int k = 1; k < 8; ++k) xy::umma_ts(od, pa + k * 8, vd + (uint64_t)(k * (2048 >> 4)), id_o, 1u);
                xy::umma_commit(bar(B_OBAR0 + x));
            };
            TaskCursor tc;
            tc.attach(q, true, false);
            tc.begin(p);
            while (tc.have && ok) {
                tc.load_next_record(p);
                if (!mine(tc.cur, p) || !tile_ok(tc.cur, p)) {
                    tc.advance(p);
                    continue;
                }
                const xy_task t = tc.cur.t;
                const int n = (t.kv_end - t.kv_start + kTileKeys - 1) / kTileKeys;
                const int nx = t.q_rows * p.G > 128 ? 2 : 1;
                if (!wait(bar(B_QFULL), qk & 1)) break;
                xy::tc_fence_after();
                tc.prefetch_next(p);
                issued = true;
                for (int j = 0; j <= n && ok; ++j) {
                    if (j >= 1) {  // V_{j-1} has landed
                        const int cv = c + 2 * (j - 1) + 1;
                        if (!wait(bar(B_FULL0 + cv % kSlots), (cv / kSlots) & 1)) break;
                    }
                    // K_j is waited for only before the first S that reads it, so that a K tile
                    // still in flight does not hold back tile A's PV of the previous tile
                    bool k_here = j >= n;
                    for (int x = 0; x < nx && ok; ++x) {
                        if (j >= 1) {
                            // P_X(j-1) written (and O_X corrected) by its softmax group; for the
                            // first PV of the task the previous task's epilogue must have read O_X
                            if (!wait(bar(B_PFULL0 + x), (ns[x] - 1) & 1)) break;
                            if (j == 1 && nt[x] >= 1 && !wait(bar(B_OFREE0 + x), (nt[x] - 1) & 1)) break;
                            xy::tc_fence_after();
                            issue_pv(x, j - 1);
                        }
                        if (j < n) {
                            if (!k_here) {
                                const int ck = c + 2 * j;
                                if (!wait(bar(B_FULL0 + ck % kSlots), (ck / kSlots) & 1)) break;
                                k_here = true;
                            }
                            issue_s(x, j);
                        }
                    }
                    if (!ok) break;
                    if (j >= 1) xy::umma_commit(bar(B_EMPTY0 + (c + 2 * (j - 1) + 1) % kSlots));  // V_{j-1}
                    if (j < n) xy::umma_commit(bar(B_EMPTY0 + (c + 2 * j) % kSlots));             // K_j
                    if (j == n - 1) xy::umma_commit(bar(B_QEMPTY));  // the last S of the task
                }
                c += 2 * n;
                ++qk;
                for (int x = 0; x < nx; ++x) ++nt[x];
                tc.advance(p);
            }
            if (!ok || tc.failed) {
                xy::set_err(p.err, XY_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            if (issued) {  // everything issued has completed before TMEM is freed
                xy::umma_commit(bar(B_DONE));
                xy::mbar_wait(bar(B_DONE), 0);
            }
        }
        __syncwarp();
    } else if (warp == kDecProducerWarp) {
        // ------------------------- second decode-ring producer -------------------------
        // Issuing a decode stage (block-table window, page boxes, barrier bookkeeping) takes a
        // warp about as long as the math warps need to consume one; with the producer warp on the
        // even stages and this warp on the odd ones the ring stays ahead of the math.
        int dctr = 0, nd = 0, pref_win = -1;
        bool ok = true, pref_valid = false, after_tile = false, dep_ready = false;
        TaskCursor tc;
        tc.attach(q, false, false);
        tc.begin(p);
        while (tc.have && ok) {
            tc.load_next_record(p);
            if (mine(tc.cur, p)) {
                after_tile = after_tile || tile_ok(tc.cur, p);
                pref_valid = false;
                tc.advance(p);
                continue;
            }
            if (!xy::dec::task_ok<DecRing>(tc.cur, p)) {
                pref_valid = false;
                tc.advance(p);
                continue;
            }
            if (after_tile) {
                // the decode ring overlays the tile buffers: wait until the producer warp has seen
                // the tile work before this task stop reading shared memory
                bool w = true;
                if (lane == 0) {
                    const uint64_t t0 = xy::global_timer_ns();
                    while (*dec_go < nd + 1) {
                        if (*abort_flag || xy::global_timer_ns() - t0 > xy::kWaitTimeoutNs) {
                            w = false;
                            break;
                        }
                    }
                }
                if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) {
                    ok = false;
                    break;
                }
                __threadfence_block();
                after_tile = false;
            }
            ++nd;
            const TaskInfo f = tc.cur;
            const bool have_first = DYN || pref_valid;
            const int first_win = DYN ? tc.win : pref_win;
            pref_valid = false;
            ok = xy::dec::produce_task<HD, DecRing>(
                p, f, &kmap_d, &vmap_d, nullptr, nullptr, dsm, dctr, lane, first_win, have_first, dep_ready,
                [&]() {
                    tc.prefetch_next(p);
                    if (tc.have_next) {
                        const xy_task &tn = tc.nxt.t;
                        pref_valid = tn.seq >= 0 && tn.seq < p.S && tn.kv_start >= 0;
                        if (pref_valid) pref_win = xy::load_window(p, tn.seq, tn.kv_start / p.bs, lane);
                    }
                },
                1, 2);
            tc.advance(p);
        }
        if (!ok || tc.failed) {
            if (lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
            *abort_flag = 1;
        }
        // every stage this warp issued must land before the CTA may exit
        xy::dec::drain<DecRing>(dsm, dctr, 1, 2);
    } else if (warp == kSchedWarp) {
        // ---------------------------- scheduler (dynamic deal) ----------------------------
        if constexpr (DYN) {
            int r = 1;
            for (int e = 0; r == 1; ++e) r = dq.publish(e, p, p.dyn, lane);
            dq.finish(p.dyn, lane);
            if (r < 0) {
                if (lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
                *abort_flag = 1;
            }
        }
    }
    } else {
        xy::setmaxnreg_inc<kRegsSoftmax>();
        // ---------------------------------- softmax ----------------------------------
        const int x = warp >> 2;                            // query tile of this group
        const int trow = (warp & 3) * 32 + lane;            // row within the tile = TMEM lane
        const int row = x * 128 + trow;                     // row within the task
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_addr = tbase + lane_off + x * 128;
        const uint32_t o_addr = tbase + lane_off + kTmemO + x * 128;
        int c = 0, qk = 0, ns = 0;   // ns: tiles this group has processed (= its S and PV count)
        int dctr = 0, diter = 0;     // decode path (warps 0..3): stages consumed, tasks run
        bool ok = true;
        TaskCursor tc;
        // the group passes named barrier 1 + x together, so its four warps vote on each queue read
        tc.attach(q, false, false, reinterpret_cast<volatile int *>(gbase + kQueueVoteOff) + 8 * x, 1 + x, 4,
                  warp & 3);
        tc.begin(p);
        while (tc.have) {
            tc.load_next_record(p);
            if (!mine(tc.cur, p)) {
                // a decode-path task: warps 0..3 are its math warps, warps 4..7 sit it out
                if (warp < 4 && xy::dec::task_ok<DecRing>(tc.cur, p)) {
                    const TaskInfo f = tc.cur;
                    if (!xy::dec::consume_task<HD, DecRing>(p, f, dsm, dctr, diter, warp, lane,
                                                            [&]() { tc.prefetch_next(p); })) {
                        *abort_flag = 1;
                        if (warp == 0 && lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
                        break;
                    }
                    __syncwarp();
                    if (lane == 0) xy::mbar_arrive(dec_done + 8 * ((diter - 1) & 1));
                }
                tc.advance(p);
                continue;
            }
            if (!tile_ok(tc.cur, p)) {
                tc.advance(p);
                continue;
            }
            const TaskInfo f = tc.cur;
            const xy_task t = f.t;
            const int R = t.q_rows * p.G;
            const int n = (t.kv_end - t.kv_start + kTileKeys - 1) / kTileKeys;
            // tile B exists only for tasks with more than 128 rows; a warp whose 32 rows are all
            // padding does no softmax work (its P and O rows are never stored; rows of an MMA are
            // independent, so whatever its TMEM lanes hold cannot reach a real row)
            const bool active = x == 0 || R > 128;
            const bool rows_on = active && (row - lane) < R;
            const bool valid = row < R;
            const int lim = valid ? min(t.kv_end, p.causal ? f.L - f.qn + t.q_start + row / p.G + 1 : f.L) : t.kv_end;
            float m = -INFINITY, l = 0.f;
            if (active) {
                for (int j = 0; j < n; ++j) {
                    // a failed wait (timeout or abort) is recorded, not acted on: the group keeps
                    // executing the same steps and the decision to stop is voted below
                    ok = warp_all(xy::mbar_wait(bar(B_SFULL0 + x), ns & 1, abort_flag)) && ok;
                    xy::tc_fence_after();
                    if (j == 0) tc.prefetch_next(p);
                    const int kt0 = t.kv_start + j * kTileKeys;
                    if (rows_on) {
                    // a warp whose rows all see the whole tile skips the per-key mask
                        const bool full = __all_sync(0xffffffffu, kt0 + kTileKeys <= lim);
                        // The tile's softmax is compiled twice -- without any masking code for
                        // tiles every row of the warp sees whole, and with the per-key mask -- so
                        // the common case carries no selects (the warp picks one per tile).
                        auto tile_softmax = [&](auto full_c) {
                            constexpr bool kFull = decltype(full_c)::value;
                            // pass 1: masked row max; 32-column TMEM loads, the next one in flight while
                            // the current one is reduced
                            uint32_t ca[32], cb[32];
                            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                            // in a masked tile a 32-key chunk is still whole or empty for all rows of
                            // the warp unless it holds one of their limits (warp-uniform tests)
                            auto chunk_whole = [&](int c0) { return kFull || __all_sync(0xffffffffu, kt0 + c0 + 32 <= lim); };
                            auto chunk_empty = [&](int c0) { return !kFull && __all_sync(0xffffffffu, kt0 + c0 >= lim); };
                            auto max_chunk = [&](const uint32_t (&r)[32], int c0) {
                                if (chunk_whole(c0)) {
        #pragma unroll
                                    for (int i = 0; i < 32; i += 8) {
                                        m4[0] = xy::max3(m4[0], __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                                        m4[1] = xy::max3(m4[1], __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                                        m4[2] = xy::max3(m4[2], __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
                                        m4[3] = xy::max3(m4[3], __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
                                    }
                                } else if (!chunk_empty(c0)) {
        #pragma unroll
                                    for (int i = 0; i < 32; ++i)
                                        m4[i & 3] = fmaxf(m4[i & 3], kt0 + c0 + i < lim ? __uint_as_float(r[i]) : -INFINITY);
                                }
                            };
                            float mx;
                            if constexpr (kFull) {
                                // every key is visible: the TMEM load itself returns each chunk's
                                // maximum (tcgen05.ld.red), two chunks in flight per round trip
                                float mxa, mxb;
                                xy::tmem_ld32_max_nowait(s_addr, ca, mxa);
                                xy::tmem_ld32_max_nowait(s_addr + 32, cb, mxb);
                                xy::tmem_wait_ld_max(ca, mxa);
                                xy::tmem_wait_ld_max(cb, mxb);
                                const float mx01 = fmaxf(mxa, mxb);
                                xy::tmem_ld32_max_nowait(s_addr + 64, ca, mxa);
                                xy::tmem_ld32_max_nowait(s_addr + 96, cb, mxb);
                                xy::tmem_wait_ld_max(ca, mxa);
                                xy::tmem_wait_ld_max(cb, mxb);
                                mx = fmaxf(mx01, fmaxf(mxa, mxb));
                                xy::tmem_ld32_nowait(s_addr, ca);  // pass 2's first chunk
                            } else {
                                xy::tmem_ld32_nowait(s_addr, ca);
                                xy::tmem_wait_ld(ca);
                                xy::tmem_ld32_nowait(s_addr + 32, cb);
                                max_chunk(ca, 0);
                                xy::tmem_wait_ld(cb);
                                xy::tmem_ld32_nowait(s_addr + 64, ca);
                                max_chunk(cb, 32);
                                xy::tmem_wait_ld(ca);
                                xy::tmem_ld32_nowait(s_addr + 96, cb);
                                max_chunk(ca, 64);
                                xy::tmem_wait_ld(cb);
                                xy::tmem_ld32_nowait(s_addr, ca);  // pass 2's first chunk
                                max_chunk(cb, 96);
                                mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                            }
                            const float m_new = fmaxf(m, mx * p.scale_log2);  // the scale is positive
                            const bool rescale = __any_sync(0xffffffffu, m_new > m + kRescaleThreshold);
                            xy::tmem_wait_ld(ca);
                            if (rescale) {
                                const float alpha = m_new == -INFINITY ? 1.f : ex2(m - m_new);
                                m = m_new;
                                l *= alpha;
                                if (j > 0) {  // O_X has PV_X(0..j-1); rescale once the last of them is done
                                    ok = warp_all(xy::mbar_wait(bar(B_OBAR0 + x), (ns - 1) & 1, abort_flag)) && ok;
                                    xy::tc_fence_after();
        #pragma unroll 1
                                    for (int h = 0; h < 4; ++h) {
                                        uint32_t orow[32];
                                        xy::tmem_ld32(o_addr + h * 32, orow);
        #pragma unroll
                                        for (int i = 0; i < 32; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * alpha);
                                        xy::tmem_st32(o_addr + h * 32, orow);
                                    }
                                }
                            }
                            // pass 2: p = 2^(s * scale_log2 - m) for 32 columns at a time, packed to bf16
                            // pairs and written over S columns that pass 2 has already read
                            const float neg_mu = m == -INFINITY ? 0.f : -m;
                            const uint64_t sc2 = xy::f2_pack(p.scale_log2, p.scale_log2), nm2 = xy::f2_pack(neg_mu, neg_mu);
                            uint64_t acc2[2] = {0ull, 0ull};
                            auto exp_loop = [&](const uint32_t (&r)[32], int c0, uint32_t (&pk)[16], auto masked_c) {
                                constexpr bool kMasked = decltype(masked_c)::value;
        #pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    float s0 = __uint_as_float(r[2 * i]), s1 = __uint_as_float(r[2 * i + 1]);
                                    if constexpr (kMasked) {
                                        s0 = kt0 + c0 + 2 * i < lim ? s0 : -INFINITY;
                                        s1 = kt0 + c0 + 2 * i + 1 < lim ? s1 : -INFINITY;
                                    }
                                    float e0, e1;
                                    xy::f2_unpack(xy::f2_fma(xy::f2_pack(s0, s1), sc2, nm2), e0, e1);
                                    const float p0 = ex2(e0), p1 = ex2(e1);
                                    acc2[i & 1] = xy::f2_add(acc2[i & 1], xy::f2_pack(p0, p1));
                                    pk[i] = xy::pack_bf16x2(p0, p1);
                                }
                            };
                            auto exp_chunk = [&](const uint32_t (&r)[32], int c0, int chunk) {
                                uint32_t pk[16];
                                if (chunk_whole(c0)) {
                                    exp_loop(r, c0, pk, std::false_type{});
                                } else if (chunk_empty(c0)) {
        #pragma unroll
                                    for (int i = 0; i < 16; ++i) pk[i] = 0u;
                                } else {
                                    exp_loop(r, c0, pk, std::true_type{});
                                }
                                xy::tmem_st16(s_addr + 16 * chunk, pk);
                            };
                            xy::tmem_ld32_nowait(s_addr + 32, cb);
                            exp_chunk(ca, 0, 0);
                            xy::tmem_wait_ld(cb);
                            xy::tmem_ld32_nowait(s_addr + 64, ca);
                            exp_chunk(cb, 32, 1);
                            xy::tmem_wait_ld(ca);
                            xy::tmem_ld32_nowait(s_addr + 96, cb);
                            exp_chunk(ca, 64, 2);
                            xy::tmem_wait_ld(cb);
                            exp_chunk(cb, 96, 3);
                            float ls4[4];
                            xy::f2_unpack(acc2[0], ls4[0], ls4[1]);
                            xy::f2_unpack(acc2[1], ls4[2], ls4[3]);
                            l += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
                        };
                        // A tile that cuts through some row's visible keys (the causal diagonal, the
                        // end of the context) runs once per task: its code is kept compact (one 32-key
                        // chunk per loop step, the mask as the row's count of visible keys in the chunk)
                        // so that it stays in the instruction cache beside the steady loop.
                        // Each 32-key chunk is classified for the whole warp: no row sees any of its
                        // keys (no load; P = 0), every row sees all of them (no per-key mask), or the
                        // chunk holds some row's limit (masked).  On the causal diagonal most chunks
                        // of a warp's eight tokens are whole or empty.
                        auto masked_softmax = [&]() {
                            float mx = -INFINITY;
#pragma unroll 1
                            for (int ci = 0; ci < 4; ++ci) {
                                const int nv = lim - (kt0 + 32 * ci);
                                if (__all_sync(0xffffffffu, nv <= 0)) continue;
                                uint32_t r[32];
                                xy::tmem_ld32(s_addr + 32 * ci, r);
                                if (__all_sync(0xffffffffu, nv >= 32)) {
#pragma unroll
                                    for (int i = 0; i < 32; i += 2) mx = xy::max3(mx, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                                } else {
#pragma unroll
                                    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, i < nv ? __uint_as_float(r[i]) : -INFINITY);
                                }
                            }
                            const float m_new = fmaxf(m, mx * p.scale_log2);  // the scale is positive
                            if (__any_sync(0xffffffffu, m_new > m + kRescaleThreshold)) {
                                const float alpha = m_new == -INFINITY ? 1.f : ex2(m - m_new);
                                m = m_new;
                                l *= alpha;
                                if (j > 0) {  // O_X has PV_X(0..j-1); rescale once the last of them is done
                                    ok = warp_all(xy::mbar_wait(bar(B_OBAR0 + x), (ns - 1) & 1, abort_flag)) && ok;
                                    xy::tc_fence_after();
#pragma unroll 1
                                    for (int h = 0; h < 4; ++h) {
                                        uint32_t orow[32];
                                        xy::tmem_ld32(o_addr + h * 32, orow);
#pragma unroll
                                        for (int i = 0; i < 32; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * alpha);
                                        xy::tmem_st32(o_addr + h * 32, orow);
                                    }
                                }
                            }
                            const float neg_mu = m == -INFINITY ? 0.f : -m;
                            float ls[2] = {0.f, 0.f};
#pragma unroll 1
                            for (int ci = 0; ci < 4; ++ci) {
                                uint32_t r[32], pk[16];
                                const int nv = lim - (kt0 + 32 * ci);
                                if (__all_sync(0xffffffffu, nv <= 0)) {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) pk[i] = 0u;
                                } else {
                                    xy::tmem_ld32(s_addr + 32 * ci, r);
                                    if (__all_sync(0xffffffffu, nv >= 32)) {
#pragma unroll
                                        for (int i = 0; i < 16; ++i) {
                                            const float p0 = ex2(fmaf(__uint_as_float(r[2 * i]), p.scale_log2, neg_mu));
                                            const float p1 = ex2(fmaf(__uint_as_float(r[2 * i + 1]), p.scale_log2, neg_mu));
                                            ls[i & 1] += p0 + p1;
                                            pk[i] = xy::pack_bf16x2(p0, p1);
                                        }
                                    } else {
#pragma unroll
                                        for (int i = 0; i < 16; ++i) {
                                            const float e0 = fmaf(__uint_as_float(r[2 * i]), p.scale_log2, neg_mu);
                                            const float e1 = fmaf(__uint_as_float(r[2 * i + 1]), p.scale_log2, neg_mu);
                                            const float p0 = 2 * i < nv ? ex2(e0) : 0.f, p1 = 2 * i + 1 < nv ? ex2(e1) : 0.f;
                                            ls[i & 1] += p0 + p1;
                                            pk[i] = xy::pack_bf16x2(p0, p1);
                                        }
                                    }
                                }
                                xy::tmem_st16(s_addr + 16 * ci, pk);  // over S columns already read
                            }
                            l += ls[0] + ls[1];
                        };
                        if (full)
                            tile_softmax(std::true_type{});
                        else
                            masked_softmax();
                    }
                    if (x == 0 && kt0 + kTileKeys > t.kv_end) {
                        // keys at or past kv_end: unused page slots or stale data; their P is 0 and
                        // their V rows are zeroed (group A, before both tiles' PV of this K/V tile)
                        // so that 0 * NaN cannot occur.  Wait for the V copy to land first.
                        const int cv = c + 2 * j + 1, s = cv % kSlots;
                        ok = warp_all(xy::mbar_wait(bar(B_FULL0 + s), (cv / kSlots) & 1, abort_flag)) && ok;
                        if (kt0 + trow >= t.kv_end) {
                            uint4 *v0 = reinterpret_cast<uint4 *>(gbase + kSlotOff + s * kTileBytes + trow * 128);
                            uint4 *v1 = reinterpret_cast<uint4 *>(gbase + kSlotOff + s * kTileBytes + kHalfBytes + trow * 128);
                            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                v0[i] = z;
                                v1[i] = z;
                            }
                        }
                        xy::fence_async_smem();
                    }
                    xy::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) xy::mbar_arrive(bar(B_PFULL0 + x));
                    ++ns;
                }
                if (rows_on) {
                    ok = warp_all(xy::mbar_wait(bar(B_OBAR0 + x), (ns - 1) & 1, abort_flag)) && ok;
                    xy::tc_fence_after();
                }
            }
            // the group's vote on whether to go on
            if (lane == 0) vote[warp] = ok ? 0 : 1;
            xy::named_bar_sync(1 + x, 128);
            int bad = 0;
#pragma unroll
            for (int w = 0; w < 4; ++w) bad |= vote[x * 4 + w];
            // A whole query tile (all 128 rows valid) with bf16 output: the group stages its normalized
            // rows in shared memory (one 64-column half at a time, the TMA's 128-byte swizzle) and one
            // thread writes each half with a TMA store, which moves whole lines instead of 32-byte
            // pieces of 128 different rows.  Uniform in the group (it depends on the task and x).
            const bool tma_out = active && t.num_splits == 1 && R - x * 128 >= 128;
            if (tma_out) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const bool leader = (warp & 3) == 0 && lane == 0;
                const uint32_t stage = base + kStageOff + x * kHalfBytes;
                uint8_t *stage_row = gbase + kStageOff + x * kHalfBytes + trow * 128;
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    if (leader) xy::bulk_wait_read();   // the group's previous store has read the staging
                    xy::named_bar_sync(1 + x, 128);
                    uint32_t ra[32], rb[32];
                    xy::tmem_ld32_nowait(o_addr + hh * 64, ra);
                    xy::tmem_ld32_nowait(o_addr + hh * 64 + 32, rb);
                    xy::tmem_wait_ld(ra);
                    xy::tmem_wait_ld(rb);
                    if (!bad) {
                        auto stage_chunks = [&](const uint32_t (&r)[32], int c0) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {   // 16-byte chunk c0 + c: 8 columns
                                uint4 v;
                                v.x = xy::pack_bf16x2(__uint_as_float(r[8 * c]) * inv, __uint_as_float(r[8 * c + 1]) * inv);
                                v.y = xy::pack_bf16x2(__uint_as_float(r[8 * c + 2]) * inv, __uint_as_float(r[8 * c + 3]) * inv);
                                v.z = xy::pack_bf16x2(__uint_as_float(r[8 * c + 4]) * inv, __uint_as_float(r[8 * c + 5]) * inv);
                                v.w = xy::pack_bf16x2(__uint_as_float(r[8 * c + 6]) * inv, __uint_as_float(r[8 * c + 7]) * inv);
                                *reinterpret_cast<uint4 *>(stage_row + (((c0 + c) ^ (trow & 7)) << 4)) = v;
                            }
                        };
                        stage_chunks(ra, 0);
                        stage_chunks(rb, 4);
                    }
                    xy::fence_async_smem();
                    xy::named_bar_sync(1 + x, 128);
                    if (leader && !bad) {
                        xy::tma_store_3d(&omap, stage, hh * 64, t.kv_head * p.G, f.seq_start + t.q_start + x * qt_tokens);
                        xy::bulk_commit();
                    }
                }
            } else if (rows_on) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                // each thread writes its own row, 32 O columns per loop step: 32-byte stores (one full
                // sector each) when the buffers allow.  The epilogue runs once per task, so its code
                // is kept compact (one step's code, not four unrolled copies).
                const bool v8 = ((reinterpret_cast<uintptr_t>(p.out) | reinterpret_cast<uintptr_t>(p.ws_o)) & 31) == 0;
                const bool st_ok = valid && !bad, to_out = t.num_splits == 1;
                __nv_bfloat16 *dst_o = p.out;
                float *dst_w = p.ws_o;
                if (to_out) {
                    const int64_t tok = f.seq_start + t.q_start + row / p.G;
                    dst_o += (tok * p.Hq + t.kv_head * p.G + row % p.G) * HD;
                } else {
                    dst_w += ((int64_t)t.ws_row + row) * HD;
                }
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t r[32];
                    xy::tmem_ld32(o_addr + 32 * cc, r);
                    if (!st_ok) continue;
                    if (to_out) {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            w[i] = xy::pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
                        __nv_bfloat16 *dst = dst_o + cc * 32;
                        if (v8) {
                            xy::st_global_v8(dst, reinterpret_cast<const uint32_t(&)[8]>(w[0]));
                            xy::st_global_v8(dst + 16, reinterpret_cast<const uint32_t(&)[8]>(w[8]));
                        } else {
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                reinterpret_cast<uint4 *>(dst)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * inv);
                        float *dst = dst_w + cc * 32;
                        if (v8) {
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                xy::st_global_v8(dst + 8 * v, reinterpret_cast<const uint32_t(&)[8]>(r[8 * v]));
                        } else {
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                reinterpret_cast<uint4 *>(dst)[v] = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
                        }
                    }
                }
                if (valid && !bad && t.num_splits > 1) p.ws_lse[(int64_t)t.ws_row + row] = l > 0.f ? m + __log2f(l) : -INFINITY;
            }
            if (active) {
                xy::tc_fence_before();
                __syncwarp();
                if (lane == 0) xy::mbar_arrive(bar(B_OFREE0 + x));
            }
            c += 2 * n;
            ++qk;
            if (bad) {
                *abort_flag = 1;
                if (warp == 0 && lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
                break;
            }
            tc.advance(p);
        }
        if (tc.failed) {
            *abort_flag = 1;
            if (lane == 0) xy::set_err(p.err, XY_DEV_TIMEOUT);
        }
        // the group's output stores have completed before the CTA leaves
        if ((warp & 3) == 0 && lane == 0) xy::bulk_wait_all();
    }

    xy::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        xy::tc_fence_after();
        xy::tmem_dealloc(tbase, kTmemCols);
    }
    if (p.trace && threadIdx.x == 0 && !*abort_flag) p.trace[4 * blockIdx.x + 1] = xy::global_timer_ns();
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

xy_status launch_meta_attention(const AttnParams &p, const void *k_pages, const void *v_pages, int num_pages,
                                int block_size, int num_ctas, const CUtensorMap &kmap_d, const CUtensorMap &vmap_d,
                                cudaStream_t st) {
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
    // the output in the same layout and boxes, for the epilogue's TMA stores of whole query tiles
    CUtensorMap om;
    if (fn(&om, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.out, qdims, qstr, qbox, e3, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return XY_ERR_CUDA;
    static PerDeviceOnce configured[2];  // per instantiation and device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail(cudaGetLastError(), "cudaGetDevice");
    const int dyn = p.dyn ? 1 : 0;
    if (!configured[dyn].done(dev)) {
        const cudaError_t e = cudaFuncSetAttribute(dyn ? meta_attention_kernel<true> : meta_attention_kernel<false>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return cuda_fail(e, "meta_attention_kernel smem attribute");
        // the warpgroups' register budgets assume the kernel is launched with kLaunchRegs per thread
        cudaFuncAttributes fa;
        const cudaError_t ea =
            cudaFuncGetAttributes(&fa, dyn ? meta_attention_kernel<true> : meta_attention_kernel<false>);
        if (ea != cudaSuccess) return cuda_fail(ea, "meta_attention_kernel attributes");
        if (fa.numRegs != kLaunchRegs) {
            set_last_error("meta_attention_kernel", "unexpected register count at launch");
            return XY_ERR_UNSUPPORTED;
        }
        configured[dyn].mark(dev);
    }
    const cudaError_t e =
        dyn ? xy::launch_dependent(meta_attention_kernel<true>, dim3(num_ctas), dim3(kThreads), kSmemBytes, st, km, vm,
                                   qm, om, kmap_d, vmap_d, p)
            : xy::launch_dependent(meta_attention_kernel<false>, dim3(num_ctas), dim3(kThreads), kSmemBytes, st, km,
                                   vm, qm, om, kmap_d, vmap_d, p);
    return e == cudaSuccess ? XY_OK : cuda_fail(e, "meta_attention_kernel launch");
}

}  // namespace xy
