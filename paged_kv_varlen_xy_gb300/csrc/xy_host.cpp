// Host side of libxy: status strings, the block-table allocator (a1) and the task-table
// builder (a4).  Pure host code, no CUDA calls, so it runs and is tested without a GPU.
//
// Sources: "XY-Serve 深度实战" (chenxutan.com/d/5031) §2.2 components 1-2, §4.2, §4.4;
// cann-recipes-infer Paged KV Cache / Packed Sequence notes (dpshk.com/news/5336026) §2.2, §3.2.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <limits>
#include <utility>
#include <vector>

#include "xy.h"

extern "C" const char *xy_status_string(int status) {
    switch (status) {
        case XY_OK: return "ok";
        case XY_ERR_INVALID_ARG: return "invalid argument";
        case XY_ERR_CU_SEQLENS: return "cu_seqlens_q must start at 0 and increase strictly";
        case XY_ERR_PAGE_OOB: return "block-table entry outside [0, num_pages)";
        case XY_ERR_CONTEXT_LT_QLEN: return "context_lens[i] < q_len of sequence i";
        case XY_ERR_UNSUPPORTED: return "shape not supported by the kernels";
        case XY_ERR_WORKSPACE: return "workspace missing or too small";
        case XY_ERR_CUDA: return "CUDA call failed";
        case XY_ERR_TIMEOUT: return "timed out";
        case XY_ERR_OUT_OF_PAGES: return "KV page pool exhausted";
        case XY_ERR_CAPACITY: return "output array too small";
        default: return "unknown status";
    }
}

extern "C" int xy_version(void) { return 100; }

// Last CUDA failure seen on this host thread (written by the device-call entry points).
namespace xy {
thread_local char g_last_error[256] = "";
void set_last_error(const char *what, const char *msg) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, msg);
}
}  // namespace xy

extern "C" const char *xy_last_error_string(void) { return xy::g_last_error; }

static bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// a1: FIFO page allocation in batch order.  Sequence i takes ceil(L_i / bs) pages from the
// front of the free list; unused columns are -1 (the page table of §3.1 of the cann notes).
extern "C" xy_status xy_build_block_table(const int32_t *context_lens, int num_seqs, int block_size,
                                          const int32_t *free_list, int num_free, int max_blocks,
                                          int32_t *block_table, int *pages_used) {
    if (num_seqs < 0 || num_free < 0 || max_blocks < 1 || !is_pow2(block_size) || block_size < 16)
        return XY_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!context_lens || !block_table)) return XY_ERR_INVALID_ARG;
    if (num_free > 0 && !free_list) return XY_ERR_INVALID_ARG;
    int64_t pos = 0;
    for (int i = 0; i < num_seqs; ++i) {
        const int64_t L = context_lens[i];
        if (L < 1) return XY_ERR_INVALID_ARG;
        const int64_t n = (L + block_size - 1) / block_size;
        if (n > max_blocks) return XY_ERR_CAPACITY;
        if (pos + n > num_free) return XY_ERR_OUT_OF_PAGES;
        int32_t *row = block_table + (int64_t)i * max_blocks;
        std::memcpy(row, free_list + pos, sizeof(int32_t) * (size_t)n);
        std::fill(row + n, row + max_blocks, -1);
        pos += n;
    }
    if (pages_used) *pages_used = (int)pos;
    return XY_OK;
}

namespace {
struct Rec {
    xy_task t;
    int64_t load;
};
// Scratch of the task-table builder, kept per host thread (a batch's tables are rebuilt every
// step; this keeps the builder free of allocations once warm).
struct BuildScratch {
    std::vector<Rec> recs, sorted;
    std::vector<xy_merge> mrg;
    std::vector<uint32_t> order, order2;
    std::vector<uint64_t> keys, keys2;
    std::vector<uint32_t> hist;
    std::vector<int64_t> tload;
    std::vector<int> tree, cta_of, pos_of, count;
    std::vector<int64_t> gstart;       // dynamic deal: per (sequence, KV head) group
    std::vector<uint32_t> glist;
};
thread_local BuildScratch g_scratch;

// recs sorted stably by load, largest first: a counting sort of the complemented loads (loads are
// below 2^55) when they span few distinct steps, else an LSD radix sort with 11-bit digits,
// digits that are equal for every key skipped.  Each pass moves
// (key, index) pairs, so it reads them in order; the records move once, at the end.
void sort_by_load_desc(std::vector<Rec> &recs, BuildScratch &sc) {
    const size_t n = recs.size();
    std::vector<uint32_t> &a = sc.order, &b = sc.order2;
    std::vector<uint64_t> &ka = sc.keys, &kb = sc.keys2;
    a.resize(n);
    b.resize(n);
    ka.resize(n);
    kb.resize(n);
    const uint64_t kMask = (uint64_t(1) << 55) - 1;
    uint64_t all_or = 0, all_and = ~uint64_t(0);
    for (size_t i = 0; i < n; ++i) {
        a[i] = (uint32_t)i;
        ka[i] = kMask - (uint64_t)recs[i].load;
        all_or |= ka[i];
        all_and &= ka[i];
    }
    const uint64_t varies = all_or ^ all_and;
    if (varies == 0) return;  // every load equal: the order stays
    // Loads are multiples of a power of two (the charged rows) and usually span a narrow range:
    // then one counting pass over (key - min) >> tz, at most 2^16 buckets, sorts them.
    const int tz = __builtin_ctzll(varies);
    uint64_t kmin = ~uint64_t(0), kmax = 0;
    for (size_t i = 0; i < n; ++i) {
        kmin = std::min(kmin, ka[i]);
        kmax = std::max(kmax, ka[i]);
    }
    const uint64_t span = (kmax - kmin) >> tz;
    if (span < (uint64_t(1) << 16)) {
        sc.hist.assign((size_t)span + 1, 0u);
        for (size_t i = 0; i < n; ++i) ++sc.hist[(ka[i] - kmin) >> tz];
        uint32_t sum = 0;
        for (uint32_t &h : sc.hist) {
            const uint32_t c = h;
            h = sum;
            sum += c;
        }
        std::vector<Rec> &sorted = sc.sorted;
        sorted.resize(n);
        for (size_t i = 0; i < n; ++i) sorted[sc.hist[(ka[i] - kmin) >> tz]++] = recs[i];
        recs.swap(sorted);
        return;
    }
    sc.hist.resize(2048);
    for (int shift = 0; shift < 55; shift += 11) {
        if (((varies >> shift) & 2047u) == 0) continue;
        std::fill(sc.hist.begin(), sc.hist.end(), 0u);
        for (size_t i = 0; i < n; ++i) ++sc.hist[(ka[i] >> shift) & 2047u];
        uint32_t sum = 0;
        for (uint32_t &h : sc.hist) {
            const uint32_t c = h;
            h = sum;
            sum += c;
        }
        for (size_t i = 0; i < n; ++i) {
            const uint32_t d = sc.hist[(ka[i] >> shift) & 2047u]++;
            b[d] = a[i];
            kb[d] = ka[i];
        }
        a.swap(b);
        ka.swap(kb);
    }
    std::vector<Rec> &sorted = sc.sorted;
    sorted.resize(n);
    for (size_t k = 0; k < n; ++k) sorted[k] = recs[a[k]];
    recs.swap(sorted);
}
}  // namespace

// XY_SCHEDULE_DYNAMIC's order after the sort: the tasks of a (sequence, KV head) whose sequence is
// a chunk over a long prior context (more than one new token, prior context at least as long as
// the chunk) follow the first (largest) of them, in their sorted order; every other task keeps its
// place relative to the rest.  That is, a stable sort by (position of the task's group leader,
// position).  The chunk's query-tile tasks then run at about the same time and read the shared
// prior context while it is in L2 instead of fetching it again from DRAM.
static void group_chunk_tasks(std::vector<Rec> &recs, const int32_t *cu, const int32_t *ctx, int num_seqs,
                              int num_heads_kv, BuildScratch &sc) {
    auto grouped = [&](int i) {
        const int64_t qn = (int64_t)cu[i + 1] - cu[i], L = ctx[i];
        return qn > 1 && L - qn >= qn;
    };
    bool any = false;
    for (int i = 0; i < num_seqs && !any; ++i) any = grouped(i);
    if (!any) return;
    const size_t n = recs.size();
    const size_t ng = (size_t)num_seqs * (size_t)num_heads_kv;
    auto gid = [&](const Rec &r) -> int64_t {
        return grouped(r.t.seq) ? (int64_t)r.t.seq * num_heads_kv + r.t.kv_head : -1;
    };
    // each group's tasks in sorted order: counting sort of the positions by group
    std::vector<int64_t> &start = sc.gstart;
    start.assign(ng + 1, 0);
    for (size_t p = 0; p < n; ++p) {
        const int64_t g = gid(recs[p]);
        if (g >= 0) ++start[g + 1];
    }
    for (size_t g = 0; g < ng; ++g) start[g + 1] += start[g];
    std::vector<uint32_t> &list = sc.glist;
    list.resize((size_t)start[ng]);
    {
        std::vector<int> &fill = sc.count;
        fill.assign(ng, 0);
        for (size_t p = 0; p < n; ++p) {
            const int64_t g = gid(recs[p]);
            if (g >= 0) list[(size_t)(start[g] + fill[g]++)] = (uint32_t)p;
        }
    }
    std::vector<Rec> &out = sc.sorted;
    out.clear();
    out.reserve(n);
    for (size_t p = 0; p < n; ++p) {
        const int64_t g = gid(recs[p]);
        if (g < 0) {
            out.push_back(recs[p]);
        } else if (list[(size_t)start[g]] == (uint32_t)p) {  // the group's leader: the whole group
            for (int64_t q = start[g]; q < start[g + 1]; ++q) out.push_back(recs[list[(size_t)q]]);
        }
    }
    recs.swap(out);
}

// XY_SCHEDULE_MIXED, per CTA: the tasks at positions c, c + num_ctas, ... split into large
// (rows > XY_SCHEDULE_SMALL_ROWS) and small ones, each list in dealt order.  A task's key is
// (its start within its own list + phase) mod 1, with start = charged loads before it / the list's
// total and phase = c / num_ctas; tasks run by increasing key, a large task first on a tie.  The
// keys are compared exactly as fractions over the common denominator big_total * small_total *
// num_ctas (128-bit products; total load < 2^55 and num_ctas <= 2^16 keep them below 2^126).
static void interleave_cta(const std::vector<Rec> &recs, size_t c, size_t num_ctas, int G,
                           std::vector<Rec> &out) {
    using u128 = unsigned __int128;
    struct Item {
        u128 key;
        int kind;
        size_t pos;
    };
    const size_t n = recs.size();
    uint64_t tot[2] = {0, 0};
    for (size_t q = c; q < n; q += num_ctas)
        tot[(int64_t)recs[q].t.q_rows * G > XY_SCHEDULE_SMALL_ROWS ? 0 : 1] += (uint64_t)recs[q].load;
    out.clear();
    if (tot[0] == 0 || tot[1] == 0) {
        for (size_t q = c; q < n; q += num_ctas) out.push_back(recs[q]);
        return;
    }
    std::vector<Item> items;
    uint64_t done[2] = {0, 0};
    for (size_t q = c; q < n; q += num_ctas) {
        const int kind = (int64_t)recs[q].t.q_rows * G > XY_SCHEDULE_SMALL_ROWS ? 0 : 1;
        // numerator over tot[kind] * num_ctas, then scaled by the other list's total
        const u128 span = (u128)tot[kind] * num_ctas;
        const u128 num = ((u128)done[kind] * num_ctas + (u128)c * tot[kind]) % span;
        items.push_back({num * tot[1 - kind], kind, q});
        done[kind] += (uint64_t)recs[q].load;
    }
    std::stable_sort(items.begin(), items.end(), [](const Item &a, const Item &b) {
        return a.key != b.key ? a.key < b.key : a.kind < b.kind;
    });
    for (const Item &it : items) out.push_back(recs[it.pos]);
}

// a4: decomposer + reorder.  Enumeration order sequence -> KV head -> query tile -> KV chunk;
// stable sort by load, largest first; task at sorted position p belongs to CTA p % num_ctas.
// The decomposer and deal: the dealt records in g_scratch.recs, the merge records in
// g_scratch.mrg, the split-KV workspace rows in *ws_rows_out.
static xy_status build_tasks(const int32_t *cu_seqlens_q, const int32_t *context_lens, int num_seqs,
                             int num_heads_q, int num_heads_kv, int head_dim, int causal, int num_ctas,
                             int q_tile, int kv_chunk, int schedule, int64_t *ws_rows_out) {
    if (!cu_seqlens_q || num_seqs < 0 || num_heads_q < 1 || num_heads_kv < 1 || head_dim < 1 ||
        num_ctas < 1 || q_tile < 1 || kv_chunk < 1)
        return XY_ERR_INVALID_ARG;
    if (num_seqs > 0 && !context_lens) return XY_ERR_INVALID_ARG;
    if (num_heads_q % num_heads_kv) return XY_ERR_INVALID_ARG;
    if (schedule != XY_SCHEDULE_AREA && schedule != XY_SCHEDULE_SERPENTINE && schedule != XY_SCHEDULE_MIXED &&
        schedule != XY_SCHEDULE_GREEDY && schedule != XY_SCHEDULE_DYNAMIC)
        return XY_ERR_INVALID_ARG;
    if (cu_seqlens_q[0] != 0) return XY_ERR_CU_SEQLENS;
    const int G = num_heads_q / num_heads_kv;

    BuildScratch &sc = g_scratch;
    std::vector<Rec> &recs = sc.recs;
    std::vector<xy_merge> &mrg = sc.mrg;
    recs.clear();
    mrg.clear();
    {
        // upper bound on the task count (a chunk count from the full context), so that the
        // enumeration below never reallocates
        int64_t bound = 0;
        for (int i = 0; i < num_seqs; ++i) {
            const int64_t qn = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
            const int64_t L = context_lens[i];
            if (qn < 1 || L < qn) break;  // reported by the enumeration
            bound += num_heads_kv * ((qn + q_tile - 1) / q_tile) * ((L + kv_chunk - 1) / kv_chunk);
        }
        recs.reserve((size_t)std::min<int64_t>(bound, int64_t(1) << 26));
    }
    int64_t ws_rows = 0;
    // per query tile of the current sequence: rows, keys it sees, chunk count (the same for every
    // KV head, so computed once per sequence)
    struct Tile {
        int64_t t0, rows, kv_hi, nsplit, charged;
    };
    std::vector<Tile> tiles;
    for (int i = 0; i < num_seqs; ++i) {
        const int64_t qn = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        const int64_t L = context_lens[i];
        if (qn < 1) return XY_ERR_CU_SEQLENS;
        if (L < qn) return XY_ERR_CONTEXT_LT_QLEN;
        tiles.clear();
        for (int64_t t0 = 0; t0 < qn; t0 += q_tile) {
            Tile tl;
            tl.t0 = t0;
            tl.rows = std::min<int64_t>(q_tile, qn - t0);
            tl.kv_hi = causal ? (L - qn + t0 + tl.rows) : L;
            tl.nsplit = (tl.kv_hi + kv_chunk - 1) / kv_chunk;
            tl.charged = tl.rows * G;
            if (schedule == XY_SCHEDULE_MIXED || schedule == XY_SCHEDULE_GREEDY || schedule == XY_SCHEDULE_DYNAMIC)
                tl.charged = XY_SCHEDULE_TILE_ROWS *
                             std::max<int64_t>(1, (tl.charged + XY_SCHEDULE_TILE_ROWS - 1) / XY_SCHEDULE_TILE_ROWS);
            tiles.push_back(tl);
        }
        for (int g = 0; g < num_heads_kv; ++g) {
            for (const Tile &tl : tiles) {
                int64_t base = -1;
                if (tl.nsplit > 1) {
                    base = ws_rows;
                    xy_merge m;
                    m.seq = i;
                    m.kv_head = g;
                    m.q_start = (int32_t)tl.t0;
                    m.q_rows = (int32_t)tl.rows;
                    m.num_splits = (int32_t)tl.nsplit;
                    m.ws_row = (int32_t)base;
                    m.zero0 = 0;
                    m.zero1 = 0;
                    mrg.push_back(m);
                    ws_rows += tl.nsplit * tl.rows * G;
                    if (ws_rows > std::numeric_limits<int32_t>::max()) return XY_ERR_UNSUPPORTED;
                }
                for (int64_t c = 0, k0 = 0; c < tl.nsplit; ++c, k0 += kv_chunk) {
                    const int64_t k1 = std::min<int64_t>(tl.kv_hi, k0 + kv_chunk);
                    Rec r;
                    r.t.seq = i;
                    r.t.kv_head = g;
                    r.t.q_start = (int32_t)tl.t0;
                    r.t.q_rows = (int32_t)tl.rows;
                    r.t.kv_start = (int32_t)k0;
                    r.t.kv_end = (int32_t)k1;
                    r.t.num_splits = (int32_t)tl.nsplit;
                    r.t.ws_row = tl.nsplit == 1 ? -1 : (int32_t)(base + c * tl.rows * G);
                    const bool per_task = schedule == XY_SCHEDULE_GREEDY || schedule == XY_SCHEDULE_DYNAMIC;
                    const int64_t keys = (k1 - k0) + (per_task ? XY_SCHEDULE_TASK_KEYS : 0);
                    r.load = tl.charged * keys;
                    recs.push_back(r);
                }
            }
        }
    }
    for (const Rec &r : recs)
        if (r.load >= (int64_t(1) << 55)) return XY_ERR_UNSUPPORTED;
    {
        // stable sort by load, largest first
        sort_by_load_desc(recs, sc);
    }
    if (schedule == XY_SCHEDULE_DYNAMIC) group_chunk_tasks(recs, cu_seqlens_q, context_lens, num_seqs, num_heads_kv, sc);
    if (schedule == XY_SCHEDULE_SERPENTINE || schedule == XY_SCHEDULE_MIXED) {
        // serpentine deal: every complete odd round of num_ctas positions is reversed
        const size_t n = (size_t)num_ctas;
        for (size_t r = 1; (r + 1) * n <= recs.size(); r += 2)
            std::reverse(recs.begin() + r * n, recs.begin() + (r + 1) * n);
    }
    if (schedule == XY_SCHEDULE_MIXED) {
        int64_t total = 0;
        for (const Rec &r : recs) total += r.load;
        if (total >= (int64_t(1) << 55) || num_ctas > (1 << 16)) return XY_ERR_UNSUPPORTED;
        const size_t n = recs.size();
        std::vector<Rec> out;
        for (size_t c = 0; c < (size_t)num_ctas && c < n; ++c) {
            interleave_cta(recs, c, (size_t)num_ctas, G, out);
            size_t k = 0;
            for (size_t q = c; q < n; q += num_ctas) recs[q] = out[k++];
        }
    }
    if (schedule == XY_SCHEDULE_GREEDY) {
        int64_t total = 0;
        for (const Rec &r : recs) total += r.load;
        if (total >= (int64_t(1) << 55)) return XY_ERR_UNSUPPORTED;
        // longest processing time first: each task (in sorted order) to the least loaded CTA,
        // the lowest index on ties; unused positions become holes.  A tournament tree over the
        // CTAs (leaf c at W + c, W a power of two; padding leaves carry an infinite load) keeps
        // the winner of (load, index) at the root; a task's load re-runs one leaf-to-root path.
        const int C = num_ctas;
        int W = 1;
        while (W < C) W <<= 1;
        std::vector<int64_t> &load = sc.tload;
        std::vector<int> &tree = sc.tree, &cta_of = sc.cta_of, &pos_of = sc.pos_of, &count = sc.count;
        load.assign(W, std::numeric_limits<int64_t>::max());
        for (int c = 0; c < C; ++c) load[c] = 0;
        tree.assign(2 * W, 0);
        for (int c = 0; c < W; ++c) tree[W + c] = c;
        auto win = [&](int a, int b) { return load[b] < load[a] ? b : a; };  // a < b: ties keep a
        for (int i = W - 1; i >= 1; --i) tree[i] = win(tree[2 * i], tree[2 * i + 1]);
        cta_of.resize(recs.size());
        pos_of.resize(recs.size());
        count.assign(C, 0);
        for (size_t k = 0; k < recs.size(); ++k) {
            const int c = tree[1];
            cta_of[k] = c;
            pos_of[k] = count[c]++;
            load[c] += recs[k].load;
            for (int i = (W + c) >> 1; i >= 1; i >>= 1) tree[i] = win(tree[2 * i], tree[2 * i + 1]);
        }
        size_t depth = 0;
        for (int c = 0; c < C; ++c) depth = std::max(depth, (size_t)count[c]);
        if (depth * (size_t)num_ctas > (size_t)std::numeric_limits<int32_t>::max()) return XY_ERR_UNSUPPORTED;
        Rec hole;
        hole.t = xy_task{-1, 0, 0, 0, 0, 0, 0, -1};
        hole.load = 0;
        std::vector<Rec> &dealt = sc.sorted;
        dealt.assign(depth * (size_t)num_ctas, hole);
        for (size_t k = 0; k < recs.size(); ++k) dealt[(size_t)pos_of[k] * num_ctas + cta_of[k]] = recs[k];
        recs.swap(dealt);
    }

    *ws_rows_out = ws_rows;
    return XY_OK;
}

static void task_stats(const std::vector<Rec> &recs, int num_ctas, xy_task_stats *stats) {
    std::vector<int64_t> &cta = g_scratch.tload;   // (free once the builder has returned)
    cta.assign(num_ctas, 0);
    int64_t total = 0;
    for (size_t k = 0, c = 0; k < recs.size(); ++k) {   // position k belongs to CTA k mod num_ctas
        cta[c] += recs[k].load;
        total += recs[k].load;
        if (++c == (size_t)num_ctas) c = 0;
    }
    const int64_t mx = *std::max_element(cta.begin(), cta.end());
    const int64_t mn = *std::min_element(cta.begin(), cta.end());
    stats->total_load = total;
    stats->max_cta_load = mx;
    stats->min_cta_load = mn;
    stats->balance = mx > 0 ? (double)mn / (double)mx : 1.0;
}

extern "C" xy_status xy_default_tiles(int num_heads_q, int num_heads_kv, int head_dim, int kv_fp8, int pure_decode,
                                      int *q_tile, int *kv_chunk) {
    if (!q_tile || !kv_chunk || num_heads_kv < 1 || num_heads_q < num_heads_kv || num_heads_q % num_heads_kv)
        return XY_ERR_INVALID_ARG;
    const int G = num_heads_q / num_heads_kv;
    const int narrow = 64 / G > 1 ? 64 / G : 1;   // rows of a decode-path task: at most 64
    if (kv_fp8)
        *q_tile = pure_decode && G <= XY_FP8_NARROW_ROWS ? 1 : narrow;
    else if (head_dim == 128 && 128 % G == 0)
        *q_tile = 256 / G;   // two 128-row tcgen05 tiles
    else
        *q_tile = narrow;
    *kv_chunk = XY_DEFAULT_KV_CHUNK;
    return XY_OK;
}

// Batch-aware KV chunk: among 8192, 16384, 32768 and 65536 keys, the chunk whose estimated
// makespan is least.  Each (sequence, KV head) pair streams its L context keys in ceil(L / c)
// tasks; a task costs its keys plus a fixed overhead (task set-up, the cross-warp merge, a split
// partial), and the estimate is the larger of the average load of a CTA and what the full-size
// chunks alone need when dealt longest first (ceil(full / CTAs) of them on the busiest CTA).  Ties
// go to the longer chunk (fewer partials to merge).  The 8-bit pure-decode kernel with G <= 8 runs
// two CTAs per SM slot (xy_paged_attention_fp8_dynamic), so its chunks are sized for twice the CTAs.
extern "C" xy_status xy_default_kv_chunk(const int32_t *context_lens, int num_seqs, int num_heads_q,
                                         int num_heads_kv, int kv_fp8, int pure_decode, int num_ctas,
                                         int *kv_chunk) {
    if (!kv_chunk || num_seqs < 0 || (num_seqs > 0 && !context_lens) || num_heads_kv < 1 ||
        num_heads_q < num_heads_kv || num_heads_q % num_heads_kv || num_ctas < 1)
        return XY_ERR_INVALID_ARG;
    const int G = num_heads_q / num_heads_kv;
    // pure decode batches under the dynamic deal run two half-size CTAs per SM slot (8-bit pages:
    // G <= 8; bf16 pages: every pure decode batch, G <= 16)
    const double ctas = (double)num_ctas * (pure_decode && G <= (kv_fp8 ? 8 : 16) ? 2 : 1);
    constexpr double kTaskOverheadKeys = 512.0;
    int best = XY_DEFAULT_KV_CHUNK;
    double best_t = -1.0;
    for (int c = 8192; c <= 65536; c *= 2) {
        double keys = 0.0, tasks = 0.0, full = 0.0;
        int longest = 0;
        for (int i = 0; i < num_seqs; ++i) {
            const int L = context_lens[i];
            if (L < 0) return XY_ERR_INVALID_ARG;
            keys += L;
            tasks += (L + c - 1) / c;
            full += L / c;
            longest = L > longest ? L : longest;
        }
        keys *= num_heads_kv, tasks *= num_heads_kv, full *= num_heads_kv;
        const double avg = (keys + kTaskOverheadKeys * tasks) / ctas;
        const double rounds = std::ceil(full / ctas) * ((double)c + kTaskOverheadKeys);
        const double t = std::max(std::max(avg, rounds), (double)std::min(c, longest) + kTaskOverheadKeys);
        if (best_t < 0.0 || t <= best_t) {
            best_t = t;
            best = c;
        }
    }
    *kv_chunk = best;
    return XY_OK;
}

extern "C" xy_status xy_build_task_table(const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                         int num_seqs, int num_heads_q, int num_heads_kv,
                                         int head_dim, int causal, int num_ctas, int q_tile,
                                         int kv_chunk, int schedule, xy_task *tasks, int max_tasks,
                                         int *num_tasks, xy_merge *merges, int max_merges,
                                         int *num_merges, size_t *workspace_bytes,
                                         xy_task_stats *stats) {
    if (!num_tasks || !num_merges || !workspace_bytes) return XY_ERR_INVALID_ARG;
    int64_t ws_rows = 0;
    const xy_status st = build_tasks(cu_seqlens_q, context_lens, num_seqs, num_heads_q, num_heads_kv, head_dim,
                                     causal, num_ctas, q_tile, kv_chunk, schedule, &ws_rows);
    if (st != XY_OK) return st;
    const std::vector<Rec> &recs = g_scratch.recs;
    const std::vector<xy_merge> &mrg = g_scratch.mrg;
    *num_tasks = (int)recs.size();
    *num_merges = (int)mrg.size();
    *workspace_bytes = (size_t)ws_rows * (size_t)(head_dim + 1) * 4u;
    if (tasks) {
        if (max_tasks < (int)recs.size()) return XY_ERR_CAPACITY;
        for (size_t k = 0; k < recs.size(); ++k) tasks[k] = recs[k].t;
    }
    if (merges) {
        if (max_merges < (int)mrg.size()) return XY_ERR_CAPACITY;
        if (!mrg.empty()) std::memcpy(merges, mrg.data(), mrg.size() * sizeof(xy_merge));
    }
    if (stats) task_stats(recs, num_ctas, stats);
    return XY_OK;
}

// One step's host-built metadata packed for a single host->device copy (see xy.h).
extern "C" xy_status xy_build_step_tables(const int32_t *cu_seqlens_q, const int32_t *context_lens, int num_seqs,
                                          const int32_t *free_list, int num_free, int block_size, int max_blocks,
                                          int num_heads_q, int num_heads_kv, int head_dim, int causal, int num_ctas,
                                          int q_tile, int kv_chunk, int schedule, void *staging,
                                          size_t staging_bytes, xy_step_tables *out) {
    if (!out || (staging_bytes > 0 && !staging) || max_blocks < 1) return XY_ERR_INVALID_ARG;
    int64_t ws_rows = 0;
    xy_status st = build_tasks(cu_seqlens_q, context_lens, num_seqs, num_heads_q, num_heads_kv, head_dim, causal,
                               num_ctas, q_tile, kv_chunk, schedule, &ws_rows);
    if (st != XY_OK) return st;
    const std::vector<Rec> &recs = g_scratch.recs;
    const std::vector<xy_merge> &mrg = g_scratch.mrg;
    const size_t A = XY_STEP_TABLES_ALIGN;
    auto up = [&](size_t x) { return (x + A - 1) / A * A; };
    const size_t S = (size_t)num_seqs;
    out->err_off = 0;
    out->cu_off = up(4);
    out->ctx_off = up(out->cu_off + 4 * (S + 1));
    out->bt_off = up(out->ctx_off + 4 * S);
    out->tasks_off = up(out->bt_off + 4 * S * (size_t)max_blocks);
    out->merges_off = up(out->tasks_off + sizeof(xy_task) * recs.size());
    out->bytes = out->merges_off + sizeof(xy_merge) * mrg.size();
    out->num_tasks = (int)recs.size();
    out->num_merges = (int)mrg.size();
    out->workspace_bytes = (size_t)ws_rows * (size_t)(head_dim + 1) * 4u;
    task_stats(recs, num_ctas, &out->stats);
    out->pages_used = 0;
    if (out->bytes > staging_bytes) return XY_ERR_CAPACITY;
    uint8_t *base = static_cast<uint8_t *>(staging);
    st = xy_build_block_table(context_lens, num_seqs, block_size, free_list, num_free, max_blocks,
                              reinterpret_cast<int32_t *>(base + out->bt_off), &out->pages_used);
    if (st != XY_OK) return st;
    const int32_t zero = 0;
    std::memcpy(base + out->err_off, &zero, 4);
    std::memcpy(base + out->cu_off, cu_seqlens_q, 4 * (S + 1));
    if (S) std::memcpy(base + out->ctx_off, context_lens, 4 * S);
    xy_task *t = reinterpret_cast<xy_task *>(base + out->tasks_off);
    for (size_t k = 0; k < recs.size(); ++k) t[k] = recs[k].t;
    if (!mrg.empty()) std::memcpy(base + out->merges_off, mrg.data(), sizeof(xy_merge) * mrg.size());
    return XY_OK;
}

namespace {
thread_local std::vector<xy_task> g_tile_tasks, g_dec_tasks;
thread_local std::vector<xy_merge> g_tile_merges, g_dec_merges;
thread_local std::vector<int32_t> g_cu_part;
}  // namespace

extern "C" xy_status xy_build_fp8_step_tables(const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                              int num_seqs, const int32_t *free_list, int num_free, int block_size,
                                              int max_blocks, int num_heads_q, int num_heads_kv, int head_dim,
                                              int causal, int num_ctas, void *staging, size_t staging_bytes,
                                              xy_fp8_step_tables *out) {
    if (!out || !cu_seqlens_q || (num_seqs > 0 && !context_lens) || (staging_bytes > 0 && !staging) ||
        max_blocks < 1 || num_seqs < 0 || num_heads_kv < 1 || num_heads_q < num_heads_kv ||
        num_heads_q % num_heads_kv || num_ctas < 1 || !is_pow2(block_size) || block_size < 16)
        return XY_ERR_INVALID_ARG;
    const int G = num_heads_q / num_heads_kv;
    if (head_dim != 128 || 128 % G) return XY_ERR_UNSUPPORTED;
    if (cu_seqlens_q[0] != 0) return XY_ERR_CU_SEQLENS;
    for (int i = 0; i < num_seqs; ++i)
        if (cu_seqlens_q[i + 1] <= cu_seqlens_q[i]) return XY_ERR_CU_SEQLENS;
    // the two kinds of sequences must form one contiguous range each
    int changes = 0;
    for (int i = 1; i < num_seqs; ++i) {
        const bool a = cu_seqlens_q[i] - cu_seqlens_q[i - 1] > 1, b = cu_seqlens_q[i + 1] - cu_seqlens_q[i] > 1;
        changes += a != b;
    }
    if (changes > 1) return XY_ERR_UNSUPPORTED;
    int k = num_seqs;  // first sequence of the second range
    for (int i = 1; i < num_seqs; ++i)
        if ((cu_seqlens_q[i] - cu_seqlens_q[i - 1] > 1) != (cu_seqlens_q[i + 1] - cu_seqlens_q[i] > 1)) {
            k = i;
            break;
        }
    const bool multi_first = num_seqs > 0 && cu_seqlens_q[1] - cu_seqlens_q[0] > 1;
    int ta = 0, tb = 0, da = 0, db = 0;
    if (multi_first) {
        ta = 0, tb = k, da = k, db = num_seqs;
    } else {
        da = 0, db = k, ta = k, tb = num_seqs;
    }
    std::memset(out, 0, sizeof(*out));
    out->tile_seq_begin = ta, out->tile_seq_end = tb, out->dec_seq_begin = da, out->dec_seq_end = db;
    out->tile_tok_begin = cu_seqlens_q[ta], out->tile_tok_end = cu_seqlens_q[tb];
    out->dec_tok_begin = cu_seqlens_q[da], out->dec_tok_end = cu_seqlens_q[db];

    // the two parts' task tables (dynamic deal), each with its own sequences renumbered from 0
    g_tile_tasks.clear(), g_dec_tasks.clear(), g_tile_merges.clear(), g_dec_merges.clear();
    auto part = [&](int a, int b, int kv_fp8, std::vector<xy_task> &tasks, std::vector<xy_merge> &merges,
                    size_t *ws_bytes) -> xy_status {
        if (b <= a) return XY_OK;
        g_cu_part.resize((size_t)(b - a + 1));
        for (int i = a; i <= b; ++i) g_cu_part[(size_t)(i - a)] = cu_seqlens_q[i] - cu_seqlens_q[a];
        int q_tile = 0, kv_chunk = 0;
        xy_status st = xy_default_tiles(num_heads_q, num_heads_kv, head_dim, kv_fp8, kv_fp8, &q_tile, &kv_chunk);
        if (st != XY_OK) return st;
        st = xy_default_kv_chunk(context_lens + a, b - a, num_heads_q, num_heads_kv, kv_fp8, kv_fp8, num_ctas,
                                 &kv_chunk);
        if (st != XY_OK) return st;
        int64_t ws_rows = 0;
        st = build_tasks(g_cu_part.data(), context_lens + a, b - a, num_heads_q, num_heads_kv, head_dim, causal,
                         num_ctas, q_tile, kv_chunk, XY_SCHEDULE_DYNAMIC, &ws_rows);
        if (st != XY_OK) return st;
        tasks.resize(g_scratch.recs.size());
        for (size_t r = 0; r < tasks.size(); ++r) tasks[r] = g_scratch.recs[r].t;
        merges = g_scratch.mrg;
        *ws_bytes = (size_t)ws_rows * (size_t)(head_dim + 1) * 4u;
        return XY_OK;
    };
    xy_status st = part(ta, tb, 0, g_tile_tasks, g_tile_merges, &out->tile_workspace_bytes);
    if (st != XY_OK) return st;
    st = part(da, db, 1, g_dec_tasks, g_dec_merges, &out->dec_workspace_bytes);
    if (st != XY_OK) return st;
    // pages the tile part reads (its sequences' pages in order), copied to bf16 page i
    int64_t n_pages = 0;
    for (int i = ta; i < tb; ++i) n_pages += ((int64_t)context_lens[i] + block_size - 1) / block_size;
    if (n_pages > INT32_MAX) return XY_ERR_UNSUPPORTED;
    out->tile_num_pages = (int)n_pages;
    out->tile_num_tasks = (int)g_tile_tasks.size(), out->tile_num_merges = (int)g_tile_merges.size();
    out->dec_num_tasks = (int)g_dec_tasks.size(), out->dec_num_merges = (int)g_dec_merges.size();

    const size_t A = XY_STEP_TABLES_ALIGN;
    auto up = [&](size_t x) { return (x + A - 1) / A * A; };
    const size_t S = (size_t)num_seqs, MB = (size_t)max_blocks;
    const size_t nt = (size_t)(tb - ta), nd = (size_t)(db - da);
    out->err_off = 0;
    out->cu_off = up(4);
    out->ctx_off = up(out->cu_off + 4 * (S + 1));
    out->bt_off = up(out->ctx_off + 4 * S);
    out->tile_cu_off = up(out->bt_off + 4 * S * MB);
    out->tile_bt_off = up(out->tile_cu_off + 4 * (nt + 1));
    out->tile_pages_off = up(out->tile_bt_off + 4 * nt * MB);
    out->tile_tasks_off = up(out->tile_pages_off + 4 * (size_t)n_pages);
    out->tile_merges_off = up(out->tile_tasks_off + sizeof(xy_task) * g_tile_tasks.size());
    out->dec_cu_off = up(out->tile_merges_off + sizeof(xy_merge) * g_tile_merges.size());
    out->dec_tasks_off = up(out->dec_cu_off + 4 * (nd + 1));
    out->dec_merges_off = up(out->dec_tasks_off + sizeof(xy_task) * g_dec_tasks.size());
    out->bytes = out->dec_merges_off + sizeof(xy_merge) * g_dec_merges.size();
    if (out->bytes > staging_bytes) return XY_ERR_CAPACITY;

    uint8_t *base = static_cast<uint8_t *>(staging);
    int32_t *bt = reinterpret_cast<int32_t *>(base + out->bt_off);
    st = xy_build_block_table(context_lens, num_seqs, block_size, free_list, num_free, max_blocks, bt,
                              &out->pages_used);
    if (st != XY_OK) return st;
    const int32_t zero = 0;
    std::memcpy(base + out->err_off, &zero, 4);
    std::memcpy(base + out->cu_off, cu_seqlens_q, 4 * (S + 1));
    if (S) std::memcpy(base + out->ctx_off, context_lens, 4 * S);
    int32_t *cu_t = reinterpret_cast<int32_t *>(base + out->tile_cu_off);
    int32_t *bt_t = reinterpret_cast<int32_t *>(base + out->tile_bt_off);
    int32_t *pages = reinterpret_cast<int32_t *>(base + out->tile_pages_off);
    int32_t next = 0;
    for (int i = ta; i <= tb && tb > ta; ++i) cu_t[i - ta] = cu_seqlens_q[i] - cu_seqlens_q[ta];
    for (int i = ta; i < tb; ++i) {
        const int32_t n = (int32_t)(((int64_t)context_lens[i] + block_size - 1) / block_size);
        int32_t *row = bt_t + (size_t)(i - ta) * MB;
        for (int32_t j = 0; j < max_blocks; ++j) row[j] = j < n ? next + j : -1;
        for (int32_t j = 0; j < n; ++j) pages[next + j] = bt[(size_t)i * MB + j];
        next += n;
    }
    int32_t *cu_d = reinterpret_cast<int32_t *>(base + out->dec_cu_off);
    for (int i = da; i <= db && db > da; ++i) cu_d[i - da] = cu_seqlens_q[i] - cu_seqlens_q[da];
    if (!g_tile_tasks.empty())
        std::memcpy(base + out->tile_tasks_off, g_tile_tasks.data(), sizeof(xy_task) * g_tile_tasks.size());
    if (!g_tile_merges.empty())
        std::memcpy(base + out->tile_merges_off, g_tile_merges.data(), sizeof(xy_merge) * g_tile_merges.size());
    if (!g_dec_tasks.empty())
        std::memcpy(base + out->dec_tasks_off, g_dec_tasks.data(), sizeof(xy_task) * g_dec_tasks.size());
    if (!g_dec_merges.empty())
        std::memcpy(base + out->dec_merges_off, g_dec_merges.data(), sizeof(xy_merge) * g_dec_merges.size());
    return XY_OK;
}
