// Host side of libxy: status strings, the block-table allocator (a1) and the task-table
// builder (a4).  Pure host code, no CUDA calls, so it runs and is tested without a GPU.
//
// Sources: "XY-Serve 深度实战" (chenxutan.com/d/5031) §2.2 components 1-2, §4.2, §4.4;
// cann-recipes-infer Paged KV Cache / Packed Sequence notes (dpshk.com/news/5336026) §2.2, §3.2.

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <limits>
#include <queue>
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
        for (int64_t j = 0; j < max_blocks; ++j) row[j] = j < n ? free_list[pos + j] : -1;
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
}  // namespace

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
extern "C" xy_status xy_build_task_table(const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                         int num_seqs, int num_heads_q, int num_heads_kv,
                                         int head_dim, int causal, int num_ctas, int q_tile,
                                         int kv_chunk, int schedule, xy_task *tasks, int max_tasks,
                                         int *num_tasks, xy_merge *merges, int max_merges,
                                         int *num_merges, size_t *workspace_bytes,
                                         xy_task_stats *stats) {
    if (!cu_seqlens_q || num_seqs < 0 || num_heads_q < 1 || num_heads_kv < 1 || head_dim < 1 ||
        num_ctas < 1 || q_tile < 1 || kv_chunk < 1 || !num_tasks || !num_merges || !workspace_bytes)
        return XY_ERR_INVALID_ARG;
    if (num_seqs > 0 && !context_lens) return XY_ERR_INVALID_ARG;
    if (num_heads_q % num_heads_kv) return XY_ERR_INVALID_ARG;
    if (schedule != XY_SCHEDULE_AREA && schedule != XY_SCHEDULE_SERPENTINE && schedule != XY_SCHEDULE_MIXED &&
        schedule != XY_SCHEDULE_GREEDY)
        return XY_ERR_INVALID_ARG;
    if (cu_seqlens_q[0] != 0) return XY_ERR_CU_SEQLENS;
    const int G = num_heads_q / num_heads_kv;

    std::vector<Rec> recs;
    std::vector<xy_merge> mrg;
    int64_t ws_rows = 0;
    for (int i = 0; i < num_seqs; ++i) {
        const int64_t qn = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        const int64_t L = context_lens[i];
        if (qn < 1) return XY_ERR_CU_SEQLENS;
        if (L < qn) return XY_ERR_CONTEXT_LT_QLEN;
        for (int g = 0; g < num_heads_kv; ++g) {
            for (int64_t t0 = 0; t0 < qn; t0 += q_tile) {
                const int64_t rows = std::min<int64_t>(q_tile, qn - t0);
                const int64_t kv_hi = causal ? (L - qn + t0 + rows) : L;
                const int64_t nsplit = (kv_hi + kv_chunk - 1) / kv_chunk;
                int64_t base = -1;
                if (nsplit > 1) {
                    base = ws_rows;
                    xy_merge m;
                    m.seq = i;
                    m.kv_head = g;
                    m.q_start = (int32_t)t0;
                    m.q_rows = (int32_t)rows;
                    m.num_splits = (int32_t)nsplit;
                    m.ws_row = (int32_t)base;
                    m.zero0 = 0;
                    m.zero1 = 0;
                    mrg.push_back(m);
                    ws_rows += nsplit * rows * G;
                    if (ws_rows > std::numeric_limits<int32_t>::max()) return XY_ERR_UNSUPPORTED;
                }
                for (int64_t c = 0; c < nsplit; ++c) {
                    const int64_t k0 = c * kv_chunk;
                    const int64_t k1 = std::min<int64_t>(kv_hi, k0 + kv_chunk);
                    Rec r;
                    r.t.seq = i;
                    r.t.kv_head = g;
                    r.t.q_start = (int32_t)t0;
                    r.t.q_rows = (int32_t)rows;
                    r.t.kv_start = (int32_t)k0;
                    r.t.kv_end = (int32_t)k1;
                    r.t.num_splits = (int32_t)nsplit;
                    r.t.ws_row = nsplit == 1 ? -1 : (int32_t)(base + c * rows * G);
                    int64_t charged = rows * G, keys = k1 - k0;
                    if (schedule == XY_SCHEDULE_MIXED || schedule == XY_SCHEDULE_GREEDY)
                        charged = XY_SCHEDULE_TILE_ROWS *
                                  std::max<int64_t>(1, (charged + XY_SCHEDULE_TILE_ROWS - 1) / XY_SCHEDULE_TILE_ROWS);
                    if (schedule == XY_SCHEDULE_GREEDY) keys += XY_SCHEDULE_TASK_KEYS;
                    r.load = charged * keys;
                    recs.push_back(r);
                }
            }
        }
    }
    std::stable_sort(recs.begin(), recs.end(),
                     [](const Rec &a, const Rec &b) { return a.load > b.load; });
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
        // the lowest index on ties; unused positions become holes
        using Slot = std::pair<int64_t, int>;
        std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
        for (int c = 0; c < num_ctas; ++c) heap.push({0, c});
        std::vector<std::vector<size_t>> lists(num_ctas);
        for (size_t k = 0; k < recs.size(); ++k) {
            Slot s = heap.top();
            heap.pop();
            lists[s.second].push_back(k);
            heap.push({s.first + recs[k].load, s.second});
        }
        size_t depth = 0;
        for (const auto &l : lists) depth = std::max(depth, l.size());
        if (depth * (size_t)num_ctas > (size_t)std::numeric_limits<int32_t>::max()) return XY_ERR_UNSUPPORTED;
        Rec hole;
        hole.t = xy_task{-1, 0, 0, 0, 0, 0, 0, -1};
        hole.load = 0;
        std::vector<Rec> dealt(depth * (size_t)num_ctas, hole);
        for (int c = 0; c < num_ctas; ++c)
            for (size_t pos = 0; pos < lists[c].size(); ++pos) dealt[pos * num_ctas + c] = recs[lists[c][pos]];
        recs.swap(dealt);
    }

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
    if (stats) {
        std::vector<int64_t> cta(num_ctas, 0);
        int64_t total = 0;
        for (size_t k = 0; k < recs.size(); ++k) {
            cta[k % num_ctas] += recs[k].load;
            total += recs[k].load;
        }
        const int64_t mx = *std::max_element(cta.begin(), cta.end());
        const int64_t mn = *std::min_element(cta.begin(), cta.end());
        stats->total_load = total;
        stats->max_cta_load = mx;
        stats->min_cta_load = mn;
        stats->balance = mx > 0 ? (double)mn / (double)mx : 1.0;
    }
    return XY_OK;
}
