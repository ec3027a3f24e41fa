/*
 * xy.h — C ABI of libxy: unified attention over a block-paged KV cache for a continuous
 * batch of packed variable-length queries, on one NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages on the subject, cited by title and section):
 *   [XY]    "XY-Serve 深度实战：当昇腾 NPU 终于学会「驯服动态负载」" (chenxutan.com/d/5031)
 *   [MindIE] MindIE serving notes (hwcomputing.csdn.net/6a130621662f9a54cb76c319)
 *   [CANN]  cann-recipes-infer Paged KV Cache / Packed Sequence notes (dpshk.com/news/5336026)
 *   [ATB]   ATB dynamic batching / speculative decoding / KV reuse notes (ai6s.net/6a38a2a6662f9a54cb828d66)
 *
 * One step of the path, in call order:
 *   xy_build_block_table  (host)   logical -> physical page table from a FIFO free list
 *   xy_slot_mapping       (device) physical slot of every new packed token
 *   xy_kv_append          (device) write the new tokens' K/V into their slots
 *   xy_build_task_table   (host)   decompose the batch into load-sorted, round-robin dealt tasks
 *   xy_paged_attention    (device) fused QK^T -> masked online softmax -> PV over the pages,
 *                                  plus the split-KV merge
 *
 * Conventions shared by every call:
 *   - Notation: S sequences, T = cu_seqlens_q[S] packed new tokens, Hq query heads, Hkv KV heads
 *     (Hq % Hkv == 0, query head h reads KV head h / (Hq/Hkv)), d = head_dim, bs = block_size,
 *     P = num_pages, MB = max_blocks (columns of the block table).
 *   - context_lens[i] = L_i counts the keys of sequence i INCLUDING its q_i new tokens;
 *     new token j of sequence i sits at absolute position L_i - q_i + j.  1 <= q_i <= L_i.
 *   - Causal attention is aligned bottom-right: new token j sees keys 0 .. L_i - q_i + j.
 *   - Layouts (all row-major, contiguous): q/out [T, Hq, d] bf16; k_new/v_new [T, Hkv, d] bf16;
 *     k_pages/v_pages [P, Hkv, bs, d] bf16 (one page of one head is a contiguous bs*d block);
 *     block_table [S, MB] int32, -1 = unallocated; cu_seqlens_q [S+1] int32; context_lens [S]
 *     int32; slot_mapping [T] int64, slot = page * bs + offset, negative = skip.
 *   - Ownership: the caller allocates and frees every buffer; the library never allocates
 *     device memory, never frees, never synchronises.  Device calls are asynchronous on the
 *     given stream (a cudaStream_t passed as void*, NULL = legacy default stream).
 *   - Device: a device call launches on the calling thread's current CUDA device (cudaGetDevice)
 *     and keeps its per-device state (kernel attributes, the no-alloc scratch) by it; every device
 *     pointer and the stream must belong to that device.  The Python binding checks this.
 *   - Errors: every call returns an xy_status; no exception crosses the ABI.  Host-visible
 *     argument errors are reported before anything is launched.  Errors that only the device
 *     can see (a page index outside [0, P), a slot outside the pool, a malformed task, a
 *     bounded wait that expired) are OR-ed into *err_word (a device int32 the caller zeroes and
 *     reads back after the stream has completed, see XY_DEV_*); the contents of the outputs are
 *     then unspecified.  No kernel traps, asserts or waits without a bound.
 */
#ifndef XY_H
#define XY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    XY_OK = 0,
    XY_ERR_INVALID_ARG = -1,      /* null pointer, bad size, misaligned pointer */
    XY_ERR_CU_SEQLENS = -2,       /* cu_seqlens_q[0] != 0 or not strictly increasing ([CANN] §4.4) */
    XY_ERR_PAGE_OOB = -3,         /* a block-table entry outside [0, P) ([CANN] §4.4) */
    XY_ERR_CONTEXT_LT_QLEN = -4,  /* some context_lens[i] < q_i */
    XY_ERR_UNSUPPORTED = -5,      /* shape the kernels do not handle (head_dim, block_size, tiles) */
    XY_ERR_WORKSPACE = -6,        /* workspace missing or smaller than xy_build_task_table asked for */
    XY_ERR_CUDA = -7,             /* a CUDA runtime/driver call failed */
    XY_ERR_TIMEOUT = -8,          /* reserved for a host-side wait; device waits use XY_DEV_TIMEOUT */
    XY_ERR_OUT_OF_PAGES = -9,     /* free list exhausted ([XY] §4.2 allocator raises) */
    XY_ERR_CAPACITY = -10         /* an output array given to a host call is too small */
} xy_status;

/* Bits OR-ed into *err_word by device code. */
#define XY_DEV_PAGE_OOB   0x1     /* block-table entry needed by a key < L is outside [0, P) */
#define XY_DEV_SLOT_OOB   0x2     /* slot outside [0, P*bs) in xy_kv_append */
#define XY_DEV_BAD_TASK   0x4     /* task record violates the kernel's tile constraints */
#define XY_DEV_TIMEOUT    0x8     /* a bounded mbarrier wait expired; the kernel returned early */

/* One unit of attention work: rows [q_start, q_start + q_rows) of sequence `seq` (token index
 * relative to the sequence) for all G = Hq/Hkv query heads of KV head `kv_head`, against keys
 * [kv_start, kv_end).  num_splits > 1 means the tile's KV range is cut into that many chunks;
 * this chunk then writes its normalised partial output and log-sum-exp to workspace rows
 * ws_row + t*G + h_local (t < q_rows, h_local < G) instead of `out`; ws_row = -1 otherwise. */
typedef struct {
    int32_t seq, kv_head, q_start, q_rows, kv_start, kv_end, num_splits, ws_row;
} xy_task;

/* One split tile to merge: chunk c of the tile owns workspace rows
 * ws_row + c*q_rows*G + t*G + h_local.  zero0/zero1 are 0. */
typedef struct {
    int32_t seq, kv_head, q_start, q_rows, num_splits, ws_row, zero0, zero1;
} xy_merge;

/* Balance of the static deal ([XY] §2.2 component 2: balance ratio = min/max core load). */
typedef struct {
    int64_t total_load;
    int64_t max_cta_load;
    int64_t min_cta_load;
    double balance;           /* min/max of per-CTA load sums, 1.0 for an empty batch */
} xy_task_stats;

/* Static description of a status code ("ok", "invalid argument", ...). Never NULL. */
const char *xy_status_string(int status);

/* Text of the CUDA error behind the last XY_ERR_CUDA returned on the calling host thread (or ""
 * if none).  The pointer stays valid until the next libxy call on that thread. */
const char *xy_last_error_string(void);

/* Library ABI version (major * 100 + minor). */
int xy_version(void);

/* Number of CTAs the persistent attention kernel runs per GPU (SM count x CTAs per SM) for
 * `device`, or a negative xy_status.  Host call; needs a CUDA device. */
int xy_default_num_ctas(int device);

/*
 * a1 — block table ([CANN] §2.2 page table, §3.2 allocate_pages; [XY] §4.2 KVCacheAllocator).
 * Host call, pure.  For sequences in batch order, takes ceil(L_i / bs) pages from the front of
 * free_list (FIFO) and writes them to block_table[i][0..n_i); the rest of row i is -1.
 *   context_lens [num_seqs] host; free_list [num_free] host, physical page ids;
 *   block_table [num_seqs, max_blocks] host, written in full; *pages_used = pages taken.
 * Errors: XY_ERR_INVALID_ARG (null pointers, num_seqs < 0, block_size not a power of two >= 16,
 *   L_i < 1), XY_ERR_CAPACITY (ceil(L_i/bs) > max_blocks), XY_ERR_OUT_OF_PAGES (list exhausted).
 */
xy_status xy_build_block_table(const int32_t *context_lens, int num_seqs, int block_size,
                               const int32_t *free_list, int num_free, int max_blocks,
                               int32_t *block_table, int *pages_used);

/*
 * a2 — slot mapping (pages silent; reading: new token j of sequence i at absolute position
 * p = L_i - q_i + j goes to slot block_table[i][p / bs] * bs + p % bs).  Device call.
 *   cu_seqlens_q [num_seqs+1], context_lens [num_seqs], block_table [num_seqs, max_blocks]:
 *   device int32; slot_mapping [num_tokens] device int64, written in full.
 * A block-table entry outside [0, num_pages) sets XY_DEV_PAGE_OOB and that token's slot to -1.
 * Errors: XY_ERR_INVALID_ARG, XY_ERR_CUDA (launch failure).
 */
xy_status xy_slot_mapping(const int32_t *cu_seqlens_q, const int32_t *context_lens,
                          const int32_t *block_table, int num_seqs, int max_blocks, int num_tokens,
                          int block_size, int num_pages, int64_t *slot_mapping, int32_t *err_word,
                          void *stream);

/*
 * a3 — KV append ([CANN] §2.2 pages filled on demand, §3.1 page layout; [ATB] KV缓存复用:
 * chunked prefill appends to the existing cache).  Device call: for every token t with
 * slot_mapping[t] >= 0 and every KV head h, copies k_new[t][h][:] to
 * k_pages[slot / bs][h][slot % bs][:] and the same for V.  Bit copy; tokens are written in no
 * particular order, so two tokens with the same slot leave either one's data.
 *   k_new, v_new [num_tokens, Hkv, d] bf16 device; slot_mapping [num_tokens] int64 device;
 *   k_pages, v_pages [num_pages, Hkv, bs, d] bf16 device, updated in place.
 * All pointers 16-byte aligned; head_dim a multiple of 8.  A slot >= num_pages*bs sets
 * XY_DEV_SLOT_OOB and is skipped.
 * Errors: XY_ERR_INVALID_ARG, XY_ERR_CUDA.
 */
xy_status xy_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                       int num_tokens, void *k_pages, void *v_pages, int num_pages,
                       int num_heads_kv, int block_size, int head_dim, int32_t *err_word,
                       void *stream);

/*
 * a2 + a3 in one launch (the same two steps as xy_slot_mapping followed by xy_kv_append, fused so
 * that a step pays one kernel launch for them).  Device call: every new token t finds its slot as
 * xy_slot_mapping computes it and its K and V rows of every KV head are copied there as
 * xy_kv_append copies them; the slot is also written to slot_mapping[t] unless slot_mapping is
 * NULL.  Arguments, layouts, alignment and device error bits as for those two calls (a token
 * whose slot cannot be formed sets its bit and is skipped).  The kernel lets the next kernel on
 * the stream start at once (a programmatic dependent launch): the paged attention calls use this
 * to stream the keys older than the step's new tokens while the append still runs.
 * Errors: XY_ERR_INVALID_ARG, XY_ERR_CUDA.
 */
xy_status xy_kv_append_paged(const void *k_new, const void *v_new, const int32_t *cu_seqlens_q,
                             const int32_t *context_lens, const int32_t *block_table, int num_seqs,
                             int max_blocks, int num_tokens, void *k_pages, void *v_pages, int num_pages,
                             int num_heads_kv, int block_size, int head_dim, int64_t *slot_mapping,
                             int32_t *err_word, void *stream);

/*
 * a4 — task table: dynamic decomposer + attention task reorder ([XY] §2.2 components 1 and 2,
 * §4.4 decompose_attention / analyze_load_balance).  Host call, pure.
 * Enumerates, for sequence i -> KV head g -> query tile (q_tile tokens) -> KV chunk (kv_chunk
 * keys), one xy_task with load = q_rows * G * (kv_end - kv_start), where the tile's KV range is
 * [0, L_i) or, if causal, [0, L_i - q_i + q_start + q_rows); stable-sorts by load, largest first;
 * CTA c of the persistent launch runs tasks[c], tasks[c + num_ctas], ...  Split tiles
 * (num_splits > 1) get workspace rows in enumeration order and one xy_merge each.
 * schedule: XY_SCHEDULE_AREA follows the pages' code exactly (task i to CTA i mod num_ctas).
 * XY_SCHEDULE_SERPENTINE reads the pages' "symmetric round-robin" as a serpentine deal: the same
 * sort, then every complete odd round of num_ctas positions goes to the CTAs in reverse order, so
 * a CTA that took one of a round's largest tasks takes one of the next round's smallest (the
 * final partial round keeps the plain order, so the table stays dense).  XY_SCHEDULE_MIXED is a
 * variant for batches that mix HBM-bound decode tasks with tensor-core tiles: a task is charged
 * 128 * max(1, ceil(rows / 128)) * keys (a tile costs its padded 128-row MMA area; a task of at
 * most XY_SCHEDULE_SMALL_ROWS rows streams its KV in about the time of one such tile), sorted and
 * dealt serpentine; then each CTA interleaves its small and large tasks in proportion to their
 * charged loads, CTA c starting at phase c / num_ctas, so that at any time about the small tasks'
 * share of the CTAs streams KV from HBM while the others keep the tensor cores busy.  The per-CTA
 * load sums (stats) are those of the deal.  XY_SCHEDULE_MIXED returns XY_ERR_UNSUPPORTED when the
 * total charged load reaches 2^55 or num_ctas exceeds 65536.  XY_SCHEDULE_GREEDY charges a task
 * 128 * max(1, ceil(rows / 128)) * (keys + XY_SCHEDULE_TASK_KEYS) (its padded MMA area plus a
 * fixed per-task cost: query load, pipeline fill, output epilogue), sorts the same way and hands
 * each task to the CTA with the smallest load so far (the lowest index on ties), longest first.
 * CTAs then hold different numbers of tasks: the table keeps the layout above and the positions
 * a CTA does not use hold hole records {-1, 0, 0, 0, 0, 0, 0, -1}, which the kernels skip, so
 * *num_tasks counts the holes too (num_ctas times the longest list).  XY_SCHEDULE_DYNAMIC charges
 * tasks as XY_SCHEDULE_GREEDY does and only orders them: sorted the same way, then the tasks of a
 * (sequence, KV head) whose sequence is a chunk over a long prior context (q_len > 1 and
 * context_len - q_len >= q_len) moved up behind the first (largest) of them, keeping their order,
 * so that a chunk's query tiles run together and share its prior context in L2.  The table is
 * meant for xy_paged_attention_dynamic, whose CTAs claim tasks in table order at run time (stats
 * are the sums of positions modulo num_ctas).
 *   cu_seqlens_q [num_seqs+1], context_lens [num_seqs]: host int32.
 *   tasks [max_tasks], merges [max_merges]: host outputs; pass NULL (with max 0) to query counts.
 *   *num_tasks, *num_merges: counts; *workspace_bytes = rows * (head_dim + 1) * 4 (fp32 partial
 *   outputs followed by fp32 log-sum-exps); stats may be NULL.
 * Errors: XY_ERR_INVALID_ARG (sizes <= 0, Hq % Hkv), XY_ERR_CU_SEQLENS,
 *   XY_ERR_CONTEXT_LT_QLEN, XY_ERR_CAPACITY (non-NULL arrays too small).
 */
#define XY_SCHEDULE_AREA 0        /* the pages' reorder: load = area, sort, round-robin deal */
#define XY_SCHEDULE_SERPENTINE 1  /* the same sort, serpentine ("symmetric round-robin") deal */
#define XY_SCHEDULE_MIXED 2       /* padded-tile load, sort, serpentine deal, per-CTA interleave */
#define XY_SCHEDULE_GREEDY 3      /* padded-tile load + per-task cost, greedy deal, hole records */
#define XY_SCHEDULE_DYNAMIC 4     /* the same loads, sorted (a chunk's tasks together); claimed at run time */
#define XY_SCHEDULE_TASK_KEYS 512 /* per-task cost of XY_SCHEDULE_GREEDY, in keys */
#define XY_SCHEDULE_TILE_ROWS 128 /* MMA tile height: the unit of XY_SCHEDULE_MIXED's load */
#define XY_SCHEDULE_SMALL_ROWS 16 /* tasks of at most this many rows count as small */

/*
 * The tile policy of the kernels (no counterpart in the pages, whose 16 x 16 tiles are Ascend
 * sizes): the q_tile and kv_chunk to pass to xy_build_task_table for a batch of this shape.
 * Host call, pure.  With bf16 pages, head_dim 128 and G = Hq/Hkv dividing 128, a query tile is
 * 256/G tokens (two 128-row tcgen05 tiles sharing each K/V tile); otherwise 64/G tokens (at least
 * 1), the decode path's task height.  Over 8-bit pages (kv_fp8) every task runs on the decode
 * path: one token per task when pure_decode (one new token per sequence) and G <=
 * XY_FP8_NARROW_ROWS, else 64/G tokens.  kv_chunk is XY_DEFAULT_KV_CHUNK keys, the shape-only
 * default: a multiple of every page size and of both kernels' KV tiles, long enough that split
 * partials and merges stay few, short enough that a few long contexts still spread over the SMs;
 * xy_default_kv_chunk picks one for a batch's context lengths.
 * Errors: XY_ERR_INVALID_ARG (null outputs, Hq not a positive multiple of Hkv).
 */
#define XY_DEFAULT_KV_CHUNK 16384
#define XY_FP8_NARROW_ROWS 16
xy_status xy_default_tiles(int num_heads_q, int num_heads_kv, int head_dim, int kv_fp8, int pure_decode,
                           int *q_tile, int *kv_chunk);

/*
 * The KV chunk for one batch (no counterpart in the pages, which do not split a context): among
 * 8192, 16384, 32768 and 65536 keys, the chunk whose estimated makespan on num_ctas persistent
 * CTAs is least.  Longer chunks mean fewer tasks, partials and merges; shorter ones let a few long
 * contexts spread over more SMs.  The estimate counts each (sequence, KV head) pair's L context
 * keys in ceil(L / chunk) tasks plus a fixed per-task overhead, and takes the larger of a CTA's
 * average load and the longest-first deal of the full-size chunks; ties go to the longer chunk.
 * kv_fp8, pure_decode: as for xy_default_tiles (under the dynamic deal pure decode batches run
 * two CTAs per SM slot -- 8-bit pages with G <= 8, bf16 pages with G <= 16 -- so their chunks are
 * sized for twice num_ctas).  Host call, pure.
 *   context_lens: host int32 [num_seqs] (>= 0).  *kv_chunk receives the chunk (a multiple of
 *   every page size and of both kernels' KV tiles).
 * Errors: XY_ERR_INVALID_ARG (null output, negative length, Hq not a positive multiple of Hkv,
 * num_ctas < 1).
 */
xy_status xy_default_kv_chunk(const int32_t *context_lens, int num_seqs, int num_heads_q, int num_heads_kv,
                              int kv_fp8, int pure_decode, int num_ctas, int *kv_chunk);

xy_status xy_build_task_table(const int32_t *cu_seqlens_q, const int32_t *context_lens,
                              int num_seqs, int num_heads_q, int num_heads_kv, int head_dim,
                              int causal, int num_ctas, int q_tile, int kv_chunk, int schedule,
                              xy_task *tasks, int max_tasks, int *num_tasks,
                              xy_merge *merges, int max_merges, int *num_merges,
                              size_t *workspace_bytes, xy_task_stats *stats);

/*
 * One step's host-built metadata in one buffer (no counterpart in the pages: a runtime helper
 * for callers that re-plan every step).  Builds the block table (as xy_build_block_table) and the
 * task table (as xy_build_task_table) and packs, into the caller's host buffer `staging`
 * (ideally pinned), at offsets that are multiples of XY_STEP_TABLES_ALIGN bytes: a zero int32
 * error word, cu_seqlens_q [S+1], context_lens [S], the block table [S, max_blocks], the task
 * records and the merge records, so one host->device copy of the first `bytes` bytes gives the
 * device every table of the step (the caller passes device addresses base + offset to the device
 * calls).  *out receives the offsets, sizes, counts, workspace bytes and stats; if
 * staging_bytes < out->bytes it returns XY_ERR_CAPACITY with *out filled and nothing written.
 * Errors: those of the two builders; XY_ERR_INVALID_ARG for a null out.
 */
#define XY_STEP_TABLES_ALIGN 256

typedef struct {
    size_t err_off, cu_off, ctx_off, bt_off, tasks_off, merges_off; /* byte offsets in staging */
    size_t bytes;                                                   /* end of the merge records */
    size_t workspace_bytes;                                         /* split-KV workspace needed */
    int num_tasks, num_merges, pages_used;
    xy_task_stats stats;
} xy_step_tables;

xy_status xy_build_step_tables(const int32_t *cu_seqlens_q, const int32_t *context_lens, int num_seqs,
                               const int32_t *free_list, int num_free, int block_size, int max_blocks,
                               int num_heads_q, int num_heads_kv, int head_dim, int causal, int num_ctas,
                               int q_tile, int kv_chunk, int schedule, void *staging, size_t staging_bytes,
                               xy_step_tables *out);

/*
 * a5..a10 — paged attention ([XY] §2.2 component 3 Meta-Attention: one GEMM-softmax-GEMM
 * kernel driven by the task table, with no prefill/decode distinction; [CANN] §3.3 packed
 * paged_attention(q_packed, kv_pages, cu_seqlens, page_table, is_causal); [XY] §2.3 virtual
 * padding: only valid rows/keys are used and stored).  Device call.
 * out[t][h][:] = sum_k softmax_k(scale * q[t][h] . K_k) V_k over the keys k the token sees,
 * K/V gathered through block_table; fp32 accumulation, output rounded to bf16 (nearest even).
 *   q [num_tokens, Hq, d], k_pages/v_pages [num_pages, Hkv, bs, d], out [num_tokens, Hq, d]:
 *   bf16 device, 16-byte aligned.  cu_seqlens_q, context_lens, block_table: device int32.
 *   tasks [num_tasks], merges [num_merges]: device copies of xy_build_task_table's output for
 *   the same batch and the same num_ctas.
 *   workspace: device, >= the workspace_bytes the builder returned (may be NULL when 0).
 *   err_word: device int32 (see XY_DEV_*).
 * Launch: a programmatic dependent launch, so the kernel may start while the kernel ahead of it
 * on the stream still runs if that kernel allows it (this library's KV append kernels do).  It
 * then copies the K/V rows of each task's new tokens (keys >= context_len - q_len) only after
 * that kernel has finished; everything else it reads -- q, the tables, the older K/V rows -- it
 * may read before.  A caller's own kernel ahead of this call that lets dependents start early
 * must therefore have written those inputs before it does so.
 * Supported: head_dim 64 or 128; block_size a power of two in [16, 256]; kv_chunk (of
 * xy_build_task_table) a multiple of 128 keys.  Rows per task (q_rows * G, G = Hq/Hkv): up to 256
 * when head_dim is 128 and G divides 128 (tasks with more than 16 rows then run on tcgen05 tensor
 * cores as two 128-row tiles), otherwise up to 64.  Tasks outside these limits set XY_DEV_BAD_TASK.
 * Errors: XY_ERR_INVALID_ARG, XY_ERR_UNSUPPORTED, XY_ERR_WORKSPACE, XY_ERR_CUDA.
 */
xy_status xy_paged_attention(const void *q, const int32_t *cu_seqlens_q,
                             const int32_t *context_lens, const int32_t *block_table,
                             int max_blocks, const void *k_pages, const void *v_pages,
                             int num_pages, int num_seqs, int num_tokens, int num_heads_q,
                             int num_heads_kv, int head_dim, int block_size, float scale,
                             int causal, const xy_task *tasks, int num_tasks,
                             const xy_merge *merges, int num_merges, int num_ctas,
                             void *workspace, size_t workspace_bytes, int32_t *err_word,
                             void *out, void *stream);

/*
 * Paged attention that allocates nothing (no counterpart in the pages: it is a convenience for
 * callers of this library).
 *
 * Some callers cannot allocate device memory where they run a step: a serving process that
 * hands all free HBM to the KV page pool at start-up, so a per-step cudaMalloc of the split-KV
 * workspace would fail, or an engine whose device memory belongs to an allocator that this
 * library cannot call.  This entry point does what xy_paged_attention does, but takes its
 * split-KV scratch from a fixed array inside libxy (XY_NOALLOC_SCRATCH_BYTES bytes of device
 * memory, which every GPU that loads the library holds until the process exits) instead of a
 * caller buffer.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *   workspace_bytes: the bytes xy_build_task_table reported for this batch; a value above
 *   XY_NOALLOC_SCRATCH_BYTES returns XY_ERR_WORKSPACE before anything is launched.
 *   All other arguments, layouts and errors are those of xy_paged_attention.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  Every call on a device
 * shares the one array and it keeps the last call's contents (nothing in it has to start at
 * zero), so calls that overlap on the GPU -- on different streams, or from different host
 * threads -- race on it and must be serialised by the caller.
 */
#define XY_NOALLOC_SCRATCH_BYTES (32u << 20)

xy_status xy_paged_attention_noalloc(const void *q, const int32_t *cu_seqlens_q,
                                     const int32_t *context_lens, const int32_t *block_table,
                                     int max_blocks, const void *k_pages, const void *v_pages,
                                     int num_pages, int num_seqs, int num_tokens, int num_heads_q,
                                     int num_heads_kv, int head_dim, int block_size, float scale,
                                     int causal, const xy_task *tasks, int num_tasks,
                                     const xy_merge *merges, int num_merges, int num_ctas,
                                     size_t workspace_bytes, int32_t *err_word, void *out,
                                     void *stream);

/*
 * Paged attention with a dynamic deal (a variant of the reorder's static deal, [XY] §2.2
 * component 2: the pages deal sorted tasks to cores before the launch; here the cores take them
 * while the kernel runs).
 *
 * The kernels xy_paged_attention launches for the batch (the unified tcgen05 kernel, or the
 * decode-path kernel for pure decode batches and shapes the tile kernel does not take) run every
 * task, but instead of walking a fixed share of the table, each persistent CTA claims the next
 * unclaimed task with an atomic add on task_counter[0].  In the unified kernel a scheduler warp
 * claims the CTA's next task once the current one has at most 512 keys left to issue; in the
 * decode-path kernel when the CTA starts its current task.  CTAs thus take tasks in table order
 * (largest first for XY_SCHEDULE_DYNAMIC tables, a chunk's tasks together), and a CTA that drew
 * short tasks takes more of them.  A pure decode batch (num_tokens == num_seqs, G <= 16) runs as 2 * num_ctas half-size
 * decode-path CTAs (two per SM: two stages and two producer warps each, the first of which
 * claims the tasks), since the dynamic deal does not depend on the grid size; such a batch's
 * tables have tasks of at most 16 rows (q_rows = 1), and a hand-made table with taller tasks sets
 * XY_DEV_BAD_TASK and leaves their rows unwritten.  A task's result does not depend on which CTA
 * runs it: outputs are bit-identical to xy_paged_attention's on the same tasks.
 *   task_counter: device int32[2], 8-byte aligned, owned by the caller, zero before the first
 *   call (e.g. zeroed at allocation).  Word 0 counts claims, word 1 the CTAs done claiming; the
 *   last CTA to finish claiming returns both to zero, so every launch leaves the counter ready for
 *   the next one, with no reset on the host or the stream.  Calls that overlap on the GPU need
 *   different counters.
 *   tasks: any table of xy_build_task_table for this batch (XY_SCHEDULE_DYNAMIC: ordered as
 *   described there, no holes; hole records of other schedules are skipped).
 *   All other arguments, layouts, limits and errors are those of xy_paged_attention;
 *   XY_ERR_INVALID_ARG also for a null or misaligned task_counter.  A launch whose waits gave up
 *   (XY_DEV_TIMEOUT) still returns the counter to zero.
 */
xy_status xy_paged_attention_dynamic(const void *q, const int32_t *cu_seqlens_q,
                                     const int32_t *context_lens, const int32_t *block_table,
                                     int max_blocks, const void *k_pages, const void *v_pages,
                                     int num_pages, int num_seqs, int num_tokens, int num_heads_q,
                                     int num_heads_kv, int head_dim, int block_size, float scale,
                                     int causal, const xy_task *tasks, int num_tasks,
                                     const xy_merge *merges, int num_merges, int num_ctas,
                                     void *workspace, size_t workspace_bytes,
                                     int32_t *task_counter, int32_t *err_word, void *out,
                                     void *stream);

/*
 * Paged attention with a per-CTA trace, to measure how evenly a deal spreads the work ([XY] §2.2
 * component 2 reports the balance ratio = min/max core load; the trace gives the time each CTA
 * was busy, so the ratio and the tail -- the time the last CTA runs after the others are done --
 * can be measured for the static and the dynamic deal alike).  No counterpart in the pages beyond
 * that ratio.
 *   task_counter: NULL runs what xy_paged_attention runs (the static deal: CTA c takes positions
 *   c, c + num_ctas, ... of the table, on the unified tcgen05 kernel or the decode-path kernel);
 *   a counter runs what xy_paged_attention_dynamic runs (the dynamic deal), except that a pure
 *   decode batch keeps one decode-path CTA per SM slot (one trace record each).
 *   cta_trace: device uint64 [num_ctas][4], 8-byte aligned: {start ns, end ns, tasks run, sum of
 *   q_rows * G * (kv_end - kv_start) over them}; times from the GPU's global timer (ns), start
 *   when the CTA begins, end when its last task is stored.  A CTA whose waits gave up
 *   (XY_DEV_TIMEOUT) leaves its end, tasks and work unwritten: zero the buffer first.
 *   All other arguments, limits and errors are those of the call it stands for.  The split-KV
 *   merge that follows is not traced.
 */
xy_status xy_paged_attention_traced(const void *q, const int32_t *cu_seqlens_q,
                                    const int32_t *context_lens, const int32_t *block_table,
                                    int max_blocks, const void *k_pages, const void *v_pages,
                                    int num_pages, int num_seqs, int num_tokens, int num_heads_q,
                                    int num_heads_kv, int head_dim, int block_size, float scale,
                                    int causal, const xy_task *tasks, int num_tasks,
                                    const xy_merge *merges, int num_merges, int num_ctas,
                                    void *workspace, size_t workspace_bytes,
                                    int32_t *task_counter, uint64_t *cta_trace, int32_t *err_word,
                                    void *out, void *stream);

/* 8-bit KV pages (a variant of the pool; [CANN] §5.2 keeps scale metadata beside the pages).
 * k_pages/v_pages: uint8 [P, Hkv, bs, d] of OCP E4M3 codes ("E4M3FN": bias 7, max 448, no
 * infinities); k_scales/v_scales: fp32 [P, Hkv, bs], one scale per stored (token, KV head) row;
 * the row's values are code * scale.  Appending a row quantizes it with s = max|x| / 448 (1 for an
 * all-zero row) and codes = E4M3(x / s) rounded to nearest even and saturated to +-448, both
 * IEEE fp32 operations, so rows already in a page are never rescaled.
 *
 * xy_kv_append_fp8: the append of xy_kv_append for 8-bit pages.  k_new/v_new [T, Hkv, d] bf16
 * (16-byte aligned), slot_mapping [T] int64 (negative = skip), d in {64, 128}, bs a power of two
 * >= 16.  A slot outside [0, P*bs) sets XY_DEV_SLOT_OOB and is skipped.  Device pointers,
 * asynchronous on `stream`; XY_ERR_UNSUPPORTED for other head dims. */
xy_status xy_kv_append_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping, int num_tokens,
                           void *k_pages, void *v_pages, float *k_scales, float *v_scales, int num_pages,
                           int num_heads_kv, int block_size, int head_dim, int32_t *err_word, void *stream);

/* xy_kv_append_paged_fp8: the slot mapping and xy_kv_append_fp8 in one launch, as
 * xy_kv_append_paged is for bf16 pages: each new token's slot is formed from cu_seqlens_q,
 * context_lens and block_table (device int32, as for xy_slot_mapping), written to slot_mapping[t]
 * unless slot_mapping is NULL, and the token's K and V rows are quantized into it.  Every other
 * argument, limit and error as for xy_kv_append_fp8 and xy_slot_mapping. */
xy_status xy_kv_append_paged_fp8(const void *k_new, const void *v_new, const int32_t *cu_seqlens_q,
                                 const int32_t *context_lens, const int32_t *block_table, int num_seqs,
                                 int max_blocks, int num_tokens, void *k_pages, void *v_pages, float *k_scales,
                                 float *v_scales, int num_pages, int num_heads_kv, int block_size, int head_dim,
                                 int64_t *slot_mapping, int32_t *err_word, void *stream);

/* xy_dequant_pages_fp8: bf16 copies of listed 8-bit pages (a helper of the tensor-core path for
 * prefill and chunk tasks over 8-bit pages, which runs on dequantized copies of the pages those
 * sequences read).  Output page i of k_out / v_out (bf16 [num_out, Hkv, bs, d], device, 16-byte
 * aligned) holds source page pages[i] (device int32 [num_out]): element = bf16(fp32(E4M3 value *
 * row scale)), the product an IEEE fp32 multiply, both roundings to nearest even.  A source page
 * outside [0, num_pages) sets XY_DEV_PAGE_OOB and its output page is left unwritten.  Asynchronous
 * on `stream`; XY_ERR_UNSUPPORTED for d other than 64 and 128. */
xy_status xy_dequant_pages_fp8(const void *k_codes, const void *v_codes, const float *k_scales, const float *v_scales,
                               int num_pages, int num_heads_kv, int block_size, int head_dim, const int32_t *pages,
                               int num_out, void *k_out, void *v_out, int32_t *err_word, void *stream);

/* xy_paged_attention_fp8: xy_paged_attention over 8-bit pages.  The result is the attention of
 * xy_paged_attention over the dequantized pages (code * scale per row): K scales multiply the fp32
 * scores, V scales the softmax weights, the codes become f16 exactly on chip.  q, out, tasks,
 * merges, workspace, err_word and every other argument as for xy_paged_attention; k_pages/v_pages
 * uint8 [num_pages, Hkv, bs, 128] and k_scales/v_scales fp32 [num_pages, Hkv, bs] (device,
 * 16-byte aligned), written by xy_kv_append_fp8.  The query rows are rounded to f16 on chip
 * (exact for bf16 values of magnitude 2^-14 .. 65504).  Every task runs on the decode path: in a
 * pure decode batch (num_tokens == num_seqs) with G <= XY_FP8_NARROW_ROWS a task has at most
 * XY_FP8_NARROW_ROWS rows (q_rows = 1), otherwise at most 64 rows (q_tile <= 64 / G).  Tasks
 * outside these limits set XY_DEV_BAD_TASK.  Layout hint (results are the same either way): when
 * v_pages lies after the whole K pool in the same address space (for example both pools as halves
 * of one allocation, V second) at a distance that is a multiple of 16 bytes, one copy brings a
 * page's K and V codes, which helps small pages (16-token pages: 12 instead of 20 copies per
 * 128-key stage); otherwise each page takes a copy per pool.
 * Errors: as xy_paged_attention; XY_ERR_UNSUPPORTED for head_dim other than 128 or G > 64. */
xy_status xy_paged_attention_fp8(const void *q, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                 const int32_t *block_table, int max_blocks, const void *k_pages,
                                 const void *v_pages, const float *k_scales, const float *v_scales,
                                 int num_pages, int num_seqs, int num_tokens, int num_heads_q,
                                 int num_heads_kv, int head_dim, int block_size, float scale, int causal,
                                 const xy_task *tasks, int num_tasks, const xy_merge *merges,
                                 int num_merges, int num_ctas, void *workspace, size_t workspace_bytes,
                                 int32_t *err_word, void *out, void *stream);

/* xy_paged_attention_fp8_dynamic: xy_paged_attention_fp8 with the dynamic deal of
 * xy_paged_attention_dynamic ([XY] §2.2 component 2, the deal taken at run time).  Each CTA's
 * first producer warp claims the next task from task_counter[0] once it has issued the first
 * copy of its current task (no separate scheduler warp over 8-bit pages), so CTAs take tasks in
 * table order.  Outputs are bit-identical to xy_paged_attention_fp8's on the same tasks.  A pure
 * decode batch (num_tokens == num_seqs) with G <= 8 runs as 2 * num_ctas half-size CTAs (two per
 * SM: two stages and two producer warps each), since the dynamic deal does not depend on the grid
 * size; other batches run num_ctas CTAs.  Those half-size CTAs take tasks of at most 8 rows
 * (q_rows * G <= 8), which every table built for such a batch has (each sequence has one new
 * token, so q_rows = 1); a hand-made table with taller tasks sets XY_DEV_BAD_TASK and leaves their
 * rows unwritten.
 *   task_counter: as for xy_paged_attention_dynamic (device int32[2], 8-byte aligned, zero before
 *   the first call, returned to zero by every launch; overlapping calls need different counters).
 *   Every other argument, limit and error as for xy_paged_attention_fp8; XY_ERR_INVALID_ARG also
 *   for a null or misaligned task_counter. */
xy_status xy_paged_attention_fp8_dynamic(const void *q, const int32_t *cu_seqlens_q,
                                         const int32_t *context_lens, const int32_t *block_table,
                                         int max_blocks, const void *k_pages, const void *v_pages,
                                         const float *k_scales, const float *v_scales, int num_pages,
                                         int num_seqs, int num_tokens, int num_heads_q, int num_heads_kv,
                                         int head_dim, int block_size, float scale, int causal,
                                         const xy_task *tasks, int num_tasks, const xy_merge *merges,
                                         int num_merges, int num_ctas, void *workspace,
                                         size_t workspace_bytes, int32_t *task_counter, int32_t *err_word,
                                         void *out, void *stream);

/*
 * One step over 8-bit pages for a batch that mixes one-token (decode) sequences with sequences of
 * several new tokens (prefill, chunks, verify) -- the pages' unified batch ([XY] §2.2 component
 * 3: no prefill/decode distinction at the scheduler) with [CANN] §5.2's scale metadata beside the
 * pages.  The decode sequences run on the 8-bit decode path; the others run on the tcgen05 tile
 * path over bf16 copies of the pages they read (xy_dequant_pages_fp8), since the tensor cores take
 * no E4M3 x f16 product.  The two kinds must each form one contiguous range of sequences.
 *
 * xy_build_fp8_step_tables: host call, pure.  Splits the batch into its tile range and decode
 * range, builds the block table (as xy_build_block_table), the list of physical pages the tile
 * sequences read (in their order; bf16 copy i holds page list[i]), the tile sequences' block
 * table over those copies (row r: copies 0, 1, ... of tile sequence r, the rest -1), each part's
 * cu_seqlens_q renumbered from 0, and each part's task and merge tables (XY_SCHEDULE_DYNAMIC, the
 * xy_default_tiles policy: bf16 tiles for the tile part, 8-bit decode tasks for the other, each
 * part's KV chunk from xy_default_kv_chunk over that part's sequences), and
 * packs them into `staging` at the offsets of *out (multiples of XY_STEP_TABLES_ALIGN) after a
 * zero error word, cu_seqlens_q, context_lens and the block table, so one host->device copy of
 * out->bytes bytes carries every table.  *out also gets the parts' sequence and token ranges,
 * counts and workspace sizes.  staging_bytes < out->bytes: XY_ERR_CAPACITY with *out filled.
 * Errors: XY_ERR_INVALID_ARG, XY_ERR_CU_SEQLENS, XY_ERR_CONTEXT_LT_QLEN, XY_ERR_OUT_OF_PAGES,
 *   XY_ERR_CAPACITY (as the builders it composes); XY_ERR_UNSUPPORTED when the kinds interleave,
 *   head_dim is not 128 or G does not divide 128.
 */
typedef struct {
    size_t err_off, cu_off, ctx_off, bt_off;                                       /* whole batch */
    size_t tile_cu_off, tile_bt_off, tile_pages_off, tile_tasks_off, tile_merges_off; /* tile part */
    size_t dec_cu_off, dec_tasks_off, dec_merges_off;                              /* decode part */
    size_t bytes;                          /* end of the last table */
    size_t tile_workspace_bytes, dec_workspace_bytes;
    int tile_seq_begin, tile_seq_end, dec_seq_begin, dec_seq_end;   /* sequence ranges [begin, end) */
    int tile_tok_begin, tile_tok_end, dec_tok_begin, dec_tok_end;   /* packed token ranges */
    int tile_num_pages;                    /* pages the tile part copies to bf16 */
    int tile_num_tasks, tile_num_merges, dec_num_tasks, dec_num_merges;
    int pages_used;
} xy_fp8_step_tables;

xy_status xy_build_fp8_step_tables(const int32_t *cu_seqlens_q, const int32_t *context_lens, int num_seqs,
                                   const int32_t *free_list, int num_free, int block_size, int max_blocks,
                                   int num_heads_q, int num_heads_kv, int head_dim, int causal, int num_ctas,
                                   void *staging, size_t staging_bytes, xy_fp8_step_tables *out);

/*
 * xy_paged_attention_fp8_mixed: the attention of such a step, after the append of the step's new
 * tokens (xy_kv_append_paged_fp8 over the whole batch).  Device call: the bf16 copies of the tile
 * part's pages, its tcgen05 attention (dynamic deal) and merges, then the decode part's 8-bit
 * attention (dynamic deal) and merges, each writing its own rows of out.
 *   tables: device copy of the first t->bytes bytes of the staging buffer t describes (16-byte
 *   aligned); t: the host description xy_build_fp8_step_tables filled.
 *   copy_k, copy_v: device bf16 buffers of copy_pages pages of [Hkv, bs, d] each (caller owned,
 *   copy_pages >= t->tile_num_pages), scratch of the page copies.
 *   tile_ws / dec_ws: split-KV workspaces of at least t->tile_workspace_bytes /
 *   t->dec_workspace_bytes (NULL when 0).  task_counters: device int32[4], 8-byte aligned, zero
 *   before the first call (the two parts' claim counters, words 0-1 and 2-3, each returned to zero
 *   by its launch; overlapping calls need different counters).
 *   q/out [num_tokens, Hq, d], the 8-bit pools and their scales, err_word: as for
 *   xy_paged_attention_fp8; num_seqs, num_tokens, max_blocks, the head counts, head_dim and
 *   block_size as passed to the builder.
 * Errors: XY_ERR_INVALID_ARG (null or misaligned pointers, a description that does not fit the
 *   sizes), XY_ERR_WORKSPACE (copy or workspace buffers too small), XY_ERR_UNSUPPORTED, XY_ERR_CUDA.
 */
xy_status xy_paged_attention_fp8_mixed(const void *q, const void *tables, const xy_fp8_step_tables *t,
                                       const void *k_pages, const void *v_pages, const float *k_scales,
                                       const float *v_scales, int num_pages, int num_seqs, int num_tokens,
                                       int max_blocks, int num_heads_q, int num_heads_kv, int head_dim,
                                       int block_size, float scale, int causal, int num_ctas, void *copy_k,
                                       void *copy_v, int copy_pages, void *tile_ws, size_t tile_ws_bytes,
                                       void *dec_ws, size_t dec_ws_bytes, int32_t *task_counters,
                                       int32_t *err_word, void *out, void *stream);

/* Self-test of the bounded waits (no counterpart in the pages; not a step of the path).
 * Every mbarrier wait in the attention kernels gives up after a time limit, or when its CTA's
 * abort flag is raised, sets XY_DEV_TIMEOUT in *err_word and lets the kernel return instead of
 * hanging the GPU.  This launches one CTA whose first warp waits on a barrier nobody arrives at
 * with a limit of limit_us microseconds (1 .. 10^7), then raises the abort flag that releases the
 * second warp's wait (which has the kernels' own 2 s limit).  result (device, 3 int32, caller
 * owned): [0] 1 if the first wait succeeded (it must not), [1] microseconds it waited, [2] 1 if
 * the second wait succeeded (it must not).  *err_word (device) gets XY_DEV_TIMEOUT.  Asynchronous
 * on `stream`; XY_ERR_INVALID_ARG for null pointers or a limit out of range. */
xy_status xy_selftest_bounded_wait(uint32_t limit_us, int32_t *err_word, int32_t *result, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* XY_H */
