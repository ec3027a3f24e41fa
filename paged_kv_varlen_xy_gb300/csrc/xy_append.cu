// a2 slot mapping and a3 KV append: the new tokens' K/V rows go into their page slots.
//
// cann-recipes-infer Paged KV Cache / Packed Sequence notes (dpshk.com/news/5336026) §2.2 (pages
// are taken on demand and a sequence grows into them), §3.1 (page layout [heads, page_size,
// head_dim]); ATB notes (ai6s.net/6a38a2a6662f9a54cb828d66) "KV缓存复用" (chunked prefill appends
// to the existing cache).  Both kernels are HBM-bound copies: 16-byte vector loads and stores,
// consecutive threads on consecutive bytes of a row.

#include <cuda_runtime.h>
#include <stdint.h>

#include "xy.h"
#include "xy_device.cuh"

namespace {

// One thread per new token.  Token t of sequence i (found by binary search in cu_seqlens_q) is
// at absolute position p = L_i - q_i + j and goes to block_table[i][p / bs] * bs + p % bs.
__global__ void slot_mapping_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ ctx,
                                    const int32_t *__restrict__ bt, int S, int MB, int T, int bs,
                                    int P, int64_t *__restrict__ slots, int32_t *err) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    int lo = 0, hi = S - 1;  // largest i with cu[i] <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int i = lo;
    const int64_t q = (int64_t)cu[i + 1] - cu[i];
    const int64_t p = (int64_t)ctx[i] - q + (t - cu[i]);
    int64_t slot = -1;
    if (p < 0 || t >= cu[i + 1]) {
        xy::set_err(err, XY_DEV_BAD_TASK);
    } else {
        const int64_t lb = p / bs;
        const int32_t page = lb < MB ? bt[(int64_t)i * MB + lb] : -1;
        if (page < 0 || page >= P) xy::set_err(err, XY_DEV_PAGE_OOB);
        else slot = (int64_t)page * bs + p % bs;
    }
    slots[t] = slot;
}

// Grid-stride over 16-byte vectors of the new rows: vector v is chunk c of head h of token t.
__global__ void kv_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                 const int64_t *__restrict__ slots, int T, int H, int bs, int vec_per_row,
                                 int64_t pool_slots, uint4 *__restrict__ k_pages, uint4 *__restrict__ v_pages,
                                 int32_t *err) {
    xy::grid_dep_launch();
    const int64_t total = (int64_t)T * H * vec_per_row;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = v / vec_per_row;  // (t, h)
        const int c = (int)(v - row * vec_per_row);
        const int64_t t = row / H;
        const int h = (int)(row - t * H);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            if (h == 0 && c == 0) xy::set_err(err, XY_DEV_SLOT_OOB);
            continue;
        }
        const int64_t page = slot / bs, off = slot - page * bs;
        const int64_t dst = ((page * H + h) * bs + off) * vec_per_row + c;
        k_pages[dst] = __ldg(k_new + v);
        v_pages[dst] = __ldg(v_new + v);
    }
}

// The same copy when the page size and the 16-byte vectors per row are powers of two and there
// are fewer than 2^31 (token, head) rows: shifts instead of 64-bit divisions (which bound the
// general kernel), one 32-bit division per vector for the token.
template <int VSH>
__global__ void kv_append_pow2_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                      const int64_t *__restrict__ slots, int T, int H, int bs_sh,
                                      int64_t pool_slots, uint4 *__restrict__ k_pages, uint4 *__restrict__ v_pages,
                                      int32_t *err) {
    xy::grid_dep_launch();
    const int64_t total = ((int64_t)T * H) << VSH;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total;
         v += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t row = (uint32_t)(v >> VSH);  // (t, h)
        const int c = (int)(v & ((1 << VSH) - 1));
        const uint32_t t = row / (uint32_t)H;
        const int h = (int)(row - t * (uint32_t)H);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            if (h == 0 && c == 0) xy::set_err(err, XY_DEV_SLOT_OOB);
            continue;
        }
        const int64_t page = slot >> bs_sh, off = slot & ((int64_t(1) << bs_sh) - 1);
        const int64_t dst = ((((page * H + h) << bs_sh) + off) << VSH) + c;
        k_pages[dst] = __ldg(k_new + v);
        v_pages[dst] = __ldg(v_new + v);
    }
}

// a2 and a3 in one launch: one CTA per new token (grid-stride), whose first warp finds the
// token's slot (xy::warp_token_slot) and publishes it in shared memory; then the CTA copies the
// token's K and V rows of every KV head as 16-byte vectors, consecutive threads on consecutive
// vectors of the token's contiguous [Hkv, d] block.  slots_out (may be null) receives the slot.
__global__ void __launch_bounds__(128) kv_append_paged_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new, const int32_t *__restrict__ cu,
    const int32_t *__restrict__ ctx, const int32_t *__restrict__ bt, int S, int MB, int T, int H, int bs, int P,
    int vec_per_row, int64_t *__restrict__ slots_out, uint4 *__restrict__ k_pages, uint4 *__restrict__ v_pages,
    int32_t *err) {
    __shared__ int64_t s_slot;
    xy::grid_dep_launch();  // the attention kernel after this one may start its prologue
    const int nvec = H * vec_per_row;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (threadIdx.x < 32) {
            const int64_t slot = xy::warp_token_slot(cu, ctx, bt, S, MB, bs, P, t, threadIdx.x, err);
            if (threadIdx.x == 0) {
                s_slot = slot;
                if (slots_out) slots_out[t] = slot;
            }
        }
        __syncthreads();
        const int64_t slot = s_slot;
        __syncthreads();  // s_slot is rewritten for the next token only after every thread read it
        if (slot < 0) continue;
        const int64_t page = slot / bs, off = slot - page * bs;
        const int64_t src0 = (int64_t)t * nvec;
        for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
            const int h = v / vec_per_row, c = v - h * vec_per_row;
            const int64_t dst = ((page * H + h) * bs + off) * vec_per_row + c;
            const uint4 kv = __ldg(k_new + src0 + v), vv = __ldg(v_new + src0 + v);
            k_pages[dst] = kv;
            v_pages[dst] = vv;
        }
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace

extern "C" xy_status xy_slot_mapping(const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                     const int32_t *block_table, int num_seqs, int max_blocks,
                                     int num_tokens, int block_size, int num_pages, int64_t *slot_mapping,
                                     int32_t *err_word, void *stream) {
    if (num_tokens < 0 || num_seqs < 0 || max_blocks < 1 || block_size < 1 || num_pages < 1)
        return XY_ERR_INVALID_ARG;
    if (num_tokens == 0) return XY_OK;
    if (num_seqs < 1 || !cu_seqlens_q || !context_lens || !block_table || !slot_mapping)
        return XY_ERR_INVALID_ARG;
    const int threads = 256;
    const int blocks = (num_tokens + threads - 1) / threads;
    slot_mapping_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        cu_seqlens_q, context_lens, block_table, num_seqs, max_blocks, num_tokens, block_size, num_pages,
        slot_mapping, err_word);
    return cudaGetLastError() == cudaSuccess ? XY_OK : XY_ERR_CUDA;
}

extern "C" xy_status xy_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                  int num_tokens, void *k_pages, void *v_pages, int num_pages,
                                  int num_heads_kv, int block_size, int head_dim, int32_t *err_word,
                                  void *stream) {
    if (num_tokens < 0 || num_pages < 1 || num_heads_kv < 1 || block_size < 1 || head_dim < 8 ||
        head_dim % 8)
        return XY_ERR_INVALID_ARG;
    if (num_tokens == 0) return XY_OK;
    if (!k_new || !v_new || !slot_mapping || !k_pages || !v_pages) return XY_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
        return XY_ERR_INVALID_ARG;
    const int vec_per_row = head_dim / 8;
    const int64_t total = (int64_t)num_tokens * num_heads_kv * vec_per_row;
    const int threads = 256;
    int sms = device_sm_count();
    if (sms <= 0) return XY_ERR_CUDA;
    const int64_t want = (total + threads - 1) / threads;
    const int blocks = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    const bool pow2 = (block_size & (block_size - 1)) == 0 && (vec_per_row == 8 || vec_per_row == 16) &&
                      (int64_t)num_tokens * num_heads_kv < (int64_t(1) << 31);
    if (pow2) {
        int bs_sh = 0;
        while ((1 << bs_sh) < block_size) ++bs_sh;
        const int64_t pool_slots = (int64_t)num_pages * block_size;
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        auto *kn = static_cast<const uint4 *>(k_new);
        auto *vn = static_cast<const uint4 *>(v_new);
        auto *kp = static_cast<uint4 *>(k_pages);
        auto *vp = static_cast<uint4 *>(v_pages);
        if (vec_per_row == 16)
            kv_append_pow2_kernel<4><<<blocks, threads, 0, st>>>(kn, vn, slot_mapping, num_tokens, num_heads_kv,
                                                                 bs_sh, pool_slots, kp, vp, err_word);
        else
            kv_append_pow2_kernel<3><<<blocks, threads, 0, st>>>(kn, vn, slot_mapping, num_tokens, num_heads_kv,
                                                                 bs_sh, pool_slots, kp, vp, err_word);
        return cudaGetLastError() == cudaSuccess ? XY_OK : XY_ERR_CUDA;
    }
    kv_append_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping, num_tokens,
        num_heads_kv, block_size, vec_per_row, (int64_t)num_pages * block_size, static_cast<uint4 *>(k_pages),
        static_cast<uint4 *>(v_pages), err_word);
    return cudaGetLastError() == cudaSuccess ? XY_OK : XY_ERR_CUDA;
}

extern "C" xy_status xy_kv_append_paged(const void *k_new, const void *v_new, const int32_t *cu_seqlens_q,
                                        const int32_t *context_lens, const int32_t *block_table, int num_seqs,
                                        int max_blocks, int num_tokens, void *k_pages, void *v_pages, int num_pages,
                                        int num_heads_kv, int block_size, int head_dim, int64_t *slot_mapping,
                                        int32_t *err_word, void *stream) {
    if (num_tokens < 0 || num_seqs < 0 || max_blocks < 1 || num_pages < 1 || num_heads_kv < 1 || block_size < 1 ||
        head_dim < 8 || head_dim % 8)
        return XY_ERR_INVALID_ARG;
    if (num_tokens == 0) return XY_OK;
    if (num_seqs < 1 || !cu_seqlens_q || !context_lens || !block_table || !k_new || !v_new || !k_pages || !v_pages)
        return XY_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
        return XY_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return XY_ERR_CUDA;
    const int blocks = num_tokens < sms * 16 ? num_tokens : sms * 16;
    kv_append_paged_kernel<<<blocks, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), cu_seqlens_q, context_lens,
        block_table, num_seqs, max_blocks, num_tokens, num_heads_kv, block_size, num_pages, head_dim / 8,
        slot_mapping, static_cast<uint4 *>(k_pages), static_cast<uint4 *>(v_pages), err_word);
    return cudaGetLastError() == cudaSuccess ? XY_OK : XY_ERR_CUDA;
}
