// 8-bit KV pages: the append that quantizes new K/V rows into E4M3 pages with one fp32 scale per
// (token, KV head) row.
//
// cann-recipes-infer Paged KV Cache notes (dpshk.com/news/5336026) §5.2: scale metadata kept
// beside the pages so values can be stored narrower than they are computed in.  Here every stored
// row has its own scale s = max|x| / 448 (1 for an all-zero row) and its elements are the E4M3
// codes of x / s (round to nearest even, saturating at +-448), so appending a token never rescales
// rows already in a page.  The scale and the division are IEEE fp32 operations.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "xy.h"
#include "xy_device.cuh"

namespace {

// Two fp32 values -> two E4M3 codes in memory order (lo first).
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Quantize one bf16 row of D values (src) into E4M3 codes at dst and its scale at *scale; executed
// by one whole warp, D / 32 consecutive values per lane.
template <int D>
__device__ __forceinline__ void quantize_row(const __nv_bfloat16 *__restrict__ src, uint8_t *__restrict__ dst,
                                             float *__restrict__ scale, int lane) {
    constexpr int E = D / 32;  // elements per lane
    float x[E];
#pragma unroll
    for (int i = 0; i < E; i += 2) {
        const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162 *>(src + lane * E + i);
        x[i] = __low2float(pr);
        x[i + 1] = __high2float(pr);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint16_t code[E / 2];
#pragma unroll
    for (int i = 0; i < E; i += 2) code[i / 2] = e4m3x2(__fdiv_rn(x[i], s), __fdiv_rn(x[i + 1], s));
    if (E == 4)
        *reinterpret_cast<uint32_t *>(dst + lane * E) = (uint32_t)code[0] | ((uint32_t)code[E / 2 - 1] << 16);
    else
        *reinterpret_cast<uint16_t *>(dst + lane * E) = code[0];
    if (lane == 0) *scale = s;
}

// One warp per (token, KV head) row of K and of V; D = head_dim (64 or 128).
template <int D>
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(const __nv_bfloat16 *__restrict__ k_new,
                                                             const __nv_bfloat16 *__restrict__ v_new,
                                                             const int64_t *__restrict__ slots, int T, int H, int bs,
                                                             int64_t pool_slots, uint8_t *__restrict__ k_pages,
                                                             uint8_t *__restrict__ v_pages, float *__restrict__ k_scales,
                                                             float *__restrict__ v_scales, int32_t *err) {
    xy::grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < 2 * (int64_t)T * H;
         row += warps) {
        const int tensor = (int)(row / ((int64_t)T * H));  // 0: K, 1: V
        const int64_t th = row - tensor * (int64_t)T * H;
        const int64_t t = th / H;
        const int h = (int)(th - t * H);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            if (lane == 0 && tensor == 0 && h == 0) xy::set_err(err, XY_DEV_SLOT_OOB);
            continue;
        }
        const int64_t page = slot / bs, off = slot - page * bs;
        const int64_t drow = (page * H + h) * bs + off;
        quantize_row<D>((tensor ? v_new : k_new) + th * D, (tensor ? v_pages : k_pages) + drow * D,
                        (tensor ? v_scales : k_scales) + drow, lane);
    }
}

// The slot mapping and the quantizing append in one launch: one CTA per new token (grid-stride),
// whose first warp finds the token's slot (xy::warp_token_slot); then its eight warps quantize the
// token's 2 * H rows (K and V of every KV head).  slots_out (may be null) receives the slot.
template <int D>
__global__ void __launch_bounds__(256) kv_append_paged_fp8_kernel(
    const __nv_bfloat16 *__restrict__ k_new, const __nv_bfloat16 *__restrict__ v_new,
    const int32_t *__restrict__ cu, const int32_t *__restrict__ ctx, const int32_t *__restrict__ bt, int S, int MB,
    int T, int H, int bs, int P, int64_t *__restrict__ slots_out, uint8_t *__restrict__ k_pages,
    uint8_t *__restrict__ v_pages, float *__restrict__ k_scales, float *__restrict__ v_scales, int32_t *err) {
    __shared__ int64_t s_slot;
    xy::grid_dep_launch();  // the attention kernel after this one may start its prologue
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (warp == 0) {
            const int64_t slot = xy::warp_token_slot(cu, ctx, bt, S, MB, bs, P, t, lane, err);
            if (lane == 0) {
                s_slot = slot;
                if (slots_out) slots_out[t] = slot;
            }
        }
        __syncthreads();
        const int64_t slot = s_slot;
        __syncthreads();  // s_slot is rewritten for the next token only after every thread read it
        if (slot < 0) continue;
        const int64_t page = slot / bs, off = slot - page * bs;
        for (int r = warp; r < 2 * H; r += nwarps) {
            const int tensor = r / H, h = r - tensor * H;
            const int64_t drow = (page * H + h) * bs + off;
            quantize_row<D>((tensor ? v_new : k_new) + ((int64_t)t * H + h) * D,
                            (tensor ? v_pages : k_pages) + drow * D, (tensor ? v_scales : k_scales) + drow, lane);
        }
    }
}

// Dequantized copies of listed pages: out page i = bf16(fp32(code value * scale)) of source page
// pages[i], both tensors; one thread per 8 codes of a row (D = 64 or 128).
template <int D>
__global__ void __launch_bounds__(256) dequant_pages_kernel(const uint8_t *__restrict__ k_codes,
                                                             const uint8_t *__restrict__ v_codes,
                                                             const float *__restrict__ k_scales,
                                                             const float *__restrict__ v_scales,
                                                             const int32_t *__restrict__ pages, int num_out, int H,
                                                             int bs, int num_pages, __nv_bfloat16 *__restrict__ k_out,
                                                             __nv_bfloat16 *__restrict__ v_out, int32_t *err) {
    constexpr int C = D / 8;  // 8-code groups per row
    const int64_t rows_per_tensor = (int64_t)num_out * H * bs;
    const int64_t total = 2 * rows_per_tensor * C;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (int64_t)gridDim.x * blockDim.x) {
        const int tensor = (int)(g / (rows_per_tensor * C));
        const int64_t rem = g - tensor * rows_per_tensor * C;
        const int64_t orow = rem / C;          // (out page, head, offset) row
        const int c = (int)(rem - orow * C);
        const int64_t opage = orow / ((int64_t)H * bs);
        const int64_t in_page = orow - opage * H * bs;
        const int src = __ldg(pages + opage);
        if (src < 0 || src >= num_pages) {
            if (c == 0 && in_page == 0 && tensor == 0) xy::set_err(err, XY_DEV_PAGE_OOB);
            continue;
        }
        const int64_t srow = (int64_t)src * H * bs + in_page;
        const float s = __ldg((tensor ? v_scales : k_scales) + srow);
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>((tensor ? v_codes : k_codes) + srow * D) + c);
        uint32_t h[4];
        xy::e4m3x4_to_f16x2x2(w.x, h[0], h[1]);
        xy::e4m3x4_to_f16x2x2(w.y, h[2], h[3]);
        uint4 o;
        uint32_t *ov = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 hv = *reinterpret_cast<const __half2 *>(&h[i]);
            const float lo = __low2float(hv) * s, hi = __high2float(hv) * s;  // IEEE fp32 products
            ov[i] = xy::pack_bf16x2(lo, hi);
        }
        *(reinterpret_cast<uint4 *>((tensor ? v_out : k_out) + orow * D) + c) = o;
    }
}

}  // namespace

extern "C" xy_status xy_dequant_pages_fp8(const void *k_codes, const void *v_codes, const float *k_scales,
                                          const float *v_scales, int num_pages, int num_heads_kv, int block_size,
                                          int head_dim, const int32_t *pages, int num_out, void *k_out, void *v_out,
                                          int32_t *err_word, void *stream) {
    if (num_out < 0 || num_pages < 1 || num_heads_kv < 1 || block_size < 1) return XY_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return XY_ERR_UNSUPPORTED;
    if (num_out == 0) return XY_OK;
    if (!k_codes || !v_codes || !k_scales || !v_scales || !pages || !k_out || !v_out || !err_word)
        return XY_ERR_INVALID_ARG;
    if (((uintptr_t)k_codes | (uintptr_t)v_codes | (uintptr_t)k_out | (uintptr_t)v_out) & 15) return XY_ERR_INVALID_ARG;
    const int64_t groups = 2 * (int64_t)num_out * num_heads_kv * block_size * (head_dim / 8);
    const int threads = 256;
    const int blocks = (int)((groups + threads - 1) / threads < 152 * 16 ? (groups + threads - 1) / threads : 152 * 16);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (head_dim == 128)
        dequant_pages_kernel<128><<<blocks, threads, 0, st>>>(
            static_cast<const uint8_t *>(k_codes), static_cast<const uint8_t *>(v_codes), k_scales, v_scales, pages,
            num_out, num_heads_kv, block_size, num_pages, static_cast<__nv_bfloat16 *>(k_out),
            static_cast<__nv_bfloat16 *>(v_out), err_word);
    else
        dequant_pages_kernel<64><<<blocks, threads, 0, st>>>(
            static_cast<const uint8_t *>(k_codes), static_cast<const uint8_t *>(v_codes), k_scales, v_scales, pages,
            num_out, num_heads_kv, block_size, num_pages, static_cast<__nv_bfloat16 *>(k_out),
            static_cast<__nv_bfloat16 *>(v_out), err_word);
    return cudaGetLastError() == cudaSuccess ? XY_OK : XY_ERR_CUDA;
}

extern "C" xy_status xy_kv_append_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                      int num_tokens, void *k_pages, void *v_pages, float *k_scales,
                                      float *v_scales, int num_pages, int num_heads_kv, int block_size,
                                      int head_dim, int32_t *err_word, void *stream) {
    if (num_tokens < 0 || num_pages < 1 || num_heads_kv < 1 || block_size < 16 || (block_size & (block_size - 1)))
        return XY_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return XY_ERR_UNSUPPORTED;
    if (num_tokens == 0) return XY_OK;
    if (!k_new || !v_new || !slot_mapping || !k_pages || !v_pages || !k_scales || !v_scales || !err_word)
        return XY_ERR_INVALID_ARG;
    if (((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)k_pages | (uintptr_t)v_pages) & 15) return XY_ERR_INVALID_ARG;
    const int64_t rows = 2 * (int64_t)num_tokens * num_heads_kv;
    const int threads = 256, blocks = (int)((rows + 7) / 8 < 4096 ? (rows + 7) / 8 : 4096);
    const int64_t pool_slots = (int64_t)num_pages * block_size;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (head_dim == 128)
        kv_append_fp8_kernel<128><<<blocks, threads, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(k_new), static_cast<const __nv_bfloat16 *>(v_new), slot_mapping,
            num_tokens, num_heads_kv, block_size, pool_slots, static_cast<uint8_t *>(k_pages),
            static_cast<uint8_t *>(v_pages), k_scales, v_scales, err_word);
    else
        kv_append_fp8_kernel<64><<<blocks, threads, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(k_new), static_cast<const __nv_bfloat16 *>(v_new), slot_mapping,
            num_tokens, num_heads_kv, block_size, pool_slots, static_cast<uint8_t *>(k_pages),
            static_cast<uint8_t *>(v_pages), k_scales, v_scales, err_word);
    return cudaGetLastError() == cudaSuccess ? XY_OK : XY_ERR_CUDA;
}

extern "C" xy_status xy_kv_append_paged_fp8(const void *k_new, const void *v_new, const int32_t *cu_seqlens_q,
                                            const int32_t *context_lens, const int32_t *block_table, int num_seqs,
                                            int max_blocks, int num_tokens, void *k_pages, void *v_pages,
                                            float *k_scales, float *v_scales, int num_pages, int num_heads_kv,
                                            int block_size, int head_dim, int64_t *slot_mapping, int32_t *err_word,
                                            void *stream) {
    if (num_tokens < 0 || num_seqs < 0 || max_blocks < 1 || num_pages < 1 || num_heads_kv < 1 || block_size < 16 ||
        (block_size & (block_size - 1)))
        return XY_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return XY_ERR_UNSUPPORTED;
    if (num_tokens == 0) return XY_OK;
    if (num_seqs < 1 || !cu_seqlens_q || !context_lens || !block_table || !k_new || !v_new || !k_pages ||
        !v_pages || !k_scales || !v_scales || !err_word)
        return XY_ERR_INVALID_ARG;
    if (((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)k_pages | (uintptr_t)v_pages) & 15) return XY_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return XY_ERR_CUDA;
    const int blocks = num_tokens < sms * 8 ? num_tokens : sms * 8;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto *kn = static_cast<const __nv_bfloat16 *>(k_new);
    auto *vn = static_cast<const __nv_bfloat16 *>(v_new);
    auto *kp = static_cast<uint8_t *>(k_pages);
    auto *vp = static_cast<uint8_t *>(v_pages);
    if (head_dim == 128)
        kv_append_paged_fp8_kernel<128><<<blocks, 256, 0, st>>>(kn, vn, cu_seqlens_q, context_lens, block_table,
                                                                num_seqs, max_blocks, num_tokens, num_heads_kv,
                                                                block_size, num_pages, slot_mapping, kp, vp, k_scales,
                                                                v_scales, err_word);
    else
        kv_append_paged_fp8_kernel<64><<<blocks, 256, 0, st>>>(kn, vn, cu_seqlens_q, context_lens, block_table,
                                                               num_seqs, max_blocks, num_tokens, num_heads_kv,
                                                               block_size, num_pages, slot_mapping, kp, vp, k_scales,
                                                               v_scales, err_word);
    return cudaGetLastError() == cudaSuccess ? XY_OK : XY_ERR_CUDA;
}
