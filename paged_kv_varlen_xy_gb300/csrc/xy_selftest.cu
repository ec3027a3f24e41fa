// Self-test of the bounded waits every kernel of libxy relies on (not a step of the path).
//
// Each wait on an mbarrier in the attention kernels gives up after a time limit (or when the
// CTA's abort flag is raised), records XY_DEV_TIMEOUT in the error word and lets the kernel
// return, so a lost arrival can never hang the GPU.  This kernel exercises exactly that
// mechanism on barriers nobody arrives at: warp 0 waits with a time limit, warp 1 waits with no
// limit of its own but is released by the abort flag warp 0 raises after its wait ran out.

#include <cuda_runtime.h>
#include <stdint.h>

#include "xy.h"
#include "xy_device.cuh"

namespace {

__global__ void __launch_bounds__(64, 1) bounded_wait_kernel(uint64_t limit_ns, int32_t *err_word, int32_t *result) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ volatile int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        xy::mbar_init(xy::smem_u32(&bars[0]), 1);
        xy::mbar_init(xy::smem_u32(&bars[1]), 1);
        abort_flag = 0;
        xy::fence_mbarrier_init();
    }
    __syncthreads();
    if (warp == 0) {
        // nobody arrives: the wait must give up after limit_ns
        const uint64_t t0 = xy::global_timer_ns();
        const bool ok = xy::mbar_wait_for(xy::smem_u32(&bars[0]), 0, nullptr, limit_ns);
        const uint64_t waited = xy::global_timer_ns() - t0;
        if (lane == 0) {
            result[0] = ok ? 1 : 0;
            result[1] = (int32_t)(waited / 1000u);  // microseconds
            if (!ok) xy::set_err(err_word, XY_DEV_TIMEOUT);
            abort_flag = 1;
        }
    } else {
        // the generous limit of the kernels, cut short by the abort flag
        const bool ok = xy::mbar_wait(xy::smem_u32(&bars[1]), 0, &abort_flag);
        if (lane == 0) result[2] = ok ? 1 : 0;
    }
}

}  // namespace

extern "C" xy_status xy_selftest_bounded_wait(uint32_t limit_us, int32_t *err_word, int32_t *result,
                                              void *stream) {
    if (!err_word || !result || limit_us == 0 || limit_us > 10000000u) return XY_ERR_INVALID_ARG;
    bounded_wait_kernel<<<1, 64, 0, (cudaStream_t)stream>>>((uint64_t)limit_us * 1000u, err_word, result);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? XY_OK : XY_ERR_CUDA;
}
