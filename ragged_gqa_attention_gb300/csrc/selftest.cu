// selftest.cu - exercises the failure path of the bounded waits on the GPU
// without faulting it: one CTA waits on an mbarrier that nothing arrives on,
// using the same bounded wait as the attention kernels, gives up after the
// given number of clock cycles and reports RGA_ERR_TIMEOUT through the
// device status word, as a timed-out wait in those kernels does.  No copy or
// tensor-core work is in flight, so the CTA simply returns and the context
// stays usable.
//
// It also exposes the fp8 KV cache's in-register E4M3 decoding, so that a
// test can compare all 256 codes with the oracle's decoder, and one store
// through the bounds check of the debug-checks build.
#include <cuda_runtime.h>
#include "rga.h"
#include "device_common.cuh"
#include "ptx.cuh"

namespace rga {

__global__ void selftest_wait_kernel(int32_t *status, unsigned long long limit) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    volatile int *abort = &abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);   // expects one arrival; none ever comes
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_limit(&bar, 0, abort, limit)) set_status(status, 5);
}

// All 256 E4M3 codes through the decode kernel's conversion: out_f16[c] and
// out_bf16[c] are the f16 / bf16 bits of code c.  64 threads; thread l
// converts the word holding codes 4l .. 4l + 3.
__global__ void selftest_e4m3_kernel(uint16_t *out_f16, uint16_t *out_bf16) {
    const int l = threadIdx.x;
    const uint32_t w = (uint32_t)(4 * l) | (uint32_t)(4 * l + 1) << 8 |
                       (uint32_t)(4 * l + 2) << 16 | (uint32_t)(4 * l + 3) << 24;
    uint32_t lo, hi;
    e4m3x4_to_x2<false>(w, lo, hi);
    out_f16[4 * l] = lo & 0xffff; out_f16[4 * l + 1] = lo >> 16;
    out_f16[4 * l + 2] = hi & 0xffff; out_f16[4 * l + 3] = hi >> 16;
    e4m3x4_to_x2<true>(w, lo, hi);
    out_bf16[4 * l] = lo & 0xffff; out_bf16[4 * l + 1] = lo >> 16;
    out_bf16[4 * l + 2] = hi & 0xffff; out_bf16[4 * l + 3] = hi >> 16;
}

// One store through the debug-checks build's bounds check: buf[index] = 1
// when 0 <= index < n, else the store is skipped and the status recorded.
__global__ void selftest_bounds_kernel(int32_t *buf, long long n, long long index,
                                       int32_t *status) {
    if (dbg_ok(index >= 0 && index < n, status)) buf[index] = 1;
}

}  // namespace rga

extern "C" rga_status rga_selftest_bounds_check(int32_t *buf, int64_t n, int64_t index,
                                                 int32_t *device_status, cudaStream_t stream) {
    if (!rga::RGA_DEBUG) return RGA_ERR_UNSUPPORTED;
    if (!buf || !device_status || n <= 0) return RGA_ERR_INVALID_ARG;
    rga::selftest_bounds_kernel<<<1, 1, 0, stream>>>(buf, (long long)n, (long long)index,
                                                      device_status);
    return cudaGetLastError() == cudaSuccess ? RGA_OK : RGA_ERR_CUDA;
}

extern "C" rga_status rga_selftest_e4m3_decode(uint16_t *out_f16, uint16_t *out_bf16,
                                                cudaStream_t stream) {
    if (!out_f16 || !out_bf16) return RGA_ERR_INVALID_ARG;
    rga::selftest_e4m3_kernel<<<1, 64, 0, stream>>>(out_f16, out_bf16);
    return cudaGetLastError() == cudaSuccess ? RGA_OK : RGA_ERR_CUDA;
}

extern "C" rga_status rga_selftest_wait_timeout(int32_t *device_status, int64_t wait_cycles,
                                                 cudaStream_t stream) {
    if (!device_status || wait_cycles <= 0 || wait_cycles > (int64_t(1) << 32))
        return RGA_ERR_INVALID_ARG;
    rga::selftest_wait_kernel<<<1, 32, 0, stream>>>(device_status,
                                                    (unsigned long long)wait_cycles);
    return cudaGetLastError() == cudaSuccess ? RGA_OK : RGA_ERR_CUDA;
}
