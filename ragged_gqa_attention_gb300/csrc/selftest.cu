// selftest.cu - exercises the failure path of the bounded waits on the GPU
// without faulting it: one CTA waits on an mbarrier that nothing arrives on,
// using the same bounded wait as the attention kernels, gives up after the
// given number of clock cycles and reports RGA_ERR_TIMEOUT through the
// device status word, as a timed-out wait in those kernels does.  No copy or
// tensor-core work is in flight, so the CTA simply returns and the context
// stays usable.
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

}  // namespace rga

extern "C" rga_status rga_selftest_wait_timeout(int32_t *device_status, int64_t wait_cycles,
                                                 cudaStream_t stream) {
    if (!device_status || wait_cycles <= 0 || wait_cycles > (int64_t(1) << 32))
        return RGA_ERR_INVALID_ARG;
    rga::selftest_wait_kernel<<<1, 32, 0, stream>>>(device_status,
                                                    (unsigned long long)wait_cycles);
    return cudaGetLastError() == cudaSuccess ? RGA_OK : RGA_ERR_CUDA;
}
