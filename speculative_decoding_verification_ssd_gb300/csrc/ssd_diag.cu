// ssd_diag.cu -- a check of the bounded waits every kernel of the library uses
// (sm_103a): a wait on an mbarrier that nothing completes must give up after its
// time limit, report SSD_DEV_TIMEOUT through dev_status and leave the context
// usable for the next launch.
#include <cuda_runtime.h>

#include "../../include/ssd.h"
#include "ssd_device.cuh"

namespace ssd {
namespace {

__global__ void wait_check_kernel(int32_t *dev_status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival completes phase 0; nothing arrives
        fence_mbar_init();
    }
    __syncthreads();
    const bool done = mbar_wait_suspend_for(&bar, 0, limit_ns);
    if (!done && threadIdx.x == 0) atomicOr(dev_status, SSD_DEV_TIMEOUT);
}

}  // namespace
}  // namespace ssd

extern "C" int ssd_check_wait_timeout(int32_t *dev_status, int limit_ms, void *stream) {
    if (!dev_status || limit_ms < 1 || limit_ms > 10000) return SSD_ERR_INVALID_ARG;
    ssd::wait_check_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        dev_status, static_cast<unsigned long long>(limit_ms) * 1000000ull);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
