// ssd_launch.cuh -- host helpers used by each kernel translation unit to set
// kernel attributes and to launch with a thread-block cluster dimension.
#pragma once

#include <cuda_runtime.h>

#include "../../include/ssd.h"
#include "ssd_device.cuh"

namespace ssd {

// Opts the kernel into the largest dynamic shared memory the device allows
// (minus its static shared memory) and, where available, into non-portable
// cluster sizes (up to 16 CTAs).
template <class Kern>
int setup_kernel(Kern kern, size_t optin, size_t *max_dyn, bool *allow16) {
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess) return SSD_ERR_CUDA;
    const size_t used = attr.sharedSizeBytes + 1024;
    const size_t dyn = optin > used ? optin - used : 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(dyn)) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess) {
        cudaGetLastError();
        *allow16 = false;
    }
    *max_dyn = dyn;
    return SSD_OK;
}

template <class Kern, class Params>
int launch_clustered(Kern kern, const Params &P, int grid, int CL, size_t dyn, void *stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(CL);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, P) != cudaSuccess) {
        cudaGetLastError();
        return SSD_ERR_CUDA;
    }
    return SSD_OK;
}

// Entry points exported by the kernel translation units.
struct UnitParams;
struct ReshapeParams;
struct LookupParams;
int unit_setup(int dtype, size_t optin, size_t *max_dyn, bool *allow16);
int unit_launch(int dtype, const UnitParams &P, int grid, int CL, size_t dyn, void *stream);
int reshape_setup(int dtype, size_t optin, size_t *max_dyn, bool *allow16);
int reshape_launch(int dtype, const ReshapeParams &P, int grid, int CL, size_t dyn, void *stream);
int lookup_launch(const LookupParams &P, void *stream);

}  // namespace ssd
