// ssd_backup.cu -- the fast random-token backup speculator (sm_103a).
//
// [SSD] "Speculative Speculative Decoding" notes (papernotes.org), "关键设计"
// item 3 (batch-size-aware fallback): at large batch at least one sequence
// misses the speculation cache in almost every round, so the backup that
// drafts for the missed sequences should be as fast as possible; the paper's
// implementation drafts random tokens.  Here every sequence with hit[b] == 0
// gets K tokens drawn uniformly from the vocabulary from the caller's uniforms.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/ssd.h"

namespace ssd {
namespace {

__global__ void backup_fill_kernel(const uint8_t *__restrict__ hit, const float *__restrict__ u, int B,
                                   int K, int V, int32_t *__restrict__ next_tokens) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(B) * K) return;
    const int b = static_cast<int>(i / K);
    if (hit[b]) return;
    // u * V is exact in double (24-bit mantissa times a value below 2^31)
    const double x = static_cast<double>(u[i]) * static_cast<double>(V);
    long long t = static_cast<long long>(floor(x));
    if (t > V - 1) t = V - 1;
    if (t < 0) t = 0;
    next_tokens[i] = static_cast<int32_t>(t);
}

}  // namespace
}  // namespace ssd

extern "C" int ssd_backup_fill(const uint8_t *hit, const float *uniforms, int B, int K, int V,
                               int32_t *next_tokens, void *stream) {
    if (!hit || !uniforms || !next_tokens || B < 1 || K < 1 || K > SSD_MAX_K || V < 1)
        return SSD_ERR_INVALID_ARG;
    const int64_t n = static_cast<int64_t>(B) * K;
    const int threads = 256;
    const int64_t blocks = (n + threads - 1) / threads;
    if (blocks > 0x7FFFFFFF) return SSD_ERR_UNSUPPORTED;
    ssd::backup_fill_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
        hit, uniforms, B, K, V, next_tokens);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
    return SSD_OK;
}
