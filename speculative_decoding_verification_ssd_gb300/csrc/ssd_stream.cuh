// ssd_stream.cuh -- geometry of the persistent streaming kernel (ssd_stream.cu),
// shared with the host launcher.
#pragma once

#include <cstddef>

#include <cuda_runtime.h>

namespace ssd {

constexpr int kStreamGroups = 2;       // consumer groups, each with its own ring
constexpr int kStreamGroupWarps = 8;   // warps per consumer group
// consumer warps, then one producer warp per ring, then one tail warp per group
constexpr int kStreamThreads = kStreamGroups * kStreamGroupWarps * 32 + 2 * kStreamGroups * 32;
constexpr int kStreamRingStages = 4;   // stages per ring
constexpr int kStreamStageBytes = 16384;
constexpr int kGroupTokens = 64;   // tokens per group of the per-group arrays
constexpr int kStreamBuffers = 2;  // group-array buffers per consumer group
constexpr int kStreamMaxGroups = 3 * 32 * 32;  // groups per row the tail warp's masks cover

// Dynamic shared memory of the streaming kernel for a vocabulary of V tokens:
// the stage rings plus, per consumer group, kStreamBuffers buffers of two float
// arrays with one entry per 64-token group.
// With sigma_{F,C} found in the pass (sig), each group also keeps a candidate-key
// buffer of kStreamSigKeys 64-bit keys.
constexpr int kStreamSigKeys = 512;
inline size_t stream_dyn_bytes(int V, bool sig = false) {
    const size_t G = (static_cast<size_t>(V) + kGroupTokens - 1) / kGroupTokens;
    const size_t Gp = (G + 127) & ~static_cast<size_t>(127);  // padded to whole 4 x 32-group strips
    return static_cast<size_t>(kStreamGroups) *
           (static_cast<size_t>(kStreamRingStages) * kStreamStageBytes +
            static_cast<size_t>(kStreamBuffers) * 2 * Gp * sizeof(float) +
            (sig ? static_cast<size_t>(kStreamSigKeys) * sizeof(unsigned long long) : 0));
}

struct UnitParams;
int stream_setup(int dtype, size_t optin, size_t *max_dyn);
int stream_launch(int dtype, const UnitParams &P, int grid, size_t dyn, void *stream);
// the wide forms (ssd_stream_wide.cu), reached through the two calls above
int stream_wide_setup(int dtype, size_t optin, size_t *max_dyn);
cudaError_t stream_wide_launch(int dtype, const cudaLaunchConfig_t &cfg, const UnitParams &P);

}  // namespace ssd
