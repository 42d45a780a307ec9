// ssd_slice.cuh -- geometry and workspace layout of the slice kernel
// (ssd_slice.cu), shared with the host launcher.
//
// The slice kernel splits every logit row into S slices of whole 16 KB blocks
// and schedules (unit, slice) items dynamically over all SMs; the slices of a
// unit are combined in global memory by whichever tail warp finishes the last
// of them, and a pair's second pass is queued as further items once its
// normalisers are known.
#pragma once

#include <cstddef>
#include <cstdint>

#include "ssd_stream.cuh"
#include "ssd_unit.cuh"

namespace ssd {

constexpr int kSliceBlockBytes = 16384;  // one single-row stage; two pair stages of 8 KB per row
constexpr int kSliceMaxGroups = 1024;    // 64-token groups per slice (shared-memory arrays)
constexpr int kSliceBuffers = 3;         // group-array buffers per consumer group
constexpr int kSliceMaxSlices = 32;      // a unit's queued slices fit one 32-bit mask
constexpr int kSliceTargetItems = 1216;  // first-pass items aimed at (4 per consumer group of 152 SMs)
constexpr int kSliceScratch = kStreamMaxGroups;  // floats of a tail warp's scratch (a row's groups)

// Per-unit state in the workspace (zero between launches: the unit's finisher
// resets its counters).
struct SliceUnitState {
    uint32_t p1_done;     // first-pass slices finished
    uint32_t p2_done;     // second-pass items finished
    uint32_t p2_expect;   // second-pass items queued
    uint32_t flags;       // SSD_DEV_* bits, kSliceSkipped
    float LT, LD;         // pair: base-2 normalisers of target and draft
    float c;              // log2 e / tau
    float cthr;           // pair: a residual at least F_k tokens reach (-inf: none known)
    float p_tok, q_tok;
    int32_t accept;
    uint32_t slice_mask;  // pair: slices queued for the second pass
    float M, Ssum;        // sampled single row: base-2 statistics
    int32_t pad[2];
};
static_assert(sizeof(SliceUnitState) == 64, "slice unit state");
constexpr uint32_t kSliceSkipped = 1u << 30;

inline int slice_vec(int dtype_bytes) { return 16 / dtype_bytes; }

// 16 KB blocks per row and 64-token groups per block.
inline int slice_blocks(int V, int elem) {
    const long long bytes = static_cast<long long>(V) * elem;
    return static_cast<int>((bytes + kSliceBlockBytes - 1) / kSliceBlockBytes);
}
inline int slice_groups_per_block(int elem) { return kSliceBlockBytes / elem / kGroupTokens; }

// Slices per row: enough items to keep every consumer group busy, whole blocks,
// at most kSliceMaxGroups groups and at most kSliceMaxSlices slices.
inline int slice_count(int units, int V, int elem) {
    const int nblk = slice_blocks(V, elem);
    const int gpb = slice_groups_per_block(elem);
    int S = (units >= kSliceTargetItems) ? 1 : (kSliceTargetItems + units - 1) / units;
    const int smin = (nblk * gpb + kSliceMaxGroups - 1) / kSliceMaxGroups;
    if (S < smin) S = smin;
    if (S > nblk) S = nblk;
    if (S > kSliceMaxSlices) S = kSliceMaxSlices;
    return S < 1 ? 1 : S;
}

// First block of slice s (blocks spread evenly, so every slice has at least one).
__host__ __device__ inline int slice_block0(int s, int S, int nblk) {
    return static_cast<int>((static_cast<long long>(s) * nblk) / S);
}

// Workspace regions of the slice kernel, after the records and per-sequence
// counters the other kernels use (each region 256-byte aligned).
struct SliceWs {
    size_t counters, ustate, sstat, skeys, garr, queue, pcand, cmax, total;
};
constexpr int kSliceCand = 64;  // candidate groups a first-pass pair slice reports for the residual bound
inline int slice_pair_chunks(int V, int elem) {
    const long long bytes = static_cast<long long>(V) * elem;
    return static_cast<int>((bytes + kSliceBlockBytes / 2 - 1) / (kSliceBlockBytes / 2));
}
inline SliceWs slice_ws_layout(int B, int K, int V, int elem, int key_stride) {
    const size_t units = static_cast<size_t>(B) * (K + 1);
    const int S = slice_count(static_cast<int>(units), V, elem);
    const size_t G = (static_cast<size_t>(V) + kGroupTokens - 1) / kGroupTokens;
    const size_t GA = (G + 3) & ~static_cast<size_t>(3);  // per-unit arrays 16-byte aligned
    SliceWs L;
    size_t o = ws_total_bytes(B, K);
    L.counters = o;
    o += 256;
    L.ustate = o;
    o = align256(o + units * sizeof(SliceUnitState));
    L.sstat = o;
    o = align256(o + units * S * 16);
    L.skeys = o;
    o = align256(o + static_cast<size_t>(B) * S * key_stride * 8);
    L.garr = o;
    o = align256(o + units * 2 * GA * sizeof(float));
    L.queue = o;
    o = align256(o + units * S * 8);
    L.pcand = o;  // per (unit, slice): kSliceCand (target max, draft max) pairs
    o = align256(o + units * S * kSliceCand * 2 * sizeof(float));
    L.cmax = o;   // per unit: each pair chunk's largest target maximum
    o = align256(o + units * static_cast<size_t>(slice_pair_chunks(V, elem)) * sizeof(float));
    L.total = o;
    return L;
}

// Key entries per (sequence, slice): every position keeps max(F_k, 1) keys (a
// greedy row's argmax is its best key even without a cache).
inline int slice_key_stride(int K, const int *F_or_null) {
    int n = 0;
    for (int k = 0; k <= K; ++k) {
        const int f = F_or_null ? F_or_null[k] : 0;
        n += f > 1 ? f : 1;
    }
    return n;
}

int slice_setup(int dtype, size_t optin, size_t *max_dyn);
int slice_launch(int dtype, const UnitParams &P, int grid, size_t dyn, void *stream);
// Dynamic shared memory: per consumer group its ring and kSliceBuffers buffers of
// two group arrays, and per tail warp a scratch of one float per group of a row.
inline size_t slice_dyn_bytes() {
    return static_cast<size_t>(kStreamGroups) *
           (static_cast<size_t>(kStreamRingStages) * kStreamStageBytes +
            static_cast<size_t>(kSliceBuffers) * 2 * kSliceMaxGroups * sizeof(float) +
            static_cast<size_t>(kSliceScratch) * sizeof(float));
}

}  // namespace ssd
