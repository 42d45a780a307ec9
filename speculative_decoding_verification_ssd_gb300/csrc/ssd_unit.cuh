// ssd_unit.cuh -- parameters and workspace records of the fused verify / cache-build
// kernel (ssd_unit.cu), shared with the host launcher (ssd_api.cu).
#pragma once

#include <cstdint>
#include <vector_types.h>

#include "../../include/ssd.h"

namespace ssd {

enum : int {
    kModeVerify = 1,     // accept tests, scan, bonus draw -> accept_len / bonus / p_tok / q_tok
    kModeCache = 2,      // top-F_k per outcome -> cache_tok
    kModeLookup = 4,     // hit test of (a, t*) in the freshly built cache
    kModeEarlyExit = 8,  // units after a known rejection skip their rows
};

// One record per (sequence b, position k), k = 0..K, in the workspace.
struct UnitRecord {
    float p_tok;     // p_k(x~_k)            (k < K)
    float q_tok;     // q_k(x~_k)            (k < K)
    int32_t accept;  // 1 if x~_k accepted   (k < K)
    int32_t tk;      // bonus drawn if the round stops at k
    int32_t flags;   // SSD_DEV_* bits seen by this unit
    int32_t state;   // 1 computed, 2 skipped
    int32_t pad[2];
};
static_assert(sizeof(UnitRecord) == 32, "record layout");

struct UnitParams {
    const void *tgt;
    const void *drf;
    int64_t ld;              // elements between consecutive rows (>= V)
    int64_t tgt_seq_stride;  // elements between sequences of tgt ((K+1) ld)
    int64_t drf_seq_stride;  // elements between sequences of drf (drf_rows ld)
    int B, K, V;
    int CL;              // CTAs per unit (thread-block cluster size)
    int slice;           // vocabulary entries per CTA (multiple of the 16-byte vector)
    int row_buf_bytes;   // bytes of one staged row buffer (>= slice * elem + 64)
    int mode;            // kMode* bits
    const int32_t *tokens;
    const float *uniforms;
    const float *temperature;
    const ssd_reshape_desc *reshape;  // [B, K] or nullptr
    int budget;
    int F[SSD_MAX_K + 1];
    int off[SSD_MAX_K + 2];
    int32_t *cache_tok;
    int32_t *accept_len;
    int32_t *bonus;
    float *p_tok;
    float *q_tok;
    uint8_t *hit;
    int32_t *slot;
    UnitRecord *rec;       // [B, K+1]
    uint32_t *seq_count;   // [B] finished CTAs of the sequence (reset by the epilogue)
    uint32_t *seq_reject;  // [B] bit k set when position k rejected (reset by the epilogue)
    int32_t *dev_status;
    // persistent streaming kernel only
    uint32_t *unit_counter;  // next unit to hand out (reset by the last CTA to exit)
    unsigned long long *unit_ends;  // streaming kernel: units handed out (low 32 bits; the
                                    // high half stays zero)
    uint32_t *exit_counter;  // CTAs that have exited
    int perm_mul;            // unit u -> sequence ((u % B) * perm_mul) % B (coprime to B)
    int wide;                // streaming kernel: both consumer groups of a CTA share each unit
    // sigma_{F,C} found in the pass over the draft rows (streaming kernel only):
    // position k of a sampled sequence reshapes with F = sig_F[k] (0: none)
    int sig_on;
    int sig_F[SSD_MAX_K];
    float sig_C;
    ssd_reshape_desc *desc_out;  // [B, K] descriptors found (sampled sequences), or nullptr
    // slice kernel only: S slices of nblk 16 KB blocks per row; per-(sequence,
    // slice) key areas of key_stride entries (position k at koff[k])
    int S, nblk, key_stride;
    int koff[SSD_MAX_K + 1];
    struct SliceUnitState *ustate;  // [B, K+1]
    float4 *sstat;                  // [B, K+1, S] slice statistics / residual totals
    unsigned long long *skeys;      // [B, S, key_stride] slice top-F keys
    float *garr;                    // [B, K+1, 2, G] per-group data in global memory
    unsigned long long *queue;      // [B (K+1) S] second-pass items
    float *pcand;                   // [B, K+1, S, kSliceCand, 2] residual-bound candidates
    float *cmax;                    // [B, K+1, pair chunks] largest target maximum per chunk
    uint32_t *slice_ctr;            // scheduler counters (reset by the last CTA to exit)
};

// Workspace layout (each region 256-byte aligned).
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline size_t ws_rec_bytes(int B, int K) {
    return align256(static_cast<size_t>(B) * (K + 1) * sizeof(UnitRecord));
}
inline size_t ws_count_bytes(int B) { return align256(static_cast<size_t>(B) * sizeof(uint32_t)); }
inline size_t ws_total_bytes(int B, int K) {
    return ws_rec_bytes(B, K) + 2 * ws_count_bytes(B) + 256;  // + scheduler counters
}

}  // namespace ssd
