// ssd_reshape.cuh -- parameters of the sigma_{F,C} reshape kernel and of the
// stand-alone cache lookup kernel (ssd_reshape.cu), shared with ssd_api.cu.
#pragma once

#include <cstdint>

#include "../../include/ssd.h"

namespace ssd {

struct ReshapeParams {
    const void *drf;       // [rows, V] stored logits
    int rows, V;
    int CL, slice, row_buf_bytes;
    const float *tau;      // [rows] (needed only for q_out)
    int F;
    float C;
    ssd_reshape_desc *desc;  // [rows] (or [B, K] in draft-cache mode), or nullptr
    float *q_out;            // [rows, V] or nullptr
    int32_t *dev_status;
    // Draft-cache mode (seq_rows > 0): rows are [B, seq_rows = K+1, V] and row r
    // is position k = r mod (K+1) of sequence r / (K+1), with F = Fk[k].
    int seq_rows, K;
    int Fk[SSD_MAX_K + 1];
    int off[SSD_MAX_K + 2];
    const int32_t *tokens;   // [B, K] drafted tokens excluded from segment k < K, or nullptr
    int32_t *cache_tok;      // [B, budget] or nullptr
    int budget;
};

struct LookupParams {
    const int32_t *cache_tok;  // [B, budget]
    int B, K, budget;
    int off[SSD_MAX_K + 2];
    const int32_t *accept_len;
    const int32_t *bonus;
    uint8_t *hit;
    int32_t *slot;
};

}  // namespace ssd
