// ssd_vec.cuh -- per-storage-type operations on 16-byte vectors of staged logits
// (8 bf16 or 4 fp32 values), used by the unit and reshape kernels.
//
// Raw maxima propagate NaN (max.NaN), so a NaN logit is visible to the caller;
// raw comparisons work on the stored values without converting them.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "ssd_device.cuh"

namespace ssd {

__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ uint32_t hmax2_nan_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// 0xFFFF in each half where a >= b (bf16x2, ordered comparison).
__device__ __forceinline__ uint32_t hge2_mask_u32(uint32_t a, uint32_t b) {
    __nv_bfloat162 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    return __hge2_mask(x, y);
}

// Negative infinity in storage format.
template <class D>
struct NegInf;
template <>
struct NegInf<F32Tag> {
    static constexpr uint32_t kWord = 0xFF800000u;
};
template <>
struct NegInf<BF16Tag> {
    static constexpr uint32_t kHalf = 0xFF80u;
};

// Replaces by -inf every lane of vector w (first element e0) outside [lo, hi)
// and the lane holding token `excl` (pass -1 for none).
template <class D>
__device__ __forceinline__ void mask_vec(uint4 &w, int e0, int lo, int hi, int excl);

template <>
__device__ __forceinline__ void mask_vec<F32Tag>(uint4 &w, int e0, int lo, int hi, int excl) {
    uint32_t *p = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = e0 + i;
        if (e < lo || e >= hi || e == excl) p[i] = NegInf<F32Tag>::kWord;
    }
}

template <>
__device__ __forceinline__ void mask_vec<BF16Tag>(uint4 &w, int e0, int lo, int hi, int excl) {
    uint32_t *p = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = e0 + i;
        if (e < lo || e >= hi || e == excl) {
            const int s = (i & 1) * 16;
            p[i >> 1] = (p[i >> 1] & ~(0xFFFFu << s)) | (NegInf<BF16Tag>::kHalf << s);
        }
    }
}

// Running raw maximum of vectors (storage domain, NaN propagating).
template <class D>
struct RawMax;

template <>
struct RawMax<F32Tag> {
    float m = -INFINITY;
    __device__ __forceinline__ void add(const uint4 &w) {
        m = fmax_nan(m, fmax_nan(fmax_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                                 fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w))));
    }
    __device__ __forceinline__ float get() const { return m; }
};

template <>
struct RawMax<BF16Tag> {
    uint32_t m2 = 0xFF80FF80u;  // (-inf, -inf)
    __device__ __forceinline__ void add(const uint4 &w) {
        m2 = hmax2_nan_u32(m2, hmax2_nan_u32(hmax2_nan_u32(w.x, w.y), hmax2_nan_u32(w.z, w.w)));
    }
    __device__ __forceinline__ float get() const {
        return fmax_nan(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
    }
};

// Bit mask of the lanes of w whose stored value is >= t (t given as an fp32
// value that is exactly representable in the storage type).
template <class D>
__device__ __forceinline__ uint32_t ge_lanes(const uint4 &w, float t);

template <>
__device__ __forceinline__ uint32_t ge_lanes<F32Tag>(const uint4 &w, float t) {
    return (__uint_as_float(w.x) >= t ? 1u : 0u) | (__uint_as_float(w.y) >= t ? 2u : 0u) |
           (__uint_as_float(w.z) >= t ? 4u : 0u) | (__uint_as_float(w.w) >= t ? 8u : 0u);
}

template <>
__device__ __forceinline__ uint32_t ge_lanes<BF16Tag>(const uint4 &w, float t) {
    const uint32_t tb = __float_as_uint(t) >> 16;
    const uint32_t t2 = tb | (tb << 16);
    const uint32_t a = hge2_mask_u32(w.x, t2), b = hge2_mask_u32(w.y, t2);
    const uint32_t c = hge2_mask_u32(w.z, t2), d = hge2_mask_u32(w.w, t2);
    if ((a | b | c | d) == 0) return 0;
    return (a & 1u) | ((a >> 15) & 2u) | ((b & 1u) << 2) | ((b >> 13) & 8u) | ((c & 1u) << 4) |
           ((c >> 11) & 32u) | ((d & 1u) << 6) | ((d >> 9) & 128u);
}

// Largest storage value <= x (round toward -inf into the storage type).
template <class D>
__device__ __forceinline__ float round_down_storage(float x);
template <>
__device__ __forceinline__ float round_down_storage<F32Tag>(float x) { return x; }
template <>
__device__ __forceinline__ float round_down_storage<BF16Tag>(float x) {
    return __bfloat162float(__float2bfloat16_rd(x));
}

// Base-2 softmax partial sum of a vector: sum_i 2^(z_i c - mc) over its lanes.
template <class D>
__device__ __forceinline__ float2 exp_sum(const uint4 &w, float c, float mc, float2 acc);

template <>
__device__ __forceinline__ float2 exp_sum<F32Tag>(const uint4 &w, float c, float mc, float2 acc) {
    const float2 cc = make_float2(c, c), nm = make_float2(-mc, -mc);
    float2 x0 = __ffma2_rn(make_float2(__uint_as_float(w.x), __uint_as_float(w.y)), cc, nm);
    float2 x1 = __ffma2_rn(make_float2(__uint_as_float(w.z), __uint_as_float(w.w)), cc, nm);
    acc = __fadd2_rn(acc, make_float2(ex2(x0.x), ex2(x0.y)));
    acc = __fadd2_rn(acc, make_float2(ex2(x1.x), ex2(x1.y)));
    return acc;
}

template <>
__device__ __forceinline__ float2 exp_sum<BF16Tag>(const uint4 &w, float c, float mc, float2 acc) {
    const float2 cc = make_float2(c, c), nm = make_float2(-mc, -mc);
    const uint32_t r[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 z = make_float2(__uint_as_float(r[i] << 16), __uint_as_float(r[i] & 0xFFFF0000u));
        const float2 x = __ffma2_rn(z, cc, nm);
        acc = __fadd2_rn(acc, make_float2(ex2(x.x), ex2(x.y)));
    }
    return acc;
}

}  // namespace ssd
