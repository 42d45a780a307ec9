// ssd_stream_ops.cuh -- per-stage device operations of the persistent streaming
// kernels (ssd_stream.cu, ssd_slice.cu): staged-vector loads, raw maxima and
// base-2 exponential sums of 16-byte vectors, online softmax statistics,
// reductions over thread groups and warps, the residual of one token and the
// sigma_{F,C} draft bias, and the bulk-copy / L2-policy wrappers.
//
// Sources of the operations: [SD] "Speculative decoding" (brentwoodlivery.com),
// "The Algorithm (Step-by-Step)" step 3 (residual max(0, p - q)) and "Temperature
// and Sampling" (softmax at tau); [SSD] "Speculative Speculative Decoding" notes
// (papernotes.org), "关键设计" item 2 (sigma_{F,C}).
#pragma once

#include <cstdint>

#include "ssd_device.cuh"
#include "ssd_vec.cuh"

namespace ssd {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kLog2e = 1.4426950408889634f;

struct DraftShape {
    int on;
    float thr;
    int thr_id;
    float l2C;
};

__device__ __forceinline__ float draft_bias(const DraftShape &r, float z, int e) {
    return (r.on && (z > r.thr || (z == r.thr && e <= r.thr_id))) ? r.l2C : 0.f;
}

// Residual max(0, p - q) of one token: p = 2^(z_p c - L_T), q = 2^(z_q c + b - L_D)
// with nLT = -L_T and nLDb = b - L_D.  The stage code computes the same
// operations two tokens at a time, so both give identical bits.
__device__ __forceinline__ float resid_of(float zp, float zq, float c, float nLT, float nLDb) {
    const float ep = ex2(fmaf(zp, c, nLT));
    const float eq = ex2(fmaf(zq, c, nLDb));
    return fmaxf(ep - eq, 0.f);
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_copy_hint(void *dst, const void *src, uint32_t bytes,
                                               uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

template <class D>
__device__ __forceinline__ uint4 neg_inf_vec() {
    if (D::kBytes == 4) return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
    return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
}

// Loads the VPT vectors [vbase, vbase + VPT) of a staged row, rotated by `rot`
// so that neighbouring threads hit different shared-memory banks.  With
// `full` every vector is in the stage; otherwise vectors at or past nvec read
// as -inf.
template <class D, int VPT>
__device__ __forceinline__ void load_vecs(const unsigned char *row, int vbase, int nvec, int rot,
                                          bool full, uint4 (&w)[VPT]) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = vbase + ((k + rot) & (VPT - 1));
        if (full)
            w[k] = *reinterpret_cast<const uint4 *>(row + 16 * v);
        else
            w[k] = v < nvec ? *reinterpret_cast<const uint4 *>(row + 16 * v) : neg_inf_vec<D>();
    }
}

// The row's last vector holds `valid` tokens when the row is not a whole number
// of 16-byte vectors (a row stride longer than V): the rest read as -inf.
template <class D>
__device__ __forceinline__ uint4 mask_tail(uint4 w, int valid) {
    uint32_t r[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (D::kBytes == 4) {
            if (j >= valid) r[j] = 0xFF800000u;
        } else {
            if (2 * j >= valid) r[j] = (r[j] & 0xFFFF0000u) | 0x0000FF80u;
            if (2 * j + 1 >= valid) r[j] = (r[j] & 0x0000FFFFu) | 0xFF800000u;
        }
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}
template <class D, int VPT>
__device__ __forceinline__ void mask_partial(uint4 (&w)[VPT], int vbase, int rot, int pv, int valid) {
#pragma unroll
    for (int k = 0; k < VPT; ++k)
        if (vbase + ((k + rot) & (VPT - 1)) == pv) w[k] = mask_tail<D>(w[k], valid);
}

template <class D, int VPT>
__device__ __forceinline__ float vecs_max(const uint4 (&w)[VPT]) {
    RawMax<D> rm;
#pragma unroll
    for (int k = 0; k < VPT; ++k) rm.add(w[k]);
    return rm.get();
}

// sum over the vectors of 2^(z c - mc), two independent accumulators
template <class D, int VPT>
__device__ __forceinline__ float vecs_expsum(const uint4 (&w)[VPT], float c, float mc) {
    float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; k += 2) {
        a = exp_sum<D>(w[k], c, mc, a);
        if (k + 1 < VPT) b = exp_sum<D>(w[k + 1], c, mc, b);
    }
    return (a.x + a.y) + (b.x + b.y);
}

template <int TPG>
__device__ __forceinline__ float tpg_max_nan(float v) {
#pragma unroll
    for (int o = 1; o < TPG; o <<= 1) v = fmax_nan(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
template <int TPG>
__device__ __forceinline__ float tpg_max(float v) {
#pragma unroll
    for (int o = 1; o < TPG; o <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
template <int TPG>
__device__ __forceinline__ float tpg_sum(float v) {
#pragma unroll
    for (int o = 1; o < TPG; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// NaN-propagating merge of two online statistics (branch-free).
__device__ __forceinline__ Stat stat_merge_nan(Stat a, Stat b) {
    const float m = fmax_nan(a.m, b.m);
    const float sa = (a.m == -INFINITY) ? 0.f : a.S * ex2(a.m - m);
    const float sb = (b.m == -INFINITY) ? 0.f : b.S * ex2(b.m - m);
    return {m, (m == -INFINITY) ? 0.f : sa + sb};
}

// Folds a block whose largest base-2 value is xm into st; mass(mn) returns the
// block's sum of 2^(x - mn) for the new maximum mn (branch-free: an all -inf
// block leaves st unchanged, a NaN makes it NaN).
template <class F>
__device__ __forceinline__ void stat_fold(Stat &st, float xm, F mass) {
    const float mn = fmax_nan(st.m, xm);
    const float keep = (st.m == -INFINITY) ? 0.f : st.S * ex2(st.m - mn);
    const float add = mass(mn);
    st.S = (mn == -INFINITY) ? 0.f : keep + add;
    st.m = mn;
}

__device__ __forceinline__ Stat warp_stat(Stat s) {
    const uint32_t mo = __reduce_max_sync(kFull, ordered_bits_nz(s.m));  // -0 vs +0: same value
    const float M = value_of_ordered(mo);
    float S = (s.m == -INFINITY) ? 0.f : s.S * ex2(s.m - M);
    if (M == -INFINITY) S = 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(kFull, S, o);
    return {M, S};
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t x = __shfl_xor_sync(kFull, v, o);
        v = x > v ? x : v;
    }
    return v;
}

// Inclusive prefix sum over the warp (fp64).
__device__ __forceinline__ double warp_incl_scan(double v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

__device__ __forceinline__ bool stat_ok(Stat s) {
    return (s.m < INFINITY) && (s.S > 0.f) && (s.S < INFINITY);
}

// Pass 1 of a sigma-reshaped draft row: weights 2^(z c + log2 c_t) folded into
// st (kept out of line: the common path has no reshape).
template <class D, int VPT>
__device__ __noinline__ Stat reshaped_fold(Stat st, const unsigned char *row, int vbase, int nvec, int rot,
                                           bool full, float c, DraftShape shape, int e0, int pv, int valid) {
    constexpr int VEC = D::kVec;
    uint4 w[VPT];
    load_vecs<D, VPT>(row, vbase, nvec, rot, full, w);
    if (pv >= 0) mask_partial<D, VPT>(w, vbase, rot, pv, valid);
    float x[VPT][VEC];
    float xm = -INFINITY;
#pragma unroll
    for (int kk = 0; kk < VPT; ++kk) {
        float z[VEC];
        decode_vec<D>(w[kk], z);
        const int ev = e0 + ((kk + rot) & (VPT - 1)) * VEC;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            x[kk][i] = z[i] * c + draft_bias(shape, z[i], ev + i);
            xm = fmax_nan(xm, x[kk][i]);
        }
    }
    stat_fold(st, xm, [&](float mn) {
        float vs = 0.f;
#pragma unroll
        for (int kk = 0; kk < VPT; ++kk)
#pragma unroll
            for (int i = 0; i < VEC; ++i) vs += ex2(x[kk][i] - mn);
        return vs;
    });
    return st;
}

// Pass 2 of a pair with a sigma-reshaped draft: residual sum (x) and maximum (y)
// of this thread's tokens (out of line, as above).
template <class D, int VPT>
__device__ __noinline__ float2 reshaped_resid(const unsigned char *stg, int half, int vbase, int nvec,
                                              int rot, bool full, float c, float LT, float LD,
                                              DraftShape shape, int e0, int pv, int valid) {
    constexpr int VEC = D::kVec;
    uint4 wt[VPT], wd[VPT];
    load_vecs<D, VPT>(stg, vbase, nvec, rot, full, wt);
    load_vecs<D, VPT>(stg + half, vbase, nvec, rot, full, wd);
    if (pv >= 0) {
        mask_partial<D, VPT>(wt, vbase, rot, pv, valid);
        mask_partial<D, VPT>(wd, vbase, rot, pv, valid);
    }
    float acc = 0.f, mx = 0.f;
#pragma unroll
    for (int kk = 0; kk < VPT; ++kk) {
        float zt[VEC], zd[VEC];
        decode_vec<D>(wt[kk], zt);
        decode_vec<D>(wd[kk], zd);
        const int ev = e0 + ((kk + rot) & (VPT - 1)) * VEC;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const float wv = resid_of(zt[i], zd[i], c, -LT, draft_bias(shape, zd[i], ev + i) - LD);
            acc += wv;
            mx = fmaxf(mx, wv);
        }
    }
    return make_float2(acc, mx);
}

// Number of threads of a named-barrier group whose predicate holds (one
// barrier reduction; every thread of the group must call it).
__device__ __forceinline__ int group_count(int bar_id, int nthreads, bool pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.popc.u32 %0, %2, %3, p;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1 : 0), "r"(bar_id), "r"(nthreads)
        : "memory");
    return r;
}

}  // namespace
}  // namespace ssd
