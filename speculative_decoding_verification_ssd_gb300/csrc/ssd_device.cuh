// ssd_device.cuh -- device building blocks shared by the libssd kernels (sm_103a).
//
// * inline-PTX wrappers: mbarrier, bulk async copy (cp.async.bulk), ex2/lg2,
//   bounded mbarrier waits;
// * logit decoding from 16-byte smem vectors (fp32 x4, bf16 x8);
// * 64-bit ranking keys: (ordered value bits << 32) | (0xFFFFFFFF - token id),
//   so a larger key ranks first and equal values rank by ascending id;
// * deterministic block reductions and a block bitonic sort.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ssd.h"

namespace ssd {

constexpr int kThreads = 256;              // threads per CTA of every unit kernel
constexpr int kWarps = kThreads / 32;
constexpr int kCandCap = 512;              // candidate buffer entries per CTA (> SSD_MAX_F + 1)
constexpr uint32_t kSpinLimit = 1u << 26;  // bounded mbarrier polls (~seconds), then give up

static_assert(kCandCap > SSD_MAX_F + 1, "candidate buffer must exceed the largest F");
static_assert(kCandCap >= kThreads, "thread-maxima sort reuses the candidate buffer");

// ---------------------------------------------------------------------------
// PTX wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking test of phase `parity` of `bar`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Waits for phase `parity` of `bar`: one non-blocking test, then polls with try_wait
// (each poll may suspend the thread for up to kSuspendHintNs or until the phase completes);
// gives up after limit_ns of wall-clock time (%globaltimer; kWaitLimitNs for
// mbar_wait_suspend) and returns false (the caller records SSD_DEV_TIMEOUT).  A time bound rather than a poll count keeps roles that legitimately
// idle for a long stretch of a large launch from giving up early.  The loop
// lives in one asm block, so the compiler sees no divergent branch around it.
constexpr uint32_t kSuspendHintNs = 200000;
constexpr uint64_t kWaitLimitNs = 4000000000ull;
__device__ __forceinline__ bool mbar_wait_suspend_for(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t"
        ".reg .pred p;\n\t"
        ".reg .u64 t0, t1;\n\t"
        // a phase already complete returns before the timer is read (c4: 109.7 -> 106.5 us)
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "@p bra SSD_DONE;\n\t"
        "mov.u64 t0, %%globaltimer;\n"
        "SSD_WAIT:\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "@p bra SSD_DONE;\n\t"
        "mov.u64 t1, %%globaltimer;\n\t"
        "sub.u64 t1, t1, t0;\n\t"
        "setp.lt.u64 p, t1, %4;\n\t"
        "@p bra SSD_WAIT;\n"
        "SSD_DONE:\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs), "l"(limit_ns)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_wait_suspend(uint64_t *bar, uint32_t parity) {
    return mbar_wait_suspend_for(bar, parity, kWaitLimitNs);
}

// Waits for phase `parity` of `bar` with a bounded number of polls.  Returns
// false if the limit ran out (the caller records SSD_DEV_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i > 64) __nanosleep(64);
    }
    return false;
}

// Bulk asynchronous copy global -> this CTA's shared memory, completing `bytes`
// of transaction count on `bar`.  dst and src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Hardware base-2 exponential / logarithm (MUFU).  ex2(-inf) = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// Logit storage.
// ---------------------------------------------------------------------------
struct F32Tag {
    static constexpr int kBytes = 4;
    static constexpr int kVec = 4;  // elements per 16-byte vector
};
struct BF16Tag {
    static constexpr int kBytes = 2;
    static constexpr int kVec = 8;
};

template <class D>
__device__ __forceinline__ void decode_vec(const uint4 &w, float (&out)[D::kVec]);

template <>
__device__ __forceinline__ void decode_vec<F32Tag>(const uint4 &w, float (&out)[4]) {
    out[0] = __uint_as_float(w.x);
    out[1] = __uint_as_float(w.y);
    out[2] = __uint_as_float(w.z);
    out[3] = __uint_as_float(w.w);
}

template <>
__device__ __forceinline__ void decode_vec<BF16Tag>(const uint4 &w, float (&out)[8]) {
    const uint32_t r[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(r[i] << 16);
        out[2 * i + 1] = __uint_as_float(r[i] & 0xFFFF0000u);
    }
}

template <class D>
__device__ __forceinline__ float load_logit(const void *base, int64_t idx);
template <>
__device__ __forceinline__ float load_logit<F32Tag>(const void *base, int64_t idx) {
    return __ldg(static_cast<const float *>(base) + idx);
}
template <>
__device__ __forceinline__ float load_logit<BF16Tag>(const void *base, int64_t idx) {
    const uint16_t v = __ldg(static_cast<const unsigned short *>(base) + idx);
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

// ---------------------------------------------------------------------------
// Ranking keys.
// ---------------------------------------------------------------------------
// Monotone map of float bits to uint32 (total order; +NaN above +inf).
__device__ __forceinline__ uint32_t ordered_bits(float v) {
    uint32_t u = __float_as_uint(v);
    u = (u == 0x80000000u) ? 0u : u;  // -0 and +0 are the same value: one key, ties by id
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The same map for values that are never -0 (saves the zero test on scans
// over arrays written through canon_zero).
__device__ __forceinline__ uint32_t ordered_bits_nz(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// -0 -> +0 (IEEE: the sum of zeros of opposite sign is +0); other values unchanged.
__device__ __forceinline__ float canon_zero(float v) { return __fadd_rn(v, 0.f); }
__device__ __forceinline__ float value_of_ordered(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ uint64_t make_key(float v, int id) {
    return (static_cast<uint64_t>(ordered_bits(v)) << 32) |
           static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}
// Key of a token ranked below every real value (excluded drafted token).
__device__ __forceinline__ uint64_t excluded_key(int id) {
    return static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}
__device__ __forceinline__ int key_id(uint64_t k) {
    return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFu));
}
__device__ __forceinline__ float key_value(uint64_t k) {
    return value_of_ordered(static_cast<uint32_t>(k >> 32));
}

// ---------------------------------------------------------------------------
// Online softmax statistics (base 2): m = max x, S = sum 2^(x - m).
// ---------------------------------------------------------------------------
struct Stat {
    float m;
    float S;
};
__device__ __forceinline__ Stat stat_merge(Stat a, Stat b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return {m, 0.f};
    const float sa = (a.m == -INFINITY) ? 0.f : a.S * ex2(a.m - m);
    const float sb = (b.m == -INFINITY) ? 0.f : b.S * ex2(b.m - m);
    return {m, sa + sb};
}

// ---------------------------------------------------------------------------
// Deterministic block reductions (fixed shuffle tree, warps merged in order by
// every thread).  `red` is a kWarps-entry shared scratch.  All threads of the
// block must call; the result is returned to every thread.
// ---------------------------------------------------------------------------
__device__ __forceinline__ Stat block_stat(Stat s, Stat *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Stat t{__shfl_xor_sync(0xFFFFFFFFu, s.m, o), __shfl_xor_sync(0xFFFFFFFFu, s.S, o)};
        s = stat_merge(s, t);
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    Stat r = red[0];
    for (int w = 1; w < kWarps; ++w) r = stat_merge(r, red[w]);
    return r;
}

__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < kWarps; ++w) r += red[w];
    return r;
}

__device__ __forceinline__ uint64_t block_max_u64(uint64_t v, uint64_t *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t t = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = t > v ? t : v;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint64_t r = red[0];
    for (int w = 1; w < kWarps; ++w) r = red[w] > r ? red[w] : r;
    return r;
}

// Bitonic sort, descending, of buf[0..n) (n a power of two) by a group of
// kThreads threads: ti is the caller's index in the group and bar() the
// group's barrier.  Ends with a barrier.
struct BlockBar {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

template <class Bar>
__device__ __forceinline__ void group_sort_desc(uint64_t *buf, int n, int ti, const Bar &bar) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = ti; i < n; i += kThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const uint64_t a = buf[i], c = buf[ixj];
                    const bool desc = (i & k) == 0;
                    if (desc ? (a < c) : (a > c)) {
                        buf[i] = c;
                        buf[ixj] = a;
                    }
                }
            }
            bar();
        }
    }
}

// Block-wide form (the whole CTA of kThreads threads).
__device__ __forceinline__ void block_sort_desc(uint64_t *buf, int n) {
    group_sort_desc(buf, n, static_cast<int>(threadIdx.x), BlockBar{});
}

__host__ __device__ __forceinline__ int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

// ---------------------------------------------------------------------------
// Top-F selection by a group of kThreads threads (ti: index in the group,
// bar: the group's barrier); block_topf is the whole-CTA form.
//
// `thread_best` is this thread's largest key over its own elements (0 if it
// has none), or any key at or below it.  `visit(theta, emit)` must call emit(key) for every element of
// the CTA's slice whose key is >= theta (in any order, from any thread).
// On return cand[0..count) holds the CTA's top-min(F, #elements) keys in
// descending order (count is returned to every thread).  F <= SSD_MAX_F + 1.
//
// Method: theta = F-th largest thread maximum is a lower bound on the F-th
// largest key of the slice (F distinct elements reach it); the elements at or
// above theta are gathered and sorted.  If more than kCandCap qualify, theta
// is raised to the F-th largest of the first kCandCap gathered and the gather
// repeats (each round strictly shrinks the qualifying set).
// ---------------------------------------------------------------------------
template <class Visit, class Bar>
__device__ int group_topf(int F, uint64_t thread_best, Visit &&visit, uint64_t *cand, int *cnt,
                          int ti, const Bar &bar) {
    if (F <= 0) return 0;
    // 1. theta from the thread maxima.
    cand[ti] = thread_best;
    for (int i = kThreads + ti; i < kCandCap; i += kThreads) cand[i] = 0;
    bar();
    group_sort_desc(cand, kThreads, ti, bar);
    uint64_t theta = (F <= kThreads) ? cand[F - 1] : 0;
    bar();
    int count = 0;
    for (int round = 0; round < 64; ++round) {
        if (ti == 0) *cnt = 0;
        bar();
        visit(theta, [&](uint64_t key) {
            const int idx = atomicAdd(cnt, 1);
            if (idx < kCandCap) cand[idx] = key;
        });
        bar();
        count = *cnt;
        if (count <= kCandCap) break;
        // Overflow: all kCandCap stored keys are >= theta.
        group_sort_desc(cand, kCandCap, ti, bar);
        theta = cand[F - 1];
        bar();
    }
    if (count > kCandCap) count = kCandCap;  // unreachable for finite slices
    const int n = next_pow2(count < 2 ? 2 : count);
    for (int i = count + ti; i < n; i += kThreads) cand[i] = 0;
    bar();
    group_sort_desc(cand, n, ti, bar);
    return count < F ? count : F;
}

template <class Visit>
__device__ int block_topf(int F, uint64_t thread_best, Visit &&visit, uint64_t *cand, int *cnt) {
    return group_topf(F, thread_best, static_cast<Visit &&>(visit), cand, cnt,
                      static_cast<int>(threadIdx.x), BlockBar{});
}

// Descending bitonic sort of one key per lane across a warp.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, v, j);
            const bool keep_max = ((lane & k) == 0) == ((lane & j) == 0);
            v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
        }
    return v;
}

// Top-F of a CTA (kThreads threads) when few keys reach the F-th largest thread
// maximum: that maximum's ordered value is found bit by bit over its upper 16
// bits with block-wide counts (a lower bound on the F-th largest key), the keys
// at or above it are gathered, and one warp sorts them when at most 32 qualify;
// otherwise the general block_topf runs.  Same contract as block_topf.
template <class Visit>
__device__ int block_topf_fast(int F, uint64_t thread_best, Visit &&visit, uint64_t *cand, int *cnt) {
    if (F <= 0) return 0;
    const uint32_t ob = static_cast<uint32_t>(thread_best >> 32);
    uint32_t T = 0;
    for (int bit = 31; bit >= 16; --bit) {
        const uint32_t c = T | (1u << bit);
        if (__syncthreads_count(ob >= c) >= F) T = c;
    }
    const uint64_t theta = static_cast<uint64_t>(T) << 32;
    if (threadIdx.x == 0) *cnt = 0;
    __syncthreads();
    visit(theta, [&](uint64_t key) {
        const int idx = atomicAdd(cnt, 1);
        if (idx < kCandCap) cand[idx] = key;
    });
    __syncthreads();
    const int count = *cnt;
    if (count > 32) return block_topf(F, thread_best, visit, cand, cnt);
    if (threadIdx.x < 32) {
        const int l = static_cast<int>(threadIdx.x);
        cand[l] = warp_sort_desc(l < count ? cand[l] : 0, l);
    }
    __syncthreads();
    return count < F ? count : F;
}

}  // namespace ssd
