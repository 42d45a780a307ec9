// ssd_unit.cu -- the fused verify-and-sample / Saguaro cache-build kernel (sm_103a).
//
// One *unit* = one (sequence b, position k) pair, k = 0..K, processed by one
// thread-block cluster of CL CTAs.  Units are numbered k-major (u = k B + b),
// so all position-0 units run first and later positions can see an earlier
// rejection (early exit in verify-only mode).
//
// Each CTA of the cluster owns a contiguous slice of the vocabulary.  It stages
// its slice of target row (b, k) -- and of draft row (b, k) when the sequence
// samples (tau > 0) and k < K -- into shared memory with bulk asynchronous
// copies, so every logit byte crosses HBM exactly once:
//
//  pass 1  (smem)   per thread over its own 16-byte vectors: the raw maximum
//                   (packed, NaN-propagating), then the base-2 partial sum
//                   S = sum 2^(z c - m c), c = log2(e) / tau; greedy rows find
//                   the lowest id attaining the maximum instead;
//  exchange 1       partial statistics merged over distributed shared memory in
//                   rank order (bit-identical result in every CTA);
//  accept           rank 0 evaluates p_k(x~_k), q_k(x~_k) and the test u_k q < p
//                   ([SD] step 3; greedy: x~_k outranks every other token);
//  pass 2a (smem)   residual w_t = max(0, p_k(t) - q_k(t)): slice mass Z_c and the
//                   per-thread maximum;
//  pass 2b (smem)   block top-F_k: a lower bound theta on the F-th largest value
//                   (the smallest over warps of each warp's ceil(F/8)-th largest
//                   thread maximum), then only vectors with a lane >= theta are
//                   expanded into (value, id) keys and ranked;
//  exchange 2       slice masses and top-F lists; rank 0 merges the lists by
//                   global rank into the cache row;
//  crossing         the CTA holding the CDF crossing of u_K Z re-scans its slice
//                   and records t_k, the bonus drawn if the round stops at k;
//  epilogue         the last CTA of the sequence (atomic counter) scans the
//                   accept bits -> a, picks t_a, writes the outputs and looks
//                   (a, t_a) up in cache segment a.
//
// Operation sources: [SD] "Speculative decoding" (brentwoodlivery.com), "The
// Algorithm (Step-by-Step)" and "Temperature and Sampling"; [WHY] "Why does
// speculative decoding exist?", "How it works" (greedy rule, bonus token);
// [SSD] "Speculative Speculative Decoding" notes (papernotes.org), "关键设计"
// items 1-2 and "整体框架" (cache keys, sigma_{F,C}, hit test).
#include <cooperative_groups.h>

#include "ssd_device.cuh"
#include "ssd_launch.cuh"
#include "ssd_unit.cuh"
#include "ssd_vec.cuh"

namespace cg = cooperative_groups;

namespace ssd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSortedAt = kThreads;  // rank-sorted candidate lists live at cand[kSortedAt..]
constexpr unsigned kFull = 0xFFFFFFFFu;

struct Xchg {
    Stat st[2];     // partial (target, draft) statistics of this CTA's slice
    uint64_t best;  // largest raw key of the slice (greedy rows)
    float zsum;     // residual mass of the slice
    int flags;
    int skip;
    int nlist;      // entries of this CTA's top-F list
    int list_at;    // offset of the list in cand[]
};

struct Slice {
    int lo, hi;   // vocabulary range [lo, hi) of this CTA
    int ebase;    // token id of smem vector 0, lane 0
    int nv;       // 16-byte vectors covering the slice in smem
};

struct DraftShape {  // sigma_{F,C} membership of the draft row ([SSD] item 2)
    bool on;
    float thr;
    int thr_id;
    float l2C;  // log2 C (-inf for C = 0)
};

__device__ __forceinline__ float draft_bias(const DraftShape &r, float z, int e) {
    return (r.on && (z > r.thr || (z == r.thr && e <= r.thr_id))) ? r.l2C : 0.f;
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Computes the smem placement of row slice [lo, hi) and, when `issue`, starts
// its transfer: the 16-byte-aligned interior by one bulk copy completing on
// `bar`, the unaligned head/tail elements by plain loads.  smem byte 0 maps to
// global byte align_down_16(row + lo).  Requires mbarrier init + sync first.
template <class D>
__device__ Slice stage_row(const void *row, int lo, int hi, unsigned char *buf, uint64_t *bar,
                           bool issue) {
    constexpr int S = D::kBytes, VEC = D::kVec;
    Slice sl;
    sl.lo = lo;
    sl.hi = hi;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(lo) * S;
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(hi) * S;
    const uintptr_t base = a0 & ~static_cast<uintptr_t>(15);
    const int lead = static_cast<int>((a0 - base) / S);
    const int n = hi - lo;
    sl.ebase = lo - lead;
    sl.nv = n > 0 ? (lead + n + VEC - 1) / VEC : 0;
    if (!issue) return sl;
    const uintptr_t c0 = (a0 + 15) & ~static_cast<uintptr_t>(15);
    const uintptr_t c1 = a1 & ~static_cast<uintptr_t>(15);
    uintptr_t h1 = a1, t0 = a1;  // scalar head [a0, h1), scalar tail [t0, a1)
    uint32_t bulk = 0;
    if (n > 0 && c1 > c0) {
        h1 = c0;
        t0 = c1;
        bulk = static_cast<uint32_t>(c1 - c0);
    }
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar, bulk);
        if (bulk) bulk_copy_g2s(buf + (c0 - base), reinterpret_cast<const void *>(c0), bulk, bar);
    }
    const int nh = n > 0 ? static_cast<int>((h1 - a0) / S) : 0;
    const int nt = n > 0 ? static_cast<int>((a1 - t0) / S) : 0;
    for (int i = threadIdx.x; i < nh + nt; i += kThreads) {
        const uintptr_t ga = i < nh ? a0 + static_cast<uintptr_t>(i) * S
                                    : t0 + static_cast<uintptr_t>(i - nh) * S;
        if (S == 4)
            *reinterpret_cast<uint32_t *>(buf + (ga - base)) =
                __ldg(reinterpret_cast<const uint32_t *>(ga));
        else
            *reinterpret_cast<uint16_t *>(buf + (ga - base)) =
                __ldg(reinterpret_cast<const unsigned short *>(ga));
    }
    return sl;
}

__device__ __forceinline__ uint4 ld_vec(const unsigned char *buf, int off) {
    return *reinterpret_cast<const uint4 *>(buf + off);
}

// Loads 16 bytes of a staged row at byte `off` (a multiple of the element size;
// of 16 when `al16`, the common case where both rows share their 16-byte phase).
template <class D>
__device__ __forceinline__ uint4 ld_vec_any(const unsigned char *buf, int off, bool al16) {
    if (al16) return ld_vec(buf, off);
    uint4 w;
    uint32_t *p = reinterpret_cast<uint32_t *>(&w);
    if (D::kBytes == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = *reinterpret_cast<const uint32_t *>(buf + off + 4 * i);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            p[i] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(buf + off + 4 * i)) |
                   (static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(buf + off + 4 * i + 2))
                    << 16);
    }
    return w;
}

// Merges the base-2 softmax statistics held by the lanes of a warp: the maximum
// by an integer reduction of the ordered bits, then every lane rescales its
// sum and the sums are added over a fixed xor tree (the same bits in every
// lane, every CTA).
__device__ __forceinline__ Stat warp_stat(Stat s) {
    const uint32_t mo = __reduce_max_sync(kFull, ordered_bits(s.m));
    const float M = value_of_ordered(mo);
    float S = (s.m == -INFINITY) ? 0.f : s.S * ex2(s.m - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(kFull, S, o);
    return {M, M == -INFINITY ? 0.f : S};
}

// F-th largest (with multiplicity) of the 256 per-thread values v (ordered
// bits; 0 = no element).  `tops` is 256 words of shared scratch and `out` one
// word.  All threads call; returns to every thread.
__device__ uint32_t block_fth_largest(uint32_t v, int F, uint32_t *tops, uint32_t *out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int Fw = F < 32 ? F : 32;
    for (int it = 0; it < Fw; ++it) {  // this warp's Fw largest, in order
        const uint32_t mx = __reduce_max_sync(kFull, v);
        const uint32_t who = __ballot_sync(kFull, v == mx);
        if (lane == __ffs(who) - 1) v = 0;
        if (lane == 0) tops[warp * 32 + it] = mx;
    }
    __syncthreads();
    if (warp == 0) {
        uint32_t vals[kWarps];
        const int nq = kWarps * Fw;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) {
            const int q = lane + 32 * i;
            vals[i] = q < nq ? tops[(q / Fw) * 32 + (q % Fw)] : 0u;
        }
        uint32_t mx = 0;
        for (int it = 0; it < F; ++it) {
            uint32_t lm = vals[0];
#pragma unroll
            for (int i = 1; i < kWarps; ++i) lm = vals[i] > lm ? vals[i] : lm;
            mx = __reduce_max_sync(kFull, lm);
            const uint32_t who = __ballot_sync(kFull, lm == mx);
            if (lane == __ffs(who) - 1) {
                bool done = false;
#pragma unroll
                for (int i = 0; i < kWarps; ++i)
                    if (!done && vals[i] == mx) {
                        vals[i] = 0;
                        done = true;
                    }
            }
        }
        if (lane == 0) *out = mx;
    }
    __syncthreads();
    return *out;
}

// Sorts cand[0..n) (n <= kCandCap) descending.  n <= kThreads: rank by
// counting into cand[kSortedAt..]; otherwise an in-place bitonic sort.  Returns
// the offset of the sorted list.  All threads call; ends synchronised.
__device__ int sort_candidates(uint64_t *cand, int n) {
    if (n <= kThreads) {
        uint64_t key = 0;
        int rank = 0;
        if (threadIdx.x < n) {
            key = cand[threadIdx.x];
            for (int j = 0; j < n; ++j) rank += cand[j] > key ? 1 : 0;
        }
        __syncthreads();
        if (threadIdx.x < n) cand[kSortedAt + rank] = key;
        __syncthreads();
        return kSortedAt;
    }
    const int p2 = next_pow2(n);
    for (int i = n + threadIdx.x; i < p2; i += kThreads) cand[i] = 0;
    __syncthreads();
    block_sort_desc(cand, p2);
    return 0;
}

}  // namespace

template <class D>
__global__ void __launch_bounds__(kThreads, 3) ssd_unit_kernel(const __grid_constant__ UnitParams P) {
    constexpr int VEC = D::kVec;
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ __align__(16) uint64_t cand[kCandCap];
    __shared__ __align__(16) uint64_t mergebuf[kCandCap];
    __shared__ Xchg xc;
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ Stat w_st[2][kWarps];
    __shared__ uint64_t w_key[kWarps];
    __shared__ float w_f[kWarps];
    __shared__ double w_d[kWarps];
    __shared__ uint32_t w_u[kWarps];
    __shared__ int w_i[kWarps];
    __shared__ int s_int[8];
    __shared__ int s_base[16], s_at[16];
    __shared__ Stat g_stat[2];
    __shared__ uint64_t g_best;
    __shared__ int g_flags, g_skip;
    __shared__ double pm[16];   // per-rank p-mass of the target row (crossing search)
    __shared__ double s_cut;

    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int CL = P.CL;
    const int rank = static_cast<int>(cluster.block_rank());
    const int unit = blockIdx.x / CL;
    const int B = P.B, K = P.K, V = P.V;
    const int k = unit / B, b = unit - (unit / B) * B;
    const bool do_verify = (P.mode & kModeVerify) != 0;
    const bool do_cache = (P.mode & kModeCache) != 0;

    // ---- unit description (identical in every CTA of the cluster) --------
    const float tau = P.temperature[b];
    const bool tau_ok = (tau >= 0.f) && (tau < INFINITY);
    const bool greedy = tau_ok && tau == 0.f;
    const bool sampled = tau_ok && tau > 0.f;
    const bool rowK = (k == K);
    const bool pair = sampled && !rowK;
    int xt = -1;
    int flags = tau_ok ? 0 : SSD_DEV_BAD_TEMPERATURE;
    if (!rowK) {
        xt = P.tokens[static_cast<int64_t>(b) * K + k];
        if (xt < 0 || xt >= V) flags |= SSD_DEV_BAD_TOKEN;
    }
    const int Fk = do_cache ? P.F[k] : 0;
    if (tid == 0) {
        int sk = 0;
        if ((P.mode & kModeEarlyExit) && k > 0) {
            const uint32_t mask = (k >= 32) ? 0xFFFFFFFFu : ((1u << k) - 1u);
            sk = (__ldcg(P.seq_reject + b) & mask) ? 1 : 0;
        }
        s_int[0] = sk;
        s_int[1] = 0;  // timeout seen by any thread
    }
    const float c = sampled ? kLog2e / tau : 0.f;  // x = z * c: logits in base-2 units
    DraftShape shape{false, 0.f, 0, 0.f};
    if (pair && P.reshape) {
        const ssd_reshape_desc d = P.reshape[static_cast<int64_t>(b) * K + k];
        shape.on = d.F > 0;
        shape.thr = d.thr_val;
        shape.thr_id = d.thr_id;
        shape.l2C = d.C > 0.f ? (d.C == 1.f ? 0.f : lg2(d.C)) : -INFINITY;
    }

    // ---- staging ----------------------------------------------------------
    const int lo = min(V, rank * P.slice), hi = min(V, lo + P.slice);
    unsigned char *buf_t = dyn_smem;
    unsigned char *buf_d = dyn_smem + P.row_buf_bytes;
    const unsigned char *tgt_row = static_cast<const unsigned char *>(P.tgt) +
                                   (static_cast<int64_t>(b) * P.tgt_seq_stride +
                                    static_cast<int64_t>(k) * P.ld) * D::kBytes;
    const unsigned char *drf_row =
        pair ? static_cast<const unsigned char *>(P.drf) +
                   (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * P.ld) *
                       D::kBytes
             : nullptr;
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    int skip = s_int[0];
    bool active = !skip && flags == 0;
    const bool need_d = active && pair;
    const Slice sl = stage_row<D>(tgt_row, lo, hi, buf_t, &bars[0], active);
    // Draft vectors are addressed in the target's element grid: element e of the
    // draft row sits dshift bytes away from where it would sit in the target grid.
    int dshift = 0;
    if (need_d) {
        const Slice sd = stage_row<D>(drf_row, lo, hi, buf_d, &bars[1], true);
        dshift = (sl.ebase - sd.ebase) * D::kBytes;
    }
    const bool dal = dshift == 0;
    // The accept test's gathers: issued now so their latency hides behind the copy.
    float ztx = 0.f, zdx = 0.f, u_k = 0.f;
    if (rank == 0 && tid == 32 && active && !rowK) {
        ztx = load_logit<D>(tgt_row, xt);
        if (pair) {
            zdx = load_logit<D>(drf_row, xt);
            u_k = P.uniforms ? P.uniforms[static_cast<int64_t>(b) * (K + 1) + k] : 0.f;
        }
    }
    __syncthreads();  // scalar head/tail stores visible
    if (active) {
        bool ok = mbar_wait_bounded(&bars[0], 0);
        if (need_d) ok = mbar_wait_bounded(&bars[1], 0) && ok;
        if (!ok) atomicOr(&s_int[1], 1);
    }
    // Lanes of the edge vectors outside [lo, hi), and the drafted token of a greedy
    // row (ranked last), are overwritten with -inf once, so the passes below read
    // the staged rows without per-vector checks.  A draft row staged with another
    // 16-byte phase than the target keeps per-load masking instead.
    const bool excl = greedy && !rowK;  // greedy rows rank the drafted token last
    const int xmask = excl ? xt : -1;
    if (active && tid < 3 && sl.nv > 0) {
        int v = -1;
        if (tid == 0) v = 0;
        if (tid == 1 && sl.nv > 1) v = sl.nv - 1;
        if (tid == 2 && xmask >= lo && xmask < hi) {
            v = (xmask - sl.ebase) / VEC;
            if (v == 0 || v == sl.nv - 1) v = -1;  // already patched by thread 0 or 1
        }
        if (v >= 0) {
            const int e0 = sl.ebase + v * VEC;
            uint4 w = ld_vec(buf_t, 16 * v);
            mask_vec<D>(w, e0, lo, hi, xmask);
            *reinterpret_cast<uint4 *>(buf_t + 16 * v) = w;
            if (need_d && dshift == 0 && tid < 2) {
                uint4 wd = ld_vec(buf_d, 16 * v);
                mask_vec<D>(wd, e0, lo, hi, -1);
                *reinterpret_cast<uint4 *>(buf_d + 16 * v) = wd;
            }
        }
    }
    __syncthreads();
    if (s_int[1]) flags |= SSD_DEV_TIMEOUT;  // uniform across the CTA

    auto load_t = [&](int v) { return ld_vec(buf_t, 16 * v); };
    auto load_d = [&](int v) {
        if (dal) return ld_vec(buf_d, 16 * v);
        uint4 w = ld_vec_any<D>(buf_d, 16 * v + dshift, false);
        const int e0 = sl.ebase + v * VEC;
        if (e0 < lo || e0 + VEC > hi) mask_vec<D>(w, e0, lo, hi, -1);
        return w;
    };

    // ---- pass 1 -------------------------------------------------------------
    Stat st_t{-INFINITY, 0.f}, st_d{-INFINITY, 0.f};
    uint64_t best = 0;           // greedy: largest (value, lowest id) key of the thread
    float tmax_raw = -INFINITY;  // raw maximum of the thread's target elements
    if (active) {
        RawMax<D> rm;
        for (int v = tid; v < sl.nv; v += kThreads) rm.add(load_t(v));
        tmax_raw = rm.get();
        if (sampled && tmax_raw != -INFINITY) {
            const float mc = tmax_raw * c;
            float2 acc = make_float2(0.f, 0.f);
            for (int v = tid; v < sl.nv; v += kThreads) acc = exp_sum<D>(load_t(v), c, mc, acc);
            st_t = {mc, acc.x + acc.y};
        }
        if (greedy) {
            if (tmax_raw != tmax_raw) {
                best = ~0ull;  // NaN logits: flagged after the merge
            } else {
                // the lowest id attaining the thread maximum
                for (int v = tid; v < sl.nv; v += kThreads) {
                    const uint4 w = load_t(v);
                    if (ge_lanes<D>(w, tmax_raw) == 0) continue;
                    float z[VEC];
                    decode_vec<D>(w, z);
                    const int e0 = sl.ebase + v * VEC;
                    int e = -1;
#pragma unroll
                    for (int i = VEC - 1; i >= 0; --i) {
                        const int ei = e0 + i;
                        if (z[i] == tmax_raw && ei >= lo && ei < hi && ei != xmask) e = ei;
                    }
                    if (e >= 0) {
                        best = make_key(tmax_raw, e);
                        break;
                    }
                }
            }
        }
        if (pair) {
            if (!shape.on) {
                RawMax<D> rd;
                for (int v = tid; v < sl.nv; v += kThreads) rd.add(load_d(v));
                const float dm = rd.get();
                if (dm != -INFINITY) {
                    const float mc = dm * c;
                    float2 acc = make_float2(0.f, 0.f);
                    for (int v = tid; v < sl.nv; v += kThreads)
                        acc = exp_sum<D>(load_d(v), c, mc, acc);
                    st_d = {mc, acc.x + acc.y};
                }
            } else {
                // reshaped draft: x = z c + log2 c_t, maximum over the weighted values
                float xm = -INFINITY;
                for (int v = tid; v < sl.nv; v += kThreads) {
                    float z[VEC];
                    decode_vec<D>(load_d(v), z);
                    const int e0 = sl.ebase + v * VEC;
#pragma unroll
                    for (int i = 0; i < VEC; ++i)
                        xm = fmax_nan(xm, z[i] * c + draft_bias(shape, z[i], e0 + i));
                }
                if (xm != -INFINITY) {
                    float s = 0.f;
                    for (int v = tid; v < sl.nv; v += kThreads) {
                        float z[VEC];
                        decode_vec<D>(load_d(v), z);
                        const int e0 = sl.ebase + v * VEC;
#pragma unroll
                        for (int i = 0; i < VEC; ++i)
                            s += ex2(z[i] * c + draft_bias(shape, z[i], e0 + i) - xm);
                    }
                    st_d = {xm, s};
                }
            }
        }
    }

    // block reduction: statistics of both rows and the greedy key
    st_t = warp_stat(st_t);
    st_d = warp_stat(st_d);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t ob = __shfl_xor_sync(kFull, best, o);
        best = ob > best ? ob : best;
    }
    if (lane == 0) {
        w_st[0][warp] = st_t;
        w_st[1][warp] = st_d;
        w_key[warp] = best;
    }
    __syncthreads();
    if (warp == 0) {
        Stat a{-INFINITY, 0.f}, d{-INFINITY, 0.f};
        uint64_t bb = 0;
        if (lane < kWarps) {
            a = w_st[0][lane];
            d = w_st[1][lane];
            bb = w_key[lane];
        }
        a = warp_stat(a);
        d = warp_stat(d);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t ob = __shfl_xor_sync(kFull, bb, o);
            bb = ob > bb ? ob : bb;
        }
        if (lane == 0) {
            xc.st[0] = a;
            xc.st[1] = d;
            xc.best = bb;
            xc.flags = flags;
            xc.skip = skip;
            xc.zsum = 0.f;
            xc.nlist = 0;
            xc.list_at = 0;
        }
    }

    // ---- exchange 1 ---------------------------------------------------------
    cluster.sync();
    if (warp == 0) {
        Stat a{-INFINITY, 0.f}, d{-INFINITY, 0.f};
        uint64_t pb = 0;
        uint32_t pf = 0, ps = 0;
        if (lane < CL) {
            const Xchg *px = cluster.map_shared_rank(&xc, lane);
            a = px->st[0];
            d = px->st[1];
            pb = px->best;
            pf = static_cast<uint32_t>(px->flags);
            ps = static_cast<uint32_t>(px->skip);
        }
        // every CTA merges the same lanes with the same tree: identical bits
        const Stat gt = warp_stat(a), gd = warp_stat(d);
        uint64_t gb = pb;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t x = __shfl_xor_sync(kFull, gb, o);
            gb = x > gb ? x : gb;
        }
        const uint32_t gf = __reduce_or_sync(kFull, pf);
        const uint32_t gs = __reduce_or_sync(kFull, ps);
        if (lane < CL)
            pm[lane] = (a.m == -INFINITY)
                           ? 0.0
                           : static_cast<double>(a.S) * static_cast<double>(ex2(a.m - gt.m));
        if (lane == 0) {
            g_stat[0] = gt;
            g_stat[1] = gd;
            g_best = gb;
            g_flags = static_cast<int>(gf);
            g_skip = static_cast<int>(gs);
        }
    }
    __syncthreads();
    const Stat gT = g_stat[0], gD = g_stat[1];
    flags |= g_flags;
    skip = g_skip;
    active = !skip && (flags == 0);
    if (active && sampled) {
        const bool okT = (gT.m < INFINITY) && (gT.S > 0.f) && (gT.S < INFINITY);
        const bool okD = !pair || ((gD.m < INFINITY) && (gD.S > 0.f) && (gD.S < INFINITY));
        if (!okT || !okD) {
            flags |= SSD_DEV_NONFINITE;
            active = false;
        }
    }
    if (active && greedy && (g_best == ~0ull || g_best == 0)) {
        flags |= SSD_DEV_NONFINITE;  // NaN logits
        active = false;
    }

    // ---- the accept test (rank 0; thread 32 holds the gathers) --------------
    UnitRecord *rec = P.rec + static_cast<int64_t>(b) * (K + 1) + k;
    if (rank == 0 && tid == 32) {
        UnitRecord r{};
        r.flags = flags;
        r.state = skip ? 2 : 1;
        r.tk = -1;
        r.accept = 0;
        r.p_tok = NAN;
        r.q_tok = NAN;
        if (active && !rowK) {
            if (pair) {
                const float p = ex2(ztx * c - gT.m) / gT.S;
                const float q = ex2(zdx * c + draft_bias(shape, zdx, xt) - gD.m) / gD.S;
                r.p_tok = p;
                r.q_tok = q;
                r.accept = (u_k * q < p) ? 1 : 0;
            } else {  // greedy: accepted iff x~ outranks every other token
                r.accept = make_key(ztx, xt) > g_best ? 1 : 0;
                r.p_tok = r.accept ? 1.f : 0.f;
                r.q_tok = 1.f;
            }
            if (!r.accept && (P.mode & kModeEarlyExit)) atomicOr(P.seq_reject + b, 1u << k);
        }
        if (active && greedy) r.tk = key_id(g_best);
        rec->p_tok = r.p_tok;
        rec->q_tok = r.q_tok;
        rec->accept = r.accept;
        rec->flags = r.flags;
        rec->state = r.state;
        if (!(active && sampled)) rec->tk = r.tk;
    }

    // ---- pass 2a: residual mass and thread maxima (pair units) -------------
    // w_t = 2^(z_p c - L_T) - 2^(z_q c + log2 c_t - L_D) where positive, with
    // L = m + log2 S the base-2 log-normaliser of each row.
    const bool want_resid = active && pair && (do_verify || Fk > 0);
    const float LT = active && sampled ? gT.m + lg2(gT.S) : 0.f;
    const float LD = active && pair ? gD.m + lg2(gD.S) : 0.f;
    auto resid1 = [&](float zp, float zq, int e) -> float {
        const float xp = zp * c - LT;
        const float xq = zq * c + draft_bias(shape, zq, e) - LD;
        return xp > xq ? fmaxf(ex2(xp) - ex2(xq), 0.f) : 0.f;
    };
    float zsum = 0.f;
    float tmax_res = -1.f;
    if (want_resid) {
        float2 acc = make_float2(0.f, 0.f);
        for (int v = tid; v < sl.nv; v += kThreads) {
            float zt[VEC], zd[VEC];
            decode_vec<D>(load_t(v), zt);
            decode_vec<D>(load_d(v), zd);
            const int e0 = sl.ebase + v * VEC;
#pragma unroll
            for (int i = 0; i < VEC; i += 2) {
                const float w0 = resid1(zt[i], zd[i], e0 + i);
                const float w1 = resid1(zt[i + 1], zd[i + 1], e0 + i + 1);
                acc = __fadd2_rn(acc, make_float2(w0, w1));
                tmax_res = fmaxf(tmax_res, fmaxf(w0, w1));
            }
        }
        zsum = acc.x + acc.y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) zsum += __shfl_xor_sync(kFull, zsum, o);
        if (lane == 0) w_f[warp] = zsum;
        __syncthreads();
        zsum = w_f[0];
        for (int w = 1; w < kWarps; ++w) zsum += w_f[w];
    }

    // ---- pass 2b: block top-F_k of the cache scores --------------------------
    int nlist = 0, list_at = 0;
    if (active && Fk > 0) {
        // theta: the F-th largest of the 256 thread maxima (F distinct elements reach it)
        uint32_t tv = 0;  // ordered bits of this thread's maximum (0 = no element)
        if (tid < sl.nv) {
            if (pair)
                tv = tmax_res >= 0.f ? ordered_bits(tmax_res) : 0u;
            else
                tv = ordered_bits(tmax_raw);
        }
        uint32_t theta_u = block_fth_largest(tv, Fk, reinterpret_cast<uint32_t *>(mergebuf), &w_u[0]);
        if (tid == 0) s_int[2] = 0;
        __syncthreads();
        uint64_t theta = static_cast<uint64_t>(theta_u) << 32;
        int count = 0;
        for (int round = 0; round < 64; ++round) {
            if (pair) {
                // w_t <= p_t, so only tokens with z_p >= zthr can reach the threshold
                const bool filt = theta_u > 0x80000000u;  // threshold value > 0
                float zthr = -INFINITY;
                if (filt)
                    zthr = round_down_storage<D>((lg2(value_of_ordered(theta_u)) + LT - 1e-3f) / c -
                                                 1e-3f);
                for (int v = tid; v < sl.nv; v += kThreads) {
                    const uint4 wt = load_t(v);
                    if (filt && ge_lanes<D>(wt, zthr) == 0) continue;
                    float zt[VEC], zd[VEC];
                    decode_vec<D>(wt, zt);
                    decode_vec<D>(load_d(v), zd);
                    const int e0 = sl.ebase + v * VEC;
#pragma unroll
                    for (int i = 0; i < VEC; ++i) {
                        const int e = e0 + i;
                        if (e < lo || e >= hi) continue;
                        const uint64_t key = make_key(resid1(zt[i], zd[i], e), e);
                        if (key >= theta) {
                            const int idx = atomicAdd(&s_int[2], 1);
                            if (idx < kCandCap) cand[idx] = key;
                        }
                    }
                }
            } else {
                const float tval = value_of_ordered(theta_u);
                const bool filt = theta_u >= 0x00800000u;  // a real value (not "none")
                for (int v = tid; v < sl.nv; v += kThreads) {
                    const uint4 wt = ld_vec(buf_t, 16 * v);
                    if (filt && ge_lanes<D>(wt, tval) == 0) continue;
                    float zt[VEC];
                    decode_vec<D>(wt, zt);
                    const int e0 = sl.ebase + v * VEC;
#pragma unroll
                    for (int i = 0; i < VEC; ++i) {
                        const int e = e0 + i;
                        if (e < lo || e >= hi) continue;
                        const uint64_t key = (excl && e == xt) ? excluded_key(e) : make_key(zt[i], e);
                        if (key >= theta) {
                            const int idx = atomicAdd(&s_int[2], 1);
                            if (idx < kCandCap) cand[idx] = key;
                        }
                    }
                }
            }
            __syncthreads();
            count = s_int[2];
            if (count <= kCandCap) break;
            // overflow: every stored key is >= theta; the F-th largest of them is a
            // strictly higher bound, and the qualifying set shrinks every round
            block_sort_desc(cand, kCandCap);
            theta = cand[Fk - 1];
            theta_u = static_cast<uint32_t>(theta >> 32);
            __syncthreads();
            if (tid == 0) s_int[2] = 0;
            __syncthreads();
        }
        if (count > kCandCap) count = kCandCap;
        list_at = sort_candidates(cand, count);
        nlist = count < Fk ? count : Fk;
    }

    // ---- exchange 2 -----------------------------------------------------------
    if (tid == 0) {
        xc.zsum = zsum;
        xc.nlist = nlist;
        xc.list_at = list_at;
    }
    cluster.sync();
    if (warp == 0) {
        float zj = 0.f;
        int nl = 0, la = 0;
        if (lane < CL) {
            const Xchg *px = cluster.map_shared_rank(&xc, lane);
            zj = px->zsum;
            nl = px->nlist;
            la = px->list_at;
        }
        if (active && sampled && do_verify) {
            // crossing of u_K * total over the slices, accumulated in rank order in fp64
            double tr = 0.0;
            for (int j = 0; j < CL; ++j) tr += static_cast<double>(__shfl_sync(kFull, zj, j));
            const bool use_res = pair && tr > 0.0;
            const double part = (lane < CL) ? (use_res ? static_cast<double>(zj) : pm[lane]) : 0.0;
            double tot = 0.0;
            for (int j = 0; j < CL; ++j) tot += __shfl_sync(kFull, part, j);
            const double T = static_cast<double>(P.uniforms[static_cast<int64_t>(b) * (K + 1) + K]) * tot;
            double below = 0.0, cut = 0.0;
            int cstar = -1, lastpos = -1;
            for (int j = 0; j < CL; ++j) {
                const double pj = __shfl_sync(kFull, part, j);
                if (pj > 0.0) lastpos = j;
                if (cstar < 0 && below + pj > T) {
                    cstar = j;
                    cut = T - below;
                }
                below += pj;
            }
            if (cstar < 0) {  // T reached the total only through rounding
                cstar = lastpos;
                cut = lastpos >= 0 ? __shfl_sync(kFull, part, lastpos < 0 ? 0 : lastpos) : 0.0;
            }
            if (lane == 0) {
                s_int[3] = cstar;
                s_int[4] = use_res ? 1 : 0;
                s_cut = cut;
            }
        }
        if (rank == 0 && active && Fk > 0) {
            // exclusive prefix of list sizes over ranks
            int incl = nl;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane < CL) {
                s_base[lane] = incl - nl;
                s_at[lane] = la;
            }
            if (lane == 31) s_int[6] = incl;  // total entries
        }
    }
    __syncthreads();
    // rank 0 gathers every peer list into local memory, then ranks by counting
    if (rank == 0 && active && Fk > 0) {
        const int total = s_int[6];
        int32_t *seg = P.cache_tok + static_cast<int64_t>(b) * P.budget + P.off[k];
        if (total <= kCandCap) {
            for (int i = tid; i < total; i += kThreads) {
                int j = 0;
                while (j + 1 < CL && s_base[j + 1] <= i) ++j;
                const uint64_t *pl = cluster.map_shared_rank(cand, j);
                mergebuf[i] = pl[s_at[j] + (i - s_base[j])];
            }
            __syncthreads();
            for (int i = tid; i < total; i += kThreads) {
                const uint64_t key = mergebuf[i];
                int r = 0;
                for (int j = 0; j < total; ++j) r += mergebuf[j] > key ? 1 : 0;
                if (r < Fk) seg[r] = key_id(key);
            }
        } else {
            // long lists: rank each entry by binary search in every peer list
            for (int j0 = 0; j0 < CL; ++j0) {
                const Xchg *p0 = cluster.map_shared_rank(&xc, j0);
                const uint64_t *l0 = cluster.map_shared_rank(cand, j0) + p0->list_at;
                const int n0 = p0->nlist;
                for (int i = tid; i < n0; i += kThreads) {
                    const uint64_t key = l0[i];
                    int r = i;
                    for (int j = 0; j < CL; ++j) {
                        if (j == j0) continue;
                        const Xchg *pj = cluster.map_shared_rank(&xc, j);
                        const uint64_t *lj = cluster.map_shared_rank(cand, j) + pj->list_at;
                        int l = 0, h = pj->nlist;
                        while (l < h) {
                            const int mid = (l + h) >> 1;
                            if (lj[mid] > key)
                                l = mid + 1;
                            else
                                h = mid;
                        }
                        r += l;
                    }
                    if (r < Fk) seg[r] = key_id(key);
                }
            }
        }
    }
    __syncthreads();
    cluster_arrive();  // this CTA's reads of peer shared memory are complete

    // ---- bonus candidate t_k: inverse CDF at u_K over ascending token id ----
    if (active && sampled && do_verify && rank == s_int[3]) {
        const bool use_res = s_int[4] != 0;
        const double cut = s_cut;
        auto weight = [&](float zt, float zd, int e) -> float {
            return use_res ? resid1(zt, zd, e) : ex2(zt * c - gT.m);
        };
        // contiguous vector runs per thread: a prefix over threads is a prefix over ids
        const int G = (sl.nv + kThreads - 1) / kThreads;
        const int v0 = min(sl.nv, tid * G), v1 = min(sl.nv, v0 + G);
        float run = 0.f;
        int lastp = -1;
        for (int v = v0; v < v1; ++v) {
            float zt[VEC], zd[VEC];
            decode_vec<D>(load_t(v), zt);
            if (use_res) decode_vec<D>(load_d(v), zd);
            const int e0 = sl.ebase + v * VEC;
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                const int e = e0 + i;
                if (e >= lo && e < hi) {
                    const float w = weight(zt[i], use_res ? zd[i] : 0.f, e);
                    run += w;
                    if (w > 0.f) lastp = e;
                }
            }
        }
        // block exclusive prefix of the runs (fp64)
        double incl = static_cast<double>(run);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        int lp = lastp;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(kFull, lp, o));
        if (lane == 31) w_d[warp] = incl;
        if (lane == 0) w_i[warp] = lp;
        if (tid == 0) s_int[5] = kThreads;
        __syncthreads();
        double wbase = 0.0;
        for (int w = 0; w < warp; ++w) wbase += w_d[w];
        int lastmax = -1;
        for (int w = 0; w < kWarps; ++w) lastmax = max(lastmax, w_i[w]);
        const double before = wbase + incl - static_cast<double>(run);
        if (before + static_cast<double>(run) > cut) atomicMin(&s_int[5], tid);
        __syncthreads();
        const int jstar = s_int[5];
        if (tid == jstar) {
            double acc = before;
            int pick = -1;
            for (int v = v0; v < v1 && pick < 0; ++v) {
                float zt[VEC], zd[VEC];
                decode_vec<D>(load_t(v), zt);
                if (use_res) decode_vec<D>(load_d(v), zd);
                const int e0 = sl.ebase + v * VEC;
                for (int i = 0; i < VEC; ++i) {
                    const int e = e0 + i;
                    if (e >= lo && e < hi) {
                        acc += static_cast<double>(weight(zt[i], use_res ? zd[i] : 0.f, e));
                        if (acc > cut) {
                            pick = e;
                            break;
                        }
                    }
                }
            }
            rec->tk = pick >= 0 ? pick : lastmax;
        }
        if (jstar >= kThreads && tid == 0) rec->tk = lastmax;
    }

    // ---- completion ---------------------------------------------------------
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const uint32_t done = atomicAdd(P.seq_count + b, 1u);
        s_int[7] = (done == static_cast<uint32_t>((K + 1) * CL - 1)) ? 1 : 0;
    }
    __syncthreads();
    const bool last = s_int[7] != 0;
    cluster_wait();  // peers finished reading this CTA's shared memory
    if (!last || tid != 0) return;
    __threadfence();

    // ---- epilogue: last CTA of sequence b ------------------------------------
    const UnitRecord *R = P.rec + static_cast<int64_t>(b) * (K + 1);
    int fl = 0;
    for (int i = 0; i <= K; ++i) fl |= __ldcg(&R[i].flags);
    int a = K;
    for (int i = 0; i < K; ++i) {
        if (__ldcg(&R[i].accept) == 0) {
            a = i;
            break;
        }
    }
    const int tstar = __ldcg(&R[a].tk);
    const bool bad = fl != 0 || tstar < 0;
    if (do_verify) {
        P.accept_len[b] = bad ? -1 : a;
        P.bonus[b] = bad ? -1 : tstar;
        if (P.p_tok) {
            for (int i = 0; i < K; ++i) {
                const bool keep = !bad && i <= a;
                P.p_tok[static_cast<int64_t>(b) * K + i] = keep ? __ldcg(&R[i].p_tok) : NAN;
                P.q_tok[static_cast<int64_t>(b) * K + i] = keep ? __ldcg(&R[i].q_tok) : NAN;
            }
        }
        if (P.mode & kModeLookup) {
            int s = -1;
            if (!bad) {
                const int32_t *row = P.cache_tok + static_cast<int64_t>(b) * P.budget;
                for (int j = P.off[a]; j < P.off[a + 1]; ++j) {
                    if (__ldcg(row + j) == tstar) {
                        s = j;
                        break;
                    }
                }
            }
            P.hit[b] = s >= 0 ? 1 : 0;
            P.slot[b] = s;
        }
    }
    if (fl && P.dev_status) atomicOr(P.dev_status, fl);
    P.seq_count[b] = 0;
    P.seq_reject[b] = 0;
}

int unit_setup(int dtype, size_t optin, size_t *max_dyn, bool *allow16) {
    return dtype == SSD_F32 ? setup_kernel(ssd_unit_kernel<F32Tag>, optin, max_dyn, allow16)
                            : setup_kernel(ssd_unit_kernel<BF16Tag>, optin, max_dyn, allow16);
}

int unit_launch(int dtype, const UnitParams &P, int grid, int CL, size_t dyn, void *stream) {
    return dtype == SSD_F32 ? launch_clustered(ssd_unit_kernel<F32Tag>, P, grid, CL, dyn, stream)
                            : launch_clustered(ssd_unit_kernel<BF16Tag>, P, grid, CL, dyn, stream);
}

}  // namespace ssd
