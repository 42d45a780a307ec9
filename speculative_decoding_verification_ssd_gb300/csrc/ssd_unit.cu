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
//  pass 1  (smem)   per-slice online softmax statistics in base 2
//                   (m = max z/tau * log2 e, S = sum 2^(x - m)) of both rows,
//                   or the largest raw (value, id) key for greedy rows;
//  exchange 1       partial statistics merged over distributed shared memory in
//                   rank order (identical result in every CTA);
//  gathers          rank 0 evaluates p_k(x~_k), q_k(x~_k) and the accept test
//                   u_k q < p ([SD] step 3; greedy: x~_k == argmax);
//  pass 2a (smem)   residual w_t = max(0, p_k(t) - q_k(t)) per token: slice mass
//                   Z_c and the thread maxima for the top-F selection;
//  pass 2b (smem)   block top-F_k of the cache scores (only candidates above a
//                   lower bound are materialised);
//  exchange 2       slice masses and top-F lists; each CTA places its own list
//                   entries in the sequence's cache row by global rank;
//  crossing         the CTA holding the CDF crossing u_K Z re-scans its slice
//                   and records the bonus token t_k that the round draws if it
//                   stops at k (inverse CDF over ascending token id);
//  epilogue         the last CTA of the sequence to finish (atomic counter)
//                   scans the accept bits -> a, picks t_a, writes the outputs
//                   and looks (a, t_a) up in the cache segment a.
//
// Operation sources: [SD] "Speculative decoding" (brentwoodlivery.com), "The
// Algorithm (Step-by-Step)" and "Temperature and Sampling"; [WHY] "Why does
// speculative decoding exist?", "How it works" (greedy rule, bonus token);
// [SSD] "Speculative Speculative Decoding" notes (papernotes.org), "关键设计"
// items 1-2 and "整体框架" (cache keys, sigma_{F,C}, hit test).
#include <cooperative_groups.h>

#include <type_traits>

#include "ssd_device.cuh"
#include "ssd_launch.cuh"
#include "ssd_unit.cuh"

namespace cg = cooperative_groups;

namespace ssd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct Xchg {
    Stat st[2];     // partial (target, draft) statistics of this CTA's slice
    uint64_t best;  // largest raw key of the slice (greedy rows, row K)
    float zsum;     // residual mass of the slice
    int flags;
    int skip;
    int nlist;      // entries of this CTA's top-F list (in cand[])
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

template <class D>
__device__ __forceinline__ void load_vec(const unsigned char *buf, int v, float (&z)[D::kVec]) {
    decode_vec<D>(*reinterpret_cast<const uint4 *>(buf + 16 * v), z);
}

// Loads the VEC elements starting at byte `off` of a staged row; `off` is a
// multiple of the element size, and of 16 when `vec16` (the common case where
// both rows of a unit share their 16-byte phase).
template <class D>
__device__ __forceinline__ void load_vec_at(const unsigned char *buf, int off, bool vec16,
                                            float (&z)[D::kVec]) {
    if (vec16) {
        decode_vec<D>(*reinterpret_cast<const uint4 *>(buf + off), z);
        return;
    }
#pragma unroll
    for (int i = 0; i < D::kVec; ++i) {
        if (D::kBytes == 4)
            z[i] = *reinterpret_cast<const float *>(buf + off + 4 * i);
        else
            z[i] = __uint_as_float(
                static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(buf + off + 2 * i)) << 16);
    }
}

// Online base-2 softmax statistics over one vector of values x (masked = -inf).
template <int VEC>
__device__ __forceinline__ void stat_update(Stat &st, const float (&x)[VEC]) {
    float vm = x[0];
#pragma unroll
    for (int i = 1; i < VEC; ++i) vm = fmaxf(vm, x[i]);
    if (vm > st.m) {
        st.S *= ex2(st.m - vm);
        st.m = vm;
    }
    if (st.m != -INFINITY) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc += ex2(x[i] - st.m);
        st.S += acc;
    }
}

}  // namespace

template <class D>
__global__ void __launch_bounds__(kThreads) ssd_unit_kernel(const __grid_constant__ UnitParams P) {
    constexpr int VEC = D::kVec;
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ __align__(16) uint64_t cand[kCandCap];
    __shared__ double dscan[kThreads];
    __shared__ Xchg xc;
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ Stat red_stat[kWarps];
    __shared__ float red_f[kWarps];
    __shared__ uint64_t red_u[kWarps];
    __shared__ int s_cnt;
    __shared__ int s_int[4];
    __shared__ Stat g_stat[2];
    __shared__ uint64_t g_best;
    __shared__ int g_flags, g_skip;
    __shared__ double pm[16];   // per-rank partial masses (crossing search)
    __shared__ double s_cut;

    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x;
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
        shape.l2C = d.C > 0.f ? lg2(d.C) : -INFINITY;
        if (d.C == 1.f) shape.l2C = 0.f;
    }

    // ---- staging ----------------------------------------------------------
    const int lo = min(V, rank * P.slice), hi = min(V, lo + P.slice);
    unsigned char *buf_t = dyn_smem;
    unsigned char *buf_d = dyn_smem + P.row_buf_bytes;
    const unsigned char *tgt_row = static_cast<const unsigned char *>(P.tgt) +
                                   (static_cast<int64_t>(b) * P.tgt_seq_stride +
                                    static_cast<int64_t>(k) * V) * D::kBytes;
    const unsigned char *drf_row =
        pair ? static_cast<const unsigned char *>(P.drf) +
                   (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * V) *
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
    auto load_d = [&](int v, float (&zd)[VEC]) {
        load_vec_at<D>(buf_d, 16 * v + dshift, dshift == 0, zd);
    };
    __syncthreads();  // scalar head/tail stores visible
    if (active) {
        bool ok = mbar_wait_bounded(&bars[0], 0);
        if (need_d) ok = mbar_wait_bounded(&bars[1], 0) && ok;
        if (!ok) atomicOr(&s_int[1], 1);
    }
    __syncthreads();
    if (s_int[1]) flags |= SSD_DEV_TIMEOUT;  // uniform across the CTA

    // ---- pass 1: statistics / raw maxima ----------------------------------
    const bool want_raw = active && (greedy || (rowK && Fk > 0));
    const bool excl = greedy && !rowK;  // greedy rows rank the drafted token last
    Stat st_t{-INFINITY, 0.f}, st_d{-INFINITY, 0.f};
    uint64_t best = 0;
    if (active) {
        auto body = [&](auto full_c, int v) {
            constexpr bool FULL = decltype(full_c)::value;
            const int e0 = sl.ebase + v * VEC;
            float zt[VEC];
            load_vec<D>(buf_t, v, zt);
            if (sampled) {
                float x[VEC];
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const int e = e0 + i;
                    x[i] = (FULL || (e >= lo && e < hi)) ? zt[i] * c : -INFINITY;
                }
                stat_update<VEC>(st_t, x);
            }
            if (want_raw) {
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const int e = e0 + i;
                    if (FULL || (e >= lo && e < hi)) {
                        const uint64_t key = (excl && e == xt) ? excluded_key(e) : make_key(zt[i], e);
                        best = key > best ? key : best;
                    }
                }
            }
            if (pair) {
                float zd[VEC], x[VEC];
                load_d(v, zd);
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const int e = e0 + i;
                    x[i] = (FULL || (e >= lo && e < hi)) ? zd[i] * c + draft_bias(shape, zd[i], e)
                                                         : -INFINITY;
                }
                stat_update<VEC>(st_d, x);
            }
        };
        for (int v = tid; v < sl.nv; v += kThreads) {
            const int e0 = sl.ebase + v * VEC;
            if (e0 >= lo && e0 + VEC <= hi)
                body(std::true_type{}, v);
            else
                body(std::false_type{}, v);
        }
    }
    const uint64_t my_best = best;  // this thread's raw maximum (top-F lower bound)
    st_t = block_stat(st_t, red_stat);
    st_d = block_stat(st_d, red_stat);
    best = block_max_u64(best, red_u);

    // ---- exchange 1 ---------------------------------------------------------
    if (tid == 0) {
        xc.st[0] = st_t;
        xc.st[1] = st_d;
        xc.best = best;
        xc.flags = flags;
        xc.skip = skip;
        xc.zsum = 0.f;
        xc.nlist = 0;
    }
    cluster.sync();
    if (tid == 0) {
        Stat gt{-INFINITY, 0.f}, gd{-INFINITY, 0.f};
        uint64_t gb = 0;
        int gf = 0, gs = 0;
        Stat part[16];
        for (int j = 0; j < CL; ++j) {
            const Xchg *px = cluster.map_shared_rank(&xc, j);
            part[j] = px->st[0];
            gt = stat_merge(gt, part[j]);
            gd = stat_merge(gd, px->st[1]);
            const uint64_t pb = px->best;
            gb = pb > gb ? pb : gb;
            gf |= px->flags;
            gs |= px->skip;
        }
        // target p-mass of each slice relative to the global maximum (crossing search)
        for (int j = 0; j < CL; ++j)
            pm[j] = (part[j].m == -INFINITY)
                        ? 0.0
                        : static_cast<double>(part[j].S) * static_cast<double>(ex2(part[j].m - gt.m));
        g_stat[0] = gt;
        g_stat[1] = gd;
        g_best = gb;
        g_flags = gf;
        g_skip = gs;
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
    if (active && want_raw) {
        const float bv = key_value(g_best);
        if (bv != bv) {
            flags |= SSD_DEV_NONFINITE;
            active = false;
        }
    }

    // ---- gathers and the accept test (rank 0) -------------------------------
    const float invT = active && sampled ? 1.f / gT.S : 0.f;
    const float invD = active && pair ? 1.f / gD.S : 0.f;
    UnitRecord *rec = P.rec + static_cast<int64_t>(b) * (K + 1) + k;
    if (rank == 0 && tid == 0) {
        UnitRecord r{};
        r.flags = flags;
        r.state = skip ? 2 : 1;
        r.tk = -1;
        r.accept = 0;
        r.p_tok = NAN;
        r.q_tok = NAN;
        if (active && !rowK) {
            const float ztx = load_logit<D>(tgt_row, xt);
            if (pair) {
                const float zdx = load_logit<D>(drf_row, xt);
                const float p = ex2(ztx * c - gT.m) / gT.S;
                const float q = ex2(zdx * c + draft_bias(shape, zdx, xt) - gD.m) / gD.S;
                const float u = P.uniforms ? P.uniforms[static_cast<int64_t>(b) * (K + 1) + k] : 0.f;
                r.p_tok = p;
                r.q_tok = q;
                r.accept = (u * q < p) ? 1 : 0;
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
    const bool want_resid = active && pair && (do_verify || Fk > 0);
    float zsum = 0.f;
    uint64_t tbest = 0;
    // gate: p_t > q_t  <=>  (x_p - m_T) - (x_q - m_D) > log2 S_T - log2 S_D
    const float dthr = want_resid ? lg2(gT.S) - lg2(gD.S) : 0.f;
    auto resid = [&](float zt, float zd, int e) -> float {
        const float xp = zt * c - gT.m;
        const float xq = zd * c + draft_bias(shape, zd, e) - gD.m;
        float w = 0.f;
        if (xp - xq > dthr) w = fmaxf(ex2(xp) * invT - ex2(xq) * invD, 0.f);
        return w;
    };
    if (want_resid) {
        float acc[2] = {0.f, 0.f};
        float bs = -1.f;
        int bid = 0;
        auto body = [&](auto full_c, int v) {
            constexpr bool FULL = decltype(full_c)::value;
            const int e0 = sl.ebase + v * VEC;
            float zt[VEC], zd[VEC];
            load_vec<D>(buf_t, v, zt);
            load_d(v, zd);
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                const int e = e0 + i;
                if (FULL || (e >= lo && e < hi)) {
                    const float w = resid(zt[i], zd[i], e);
                    acc[i & 1] += w;
                    if (w > bs) {
                        bs = w;
                        bid = e;
                    }
                }
            }
        };
        for (int v = tid; v < sl.nv; v += kThreads) {
            const int e0 = sl.ebase + v * VEC;
            if (e0 >= lo && e0 + VEC <= hi)
                body(std::true_type{}, v);
            else
                body(std::false_type{}, v);
        }
        zsum = acc[0] + acc[1];
        if (bs >= 0.f) tbest = make_key(bs, bid);
    }
    if (want_resid) zsum = block_sum(zsum, red_f);

    // ---- pass 2b: block top-F_k of the cache scores --------------------------
    int nlist = 0;
    if (active && Fk > 0) {
        if (pair) {
            nlist = block_topf(
                Fk, tbest,
                [&](uint64_t theta, auto emit) {
                    const float ts = key_value(theta);
                    // w_t <= p_t: skip tokens whose p is below the threshold score
                    const float xmin =
                        (theta >> 32) > 0x80000000ull && ts > 0.f ? lg2(ts) + lg2(gT.S) - 1e-3f
                                                                  : -INFINITY;
                    for (int v = tid; v < sl.nv; v += kThreads) {
                        const int e0 = sl.ebase + v * VEC;
                        float zt[VEC];
                        load_vec<D>(buf_t, v, zt);
                        bool any = false;
#pragma unroll
                        for (int i = 0; i < VEC; ++i) any |= (zt[i] * c - gT.m) >= xmin;
                        if (!any) continue;
                        float zd[VEC];
                        load_d(v, zd);
#pragma unroll
                        for (int i = 0; i < VEC; ++i) {
                            const int e = e0 + i;
                            if (e >= lo && e < hi && (zt[i] * c - gT.m) >= xmin) {
                                const uint64_t key = make_key(resid(zt[i], zd[i], e), e);
                                if (key >= theta) emit(key);
                            }
                        }
                    }
                },
                cand, &s_cnt);
        } else {
            // raw target logits: greedy rows (drafted token last) and row K (p_K ranks as z)
            const uint64_t tb = my_best;
            nlist = block_topf(
                Fk, tb,
                [&](uint64_t theta, auto emit) {
                    const uint32_t tv = static_cast<uint32_t>(theta >> 32);
                    for (int v = tid; v < sl.nv; v += kThreads) {
                        const int e0 = sl.ebase + v * VEC;
                        float zt[VEC];
                        load_vec<D>(buf_t, v, zt);
#pragma unroll
                        for (int i = 0; i < VEC; ++i) {
                            const int e = e0 + i;
                            if (e >= lo && e < hi) {
                                const uint64_t key =
                                    (excl && e == xt) ? excluded_key(e) : make_key(zt[i], e);
                                if ((key >> 32) >= tv && key >= theta) emit(key);
                            }
                        }
                    }
                },
                cand, &s_cnt);
        }
    }

    // ---- exchange 2 -----------------------------------------------------------
    if (tid == 0) {
        xc.zsum = zsum;
        xc.nlist = nlist;
    }
    cluster.sync();

    // Cache placement: each CTA ranks its own list entries against every peer list.
    if (active && Fk > 0) {
        int32_t *seg = P.cache_tok + static_cast<int64_t>(b) * P.budget + P.off[k];
        for (int i = tid; i < nlist; i += kThreads) {
            const uint64_t key = cand[i];
            int pos = i;  // entries of my own list above this one
            for (int j = 0; j < CL; ++j) {
                if (j == rank) continue;
                const Xchg *px = cluster.map_shared_rank(&xc, j);
                const uint64_t *pl = cluster.map_shared_rank(cand, j);
                int l = 0, h = px->nlist;  // count entries > key (lists are descending)
                while (l < h) {
                    const int mid = (l + h) >> 1;
                    if (pl[mid] > key)
                        l = mid + 1;
                    else
                        h = mid;
                }
                pos += l;
            }
            if (pos < Fk) seg[pos] = key_id(key);
        }
    }

    // Bonus candidate t_k: inverse CDF at u_K over ascending token id.
    if (active && sampled && do_verify) {
        // weights: residual (pair with positive mass) or p itself (row K, or Z == 0)
        if (tid == 0) {
            double tot_res = 0.0;
            for (int j = 0; j < CL; ++j) {
                const Xchg *px = cluster.map_shared_rank(&xc, j);
                dscan[j] = static_cast<double>(px->zsum);
                tot_res += dscan[j];
            }
            const int use_res = (pair && tot_res > 0.0) ? 1 : 0;
            double tot = 0.0;
            for (int j = 0; j < CL; ++j) {
                if (!use_res) dscan[j] = pm[j];
                tot += dscan[j];
            }
            const double T = static_cast<double>(P.uniforms[static_cast<int64_t>(b) * (K + 1) + K]) * tot;
            int cstar = -1, lastpos = -1;
            double below = 0.0, cut = 0.0;
            for (int j = 0; j < CL; ++j) {
                if (dscan[j] > 0.0) lastpos = j;
                if (cstar < 0 && below + dscan[j] > T) {
                    cstar = j;
                    cut = T - below;
                }
                below += dscan[j];
            }
            if (cstar < 0) {  // T reached the total only through rounding
                cstar = lastpos;
                cut = (lastpos >= 0) ? dscan[lastpos] : 0.0;
            }
            s_int[0] = cstar;
            s_int[1] = use_res;
            s_cut = cut;
        }
        __syncthreads();
        const int cstar = s_int[0];
        const bool use_res = s_int[1] != 0;
        if (rank == cstar) {
            const double cut = s_cut;
            auto weight = [&](float zt, float zd, int e) -> float {
                return use_res ? resid(zt, zd, e) : ex2(zt * c - gT.m);
            };
            // contiguous vector runs per thread so that a prefix over threads is a prefix over ids
            const int G = (sl.nv + kThreads - 1) / kThreads;
            const int v0 = min(sl.nv, tid * G), v1 = min(sl.nv, v0 + G);
            float run = 0.f;
            int lastp = -1;
            for (int v = v0; v < v1; ++v) {
                const int e0 = sl.ebase + v * VEC;
                float zt[VEC], zd[VEC];
                load_vec<D>(buf_t, v, zt);
                if (use_res) load_d(v, zd);
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
            __syncthreads();  // dscan[] reuse
            dscan[tid] = static_cast<double>(run);
            if (tid == 0) s_int[2] = -1;
            __syncthreads();
            int lastmax = static_cast<int>(block_max_u64(static_cast<uint64_t>(lastp + 1), red_u)) - 1;
            if (tid == 0) {
                double acc = 0.0;
                int jstar = -1;
                for (int j = 0; j < kThreads; ++j) {
                    if (acc + dscan[j] > cut) {
                        jstar = j;
                        break;
                    }
                    acc += dscan[j];
                }
                s_int[2] = jstar;
                dscan[0] = acc;  // prefix before jstar
            }
            __syncthreads();
            if (tid == s_int[2]) {
                double acc = dscan[0];
                int pick = -1;
                for (int v = v0; v < v1 && pick < 0; ++v) {
                    const int e0 = sl.ebase + v * VEC;
                    float zt[VEC], zd[VEC];
                    load_vec<D>(buf_t, v, zt);
                    if (use_res) load_d(v, zd);
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
            if (s_int[2] < 0 && tid == 0) rec->tk = lastmax;
        }
    }

    // ---- completion ---------------------------------------------------------
    cluster.sync();  // peers finished reading this CTA's shared memory
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const uint32_t done = atomicAdd(P.seq_count + b, 1u);
        s_int[3] = (done == static_cast<uint32_t>((K + 1) * CL - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (s_int[3] == 0 || tid != 0) return;
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
