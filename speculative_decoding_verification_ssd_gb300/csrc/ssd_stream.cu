// ssd_stream.cu -- persistent, warp-specialised streaming form of the fused
// verify / cache-build / lookup kernel (sm_103a).
//
// One CTA per SM.  Warp 16 is the producer: it takes units (sequence b,
// position k) from a global counter and streams their logit rows into an
// 8-stage shared-memory ring with cp.async.bulk, each stage guarded by a
// full/empty mbarrier pair.  Warps 0..15 consume the ring one unit at a time:
//
//  pass 1 (HBM)  per 32-token group: the raw maximum (packed, NaN-propagating)
//                and, for sampled rows, the base-2 mass 2^(z c - gmax c) summed
//                over the group (c = log2 e / tau); stored per group in shared
//                memory.  Greedy rows keep only the group maxima (drafted token
//                excluded).  The draft row of a pair folds into running stats.
//  pass 2 (L2)   pair units only (sampled, k < K): the rows are streamed again
//                (the unit was just read, so they hit L2) and each group stores
//                its residual mass sum of max(0, p - q) and its largest residual.
//  tail          from the per-group arrays: row normalisers, the accept test
//                ([SD] step 3), the greedy argmax, the cache top-F_k (groups whose
//                maximum reaches the F-th largest per-thread maximum are
//                expanded into (value, id) keys), and the inverse-CDF bonus
//                t_k at u_K (group prefix in fp64, then one warp re-reads the
//                crossing group).  The last unit of a sequence runs the
//                epilogue (scan -> a, bonus t_a, outputs, cache lookup).
//
// While the consumers work on a unit's tail, the producer is already streaming
// the next unit, so the HBM stream does not stop for the per-unit reductions.
// Used when every row starts on a 16-byte boundary; other layouts go to the
// cluster kernel in ssd_unit.cu.
//
// Operation sources: [SD] "Speculative decoding" (brentwoodlivery.com), "The
// Algorithm (Step-by-Step)" and "Temperature and Sampling"; [WHY] "Why does
// speculative decoding exist?", "How it works"; [SSD] "Speculative Speculative
// Decoding" notes (papernotes.org), "关键设计" items 1-2 and "整体框架".
#include "ssd_device.cuh"
#include "ssd_launch.cuh"
#include "ssd_stream.cuh"
#include "ssd_unit.cuh"
#include "ssd_vec.cuh"

namespace ssd {
namespace {

constexpr int kCW = kStreamConsumerWarps;  // consumer warps
constexpr int kCT = kCW * 32;              // consumer threads
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kCandGroupsCap = 2048;

enum : int { kPassStats = 1, kPassResid = 2, kPassSkip = 3, kPassStop = 4 };

struct Hdr {
    int unit;   // unit index
    int pass;   // kPass*
    int chunk;  // chunk index within the pass
    int nvec;   // 16-byte vectors per row in this stage
    int last;   // last chunk of the pass
};

struct DraftShape {
    bool on;
    float thr;
    int thr_id;
    float l2C;
};

__device__ __forceinline__ float draft_bias(const DraftShape &r, float z, int e) {
    return (r.on && (z > r.thr || (z == r.thr && e <= r.thr_id))) ? r.l2C : 0.f;
}

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"r"(kCT) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
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

// Reductions over the GV lanes that hold one 32-token group (GV divides 32).
template <int GV>
__device__ __forceinline__ float group_max_nan(float v) {
#pragma unroll
    for (int o = 1; o < GV; o <<= 1) v = fmax_nan(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
template <int GV>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = 1; o < GV; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// ---- consumer-wide reductions (512 threads, named barrier 1) ----------------
struct Scratch {
    uint32_t u[kCW];
    float f[kCW];
    double d[kCW];
    uint64_t k[kCW];
    Stat st[kCW];
    int i[4];
    double cut;
    uint64_t bkey;  // greedy argmax key (outside the reductions' slots)
    int bid;
};

__device__ uint32_t c_max_u32(uint32_t v, Scratch &s) {
    v = __reduce_max_sync(kFull, v);
    cbar();
    if ((threadIdx.x & 31) == 0) s.u[threadIdx.x >> 5] = v;
    cbar();
    uint32_t r = s.u[0];
    for (int w = 1; w < kCW; ++w) r = s.u[w] > r ? s.u[w] : r;
    return r;
}

__device__ uint64_t c_max_u64(uint64_t v, Scratch &s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t x = __shfl_xor_sync(kFull, v, o);
        v = x > v ? x : v;
    }
    cbar();
    if ((threadIdx.x & 31) == 0) s.k[threadIdx.x >> 5] = v;
    cbar();
    uint64_t r = s.k[0];
    for (int w = 1; w < kCW; ++w) r = s.k[w] > r ? s.k[w] : r;
    return r;
}

__device__ float c_sum_f32(float v, Scratch &s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    cbar();
    if ((threadIdx.x & 31) == 0) s.f[threadIdx.x >> 5] = v;
    cbar();
    float r = s.f[0];
    for (int w = 1; w < kCW; ++w) r += s.f[w];
    return r;
}

__device__ Stat c_stat(Stat st, Scratch &s) {
    const uint32_t mo = __reduce_max_sync(kFull, ordered_bits(st.m));
    const float M = value_of_ordered(mo);
    float S = (st.m == -INFINITY) ? 0.f : st.S * ex2(st.m - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(kFull, S, o);
    cbar();
    if ((threadIdx.x & 31) == 0) s.st[threadIdx.x >> 5] = {M, M == -INFINITY ? 0.f : S};
    cbar();
    Stat r = s.st[0];
    for (int w = 1; w < kCW; ++w) r = stat_merge(r, s.st[w]);
    return r;
}

// F-th largest (with multiplicity) of the per-thread values v over all
// consumer threads (ordered bits; 0 = none).  tops: kCW * 32 words.
__device__ uint32_t c_fth_largest(uint32_t v, int F, uint32_t *tops, Scratch &s) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int Fw = F < 32 ? F : 32;
    cbar();
    for (int it = 0; it < Fw; ++it) {
        const uint32_t mx = __reduce_max_sync(kFull, v);
        const uint32_t who = __ballot_sync(kFull, v == mx);
        if (lane == __ffs(who) - 1) v = 0;
        if (lane == 0) tops[warp * 32 + it] = mx;
    }
    cbar();
    if (warp == 0) {
        uint32_t vals[kCW];
        const int nq = kCW * Fw;
#pragma unroll
        for (int i = 0; i < kCW; ++i) {
            const int q = lane + 32 * i;
            vals[i] = q < nq ? tops[(q / Fw) * 32 + (q % Fw)] : 0u;
        }
        uint32_t mx = 0;
        for (int it = 0; it < F; ++it) {
            uint32_t lm = vals[0];
#pragma unroll
            for (int i = 1; i < kCW; ++i) lm = vals[i] > lm ? vals[i] : lm;
            mx = __reduce_max_sync(kFull, lm);
            const uint32_t who = __ballot_sync(kFull, lm == mx);
            if (lane == __ffs(who) - 1) {
                bool done = false;
#pragma unroll
                for (int i = 0; i < kCW; ++i)
                    if (!done && vals[i] == mx) {
                        vals[i] = 0;
                        done = true;
                    }
            }
        }
        if (lane == 0) s.u[0] = mx;
    }
    cbar();
    const uint32_t r = s.u[0];
    cbar();
    return r;
}

}  // namespace

template <class D>
__global__ void __launch_bounds__(kStreamThreads, 1)
    ssd_stream_kernel(const __grid_constant__ UnitParams P) {
    constexpr int VEC = D::kVec, S = D::kBytes;
    constexpr int GV = kGroupTokens / VEC;                 // vectors per group
    constexpr int kHalfBytes = kStreamStageBytes / 2;
    constexpr int GPC_PAIR = kHalfBytes / S / kGroupTokens;          // groups per pair chunk
    constexpr int GPC_ONE = kStreamStageBytes / S / kGroupTokens;    // groups per single chunk
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ __align__(8) uint64_t full_bar[kStreamStages], empty_bar[kStreamStages];
    __shared__ Hdr hdr[kStreamStages];
    __shared__ __align__(16) uint64_t cand[kCandCap];
    __shared__ int cgroups[kCandGroupsCap];
    __shared__ uint32_t tops[kCW * 32];
    __shared__ Scratch sc;
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = P.B, K = P.K, V = P.V;
    const int G = (V + kGroupTokens - 1) / kGroupTokens;
    unsigned char *ring = dyn_smem;
    float *gmax = reinterpret_cast<float *>(dyn_smem + kStreamStages * kStreamStageBytes);
    float *gsum = gmax + ((G + 31) & ~31);
    const bool do_verify = (P.mode & kModeVerify) != 0;
    const bool do_cache = (P.mode & kModeCache) != 0;
    const int nunits = B * (K + 1);
    const int64_t row_bytes = static_cast<int64_t>(V) * S;

    if (tid == 0) {
        for (int i = 0; i < kStreamStages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], kCW);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // =========================== producer ===================================
    if (warp == kCW) {
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        int64_t n = 0;  // stages produced
        auto push = [&](const Hdr &h, const unsigned char *src_t, const unsigned char *src_d,
                        uint32_t bytes, bool evict_first) -> bool {
            const int s = static_cast<int>(n % kStreamStages);
            const uint32_t par = static_cast<uint32_t>(((n / kStreamStages) & 1) ^ 1);
            if (!mbar_wait_bounded(&empty_bar[s], par)) return false;
            hdr[s] = h;
            unsigned char *dst = ring + s * kStreamStageBytes;
            const uint32_t tx = bytes * (src_d ? 2u : 1u);
            mbar_arrive_expect_tx(&full_bar[s], tx);
            if (bytes) {
                if (evict_first) {
                    bulk_copy_hint(dst, src_t, bytes, &full_bar[s], pol);
                    if (src_d) bulk_copy_hint(dst + kHalfBytes, src_d, bytes, &full_bar[s], pol);
                } else {
                    bulk_copy_g2s(dst, src_t, bytes, &full_bar[s]);
                    if (src_d) bulk_copy_g2s(dst + kHalfBytes, src_d, bytes, &full_bar[s]);
                }
            }
            ++n;
            return true;
        };
        bool ok = true;
        while (ok) {
            if (atomicAdd(&s_abort, 0)) break;
            const int u = static_cast<int>(atomicAdd(P.unit_counter, 1u));
            if (u >= nunits) break;
            const int k = u / B;
            const int b = static_cast<int>((static_cast<int64_t>(u - k * B) * P.perm_mul) % B);
            const float tau = P.temperature[b];
            const bool sampled = (tau > 0.f) && (tau < INFINITY);
            const bool pair = sampled && k < K;
            const bool p2 = pair && (do_verify || (do_cache && P.F[k] > 0));
            bool skip = false;
            if ((P.mode & kModeEarlyExit) && k > 0) {
                const uint32_t mask = (k >= 32) ? 0xFFFFFFFFu : ((1u << k) - 1u);
                skip = (__ldcg(P.seq_reject + b) & mask) != 0;
            }
            const unsigned char *trow = static_cast<const unsigned char *>(P.tgt) +
                                        (static_cast<int64_t>(b) * P.tgt_seq_stride +
                                         static_cast<int64_t>(k) * V) * S;
            const unsigned char *drow =
                pair ? static_cast<const unsigned char *>(P.drf) +
                           (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * V) * S
                     : nullptr;
            if (skip) {
                ok = push(Hdr{u, kPassSkip, 0, 0, 1}, nullptr, nullptr, 0, false);
                continue;
            }
            const int cb = pair ? kHalfBytes : kStreamStageBytes;
            const int nch = static_cast<int>((row_bytes + cb - 1) / cb);
            for (int pass = kPassStats; pass <= (p2 ? kPassResid : kPassStats) && ok; ++pass) {
                for (int c = 0; c < nch && ok; ++c) {
                    const int64_t off = static_cast<int64_t>(c) * cb;
                    const uint32_t bytes = static_cast<uint32_t>(row_bytes - off < cb ? row_bytes - off : cb);
                    const bool ef = !pair || pass == kPassResid;  // data not read again
                    ok = push(Hdr{u, pass, c, static_cast<int>(bytes / 16), c == nch - 1},
                              trow + off, pair ? drow + off : nullptr, bytes, ef);
                }
            }
        }
        if (ok) push(Hdr{-1, kPassStop, 0, 0, 1}, nullptr, nullptr, 0, false);
        else {
            atomicOr(&s_abort, 1);
            if (P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
        }
        return;
    }

    // =========================== consumers ==================================
    int64_t n = 0;  // stages consumed
    int cur = -1;   // current unit
    // per-unit state (uniform over consumers)
    int b = 0, k = 0, xt = -1, flags = 0, Fk = 0, xmask = -1;
    bool greedy = false, sampled = false, pair = false, rowK = false, active = false, excl = false;
    float c = 0.f;
    DraftShape shape{false, 0.f, 0, 0.f};
    const unsigned char *trow = nullptr, *drow = nullptr;
    Stat st_d{-INFINITY, 0.f};   // running draft statistics (group-leader lanes)
    Stat gT{-INFINITY, 0.f}, gD{-INFINITY, 0.f};
    float LT = 0.f, LD = 0.f;
    float ztx = 0.f, zdx = 0.f, u_k = 0.f;  // gathers (consumer thread 0)
    UnitRecord rec{};

    auto resid1 = [&](float zp, float zq, int e) -> float {
        const float xp = zp * c - LT;
        const float xq = zq * c + draft_bias(shape, zq, e) - LD;
        return xp > xq ? fmaxf(ex2(xp) - ex2(xq), 0.f) : 0.f;
    };

    // ---- unit tail helpers ----------------------------------------------------
    // row normaliser of the target from the group arrays (sampled rows)
    auto target_stats = [&]() {
        uint32_t mo = 0;
        for (int g = tid; g < G; g += kCT) {
            const uint32_t o = ordered_bits(gmax[g]);
            mo = o > mo ? o : mo;
        }
        const float M = value_of_ordered(c_max_u32(mo, sc));
        const float Mc = M * c;
        float s = 0.f;
        if (M == M && M != -INFINITY) {
            for (int g = tid; g < G; g += kCT) {
                const float gm = gmax[g];
                if (gm != -INFINITY) s += gsum[g] * ex2(gm * c - Mc);
            }
        }
        const float Ssum = c_sum_f32(s, sc);
        return Stat{Mc, Ssum};
    };

    // top-F_k of the unit into its cache segment (gmax holds per-group maxima of
    // the scores: residuals for pairs, raw logits otherwise)
    auto top_f = [&]() {
        uint32_t tv = 0;
        for (int g = tid; g < G; g += kCT) {
            const uint32_t o = ordered_bits(gmax[g]);
            tv = o > tv ? o : tv;
        }
        const uint32_t theta_u0 = c_fth_largest(tv, Fk, tops, sc);
        uint64_t theta = static_cast<uint64_t>(theta_u0) << 32;
        if (tid == 0) {
            sc.i[0] = 0;
            sc.i[1] = 0;
        }
        cbar();
        for (int g = tid; g < G; g += kCT) {
            if (ordered_bits(gmax[g]) >= theta_u0) {
                const int idx = atomicAdd(&sc.i[0], 1);
                if (idx < kCandGroupsCap) cgroups[idx] = g;
            }
        }
        cbar();
        const int ncg = sc.i[0];
        const bool all_groups = ncg > kCandGroupsCap;
        const int ngroups = all_groups ? G : ncg;
        int count = 0;
        for (int round = 0; round < 64; ++round) {
            for (int q = warp; q < ngroups; q += kCW) {
                const int g = all_groups ? q : cgroups[q];
                const int e = g * kGroupTokens + lane;
                uint64_t key = 0;
                bool has = false;
                if (e < V) {
                    const float zt = load_logit<D>(trow, e);
                    if (pair) {
                        key = make_key(resid1(zt, load_logit<D>(drow, e), e), e);
                    } else {
                        key = (e == xmask) ? excluded_key(e) : make_key(zt, e);
                    }
                    has = key >= theta;
                }
                if (has) {
                    const int idx = atomicAdd(&sc.i[1], 1);
                    if (idx < kCandCap) cand[idx] = key;
                }
            }
            cbar();
            count = sc.i[1];
            if (count <= kCandCap) break;
            // overflow: raise theta to the F-th largest of the stored keys
            for (int kk = 2; kk <= kCandCap; kk <<= 1) {
                for (int j = kk >> 1; j > 0; j >>= 1) {
                    for (int i = tid; i < kCandCap; i += kCT) {
                        const int ixj = i ^ j;
                        if (ixj > i) {
                            const uint64_t a = cand[i], cc = cand[ixj];
                            const bool desc = (i & kk) == 0;
                            if (desc ? (a < cc) : (a > cc)) {
                                cand[i] = cc;
                                cand[ixj] = a;
                            }
                        }
                    }
                    cbar();
                }
            }
            theta = cand[Fk - 1];
            cbar();
            if (tid == 0) sc.i[1] = 0;
            cbar();
        }
        if (count > kCandCap) count = kCandCap;
        // rank by counting into cand[kCandCap ..]
        uint64_t key = 0;
        int r = 0;
        if (tid < count) {
            key = cand[tid];
            for (int j = 0; j < count; ++j) r += cand[j] > key ? 1 : 0;
        }
        if (tid < count && r < Fk) {
            P.cache_tok[static_cast<int64_t>(b) * P.budget + P.off[k] + r] = key_id(key);
        }
        cbar();
    };

    // inverse-CDF bonus at u_K over ascending token id; weights per group in gsum
    // (residual masses, or p-masses when `pmode`), element weights by `wfn`
    auto crossing = [&](bool pmode, float Mc) {
        // group weights
        const int R = (G + kCT - 1) / kCT;
        const int g0 = min(G, tid * R), g1 = min(G, g0 + R);
        float run = 0.f;
        for (int g = g0; g < g1; ++g) {
            const float gm = gmax[g];
            run += pmode ? ((gm == -INFINITY) ? 0.f : gsum[g] * ex2(gm * c - Mc)) : gsum[g];
        }
        // block exclusive prefix (fp64), warps in order
        double incl = static_cast<double>(run);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        cbar();
        if (lane == 31) sc.d[warp] = incl;
        if (tid == 0) sc.i[2] = kCT;
        cbar();
        double base = 0.0, tot = 0.0;
        for (int w = 0; w < kCW; ++w) {
            if (w < warp) base += sc.d[w];
            tot += sc.d[w];
        }
        const double T = static_cast<double>(P.uniforms[static_cast<int64_t>(b) * (K + 1) + K]) * tot;
        const double before = base + incl - static_cast<double>(run);
        if (run > 0.f && before + static_cast<double>(run) > T) atomicMin(&sc.i[2], tid);
        cbar();
        const int tstar = sc.i[2];
        // the crossing group (or, past the total by rounding, the last group with mass)
        if (tid == tstar) {
            double acc = before;
            int gstar = g1 - 1;
            double cut = 0.0;
            for (int g = g0; g < g1; ++g) {
                const float gm = gmax[g];
                const float wg = pmode ? ((gm == -INFINITY) ? 0.f : gsum[g] * ex2(gm * c - Mc)) : gsum[g];
                if (acc + static_cast<double>(wg) > T) {
                    gstar = g;
                    cut = T - acc;
                    break;
                }
                acc += static_cast<double>(wg);
            }
            sc.i[3] = gstar;
            sc.cut = cut;
        }
        if (tstar == kCT) {  // no crossing: the last group with positive weight
            uint32_t lastg = 0;
            for (int g = tid; g < G; g += kCT) {
                const float gm = gmax[g];
                const float wg = pmode ? ((gm == -INFINITY) ? 0.f : gsum[g] * ex2(gm * c - Mc)) : gsum[g];
                if (wg > 0.f) lastg = static_cast<uint32_t>(g + 1);
            }
            const uint32_t lg = c_max_u32(lastg, sc);
            if (tid == 0) {
                sc.i[3] = lg > 0 ? static_cast<int>(lg) - 1 : 0;
                sc.cut = 1e300;  // past every element: pick the last positive one
            }
        }
        cbar();
        if (warp == 0) {
            const int g = sc.i[3];
            const double cut = sc.cut;
            const int e = g * kGroupTokens + lane;
            float w = 0.f;
            if (e < V) {
                const float zt = load_logit<D>(trow, e);
                if (pmode)
                    w = ex2(zt * c - Mc);
                else
                    w = resid1(zt, load_logit<D>(drow, e), e);
            }
            double cum = static_cast<double>(w);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(kFull, cum, o);
                if (lane >= o) cum += y;
            }
            const uint32_t over = __ballot_sync(kFull, cum > cut && w >= 0.f && e < V);
            const uint32_t pos = __ballot_sync(kFull, w > 0.f && e < V);
            int pick;
            if (over)
                pick = g * kGroupTokens + __ffs(over) - 1;
            else if (pos)
                pick = g * kGroupTokens + 31 - __clz(pos);
            else
                pick = g * kGroupTokens;
            if (lane == 0) rec.tk = pick;
        }
        cbar();
    };

    auto finish_unit = [&]() {
        // record, then count the unit; the sequence's last unit runs the epilogue
        __threadfence();
        cbar();
        if (tid == 0) {
            UnitRecord *R = P.rec + static_cast<int64_t>(b) * (K + 1) + k;
            R->p_tok = rec.p_tok;
            R->q_tok = rec.q_tok;
            R->accept = rec.accept;
            R->tk = rec.tk;
            R->flags = rec.flags;
            R->state = rec.state;
            if (rec.flags == 0 && rec.state == 1 && !rowK && !rec.accept && (P.mode & kModeEarlyExit))
                atomicOr(P.seq_reject + b, 1u << k);
            __threadfence();
            const uint32_t done = atomicAdd(P.seq_count + b, 1u);
            if (done == static_cast<uint32_t>(K)) {
                __threadfence();
                const UnitRecord *RR = P.rec + static_cast<int64_t>(b) * (K + 1);
                int fl = 0;
                for (int i = 0; i <= K; ++i) fl |= __ldcg(&RR[i].flags);
                int a = K;
                for (int i = 0; i < K; ++i) {
                    if (__ldcg(&RR[i].accept) == 0) {
                        a = i;
                        break;
                    }
                }
                const int tstar = __ldcg(&RR[a].tk);
                const bool bad = fl != 0 || tstar < 0;
                if (do_verify) {
                    P.accept_len[b] = bad ? -1 : a;
                    P.bonus[b] = bad ? -1 : tstar;
                    if (P.p_tok) {
                        for (int i = 0; i < K; ++i) {
                            const bool keep = !bad && i <= a;
                            P.p_tok[static_cast<int64_t>(b) * K + i] = keep ? __ldcg(&RR[i].p_tok) : NAN;
                            P.q_tok[static_cast<int64_t>(b) * K + i] = keep ? __ldcg(&RR[i].q_tok) : NAN;
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
        }
        cbar();
    };

    for (;;) {
        const int s = static_cast<int>(n % kStreamStages);
        const uint32_t par = static_cast<uint32_t>((n / kStreamStages) & 1);
        if (!mbar_wait_bounded(&full_bar[s], par)) {
            atomicOr(&s_abort, 1);
            if (tid == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
            break;
        }
        const Hdr h = hdr[s];
        if (h.pass == kPassStop) break;
        if (h.unit != cur) {
            // ---- a new unit: per-unit constants (identical in every consumer) --
            cur = h.unit;
            k = cur / B;
            b = static_cast<int>((static_cast<int64_t>(cur - k * B) * P.perm_mul) % B);
            const float tau = P.temperature[b];
            const bool tau_ok = (tau >= 0.f) && (tau < INFINITY);
            greedy = tau_ok && tau == 0.f;
            sampled = tau_ok && tau > 0.f;
            rowK = (k == K);
            pair = sampled && !rowK;
            flags = tau_ok ? 0 : SSD_DEV_BAD_TEMPERATURE;
            xt = -1;
            if (!rowK) {
                xt = P.tokens[static_cast<int64_t>(b) * K + k];
                if (xt < 0 || xt >= V) flags |= SSD_DEV_BAD_TOKEN;
            }
            excl = greedy && !rowK;
            xmask = excl ? xt : -1;
            Fk = do_cache ? P.F[k] : 0;
            active = flags == 0;
            c = sampled ? kLog2e / tau : 0.f;
            shape = DraftShape{false, 0.f, 0, 0.f};
            if (pair && P.reshape) {
                const ssd_reshape_desc d = P.reshape[static_cast<int64_t>(b) * K + k];
                shape.on = d.F > 0;
                shape.thr = d.thr_val;
                shape.thr_id = d.thr_id;
                shape.l2C = d.C > 0.f ? (d.C == 1.f ? 0.f : lg2(d.C)) : -INFINITY;
            }
            trow = static_cast<const unsigned char *>(P.tgt) +
                   (static_cast<int64_t>(b) * P.tgt_seq_stride + static_cast<int64_t>(k) * V) * S;
            drow = pair ? static_cast<const unsigned char *>(P.drf) +
                              (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * V) * S
                        : nullptr;
            st_d = Stat{-INFINITY, 0.f};
            rec = UnitRecord{};
            rec.tk = -1;
            rec.p_tok = NAN;
            rec.q_tok = NAN;
            rec.state = 1;
            if (tid == 0 && active && !rowK) {
                ztx = load_logit<D>(trow, xt);
                if (pair) {
                    zdx = load_logit<D>(drow, xt);
                    u_k = P.uniforms ? P.uniforms[static_cast<int64_t>(b) * (K + 1) + k] : 0.f;
                }
            }
        }
        const unsigned char *st = ring + s * kStreamStageBytes;
        if (h.pass == kPassSkip) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);
            ++n;
            rec.state = 2;
            rec.flags = flags;
            finish_unit();
            continue;
        }

        // ---- stage processing -----------------------------------------------
        if (active) {
            if (h.pass == kPassStats && pair) {
                const int j = tid;
                const bool ok = j < h.nvec;
                const uint4 wt = ok ? *reinterpret_cast<const uint4 *>(st + 16 * j) : neg_inf_vec<D>();
                const uint4 wd = ok ? *reinterpret_cast<const uint4 *>(st + kHalfBytes + 16 * j)
                                    : neg_inf_vec<D>();
                const int g = h.chunk * GPC_PAIR + j / GV;
                // target: group maximum and mass
                RawMax<D> rm;
                rm.add(wt);
                const float gm = group_max_nan<GV>(rm.get());
                float vs = 0.f;
                if (gm != -INFINITY) {
                    const float2 a = exp_sum<D>(wt, c, gm * c, make_float2(0.f, 0.f));
                    vs = a.x + a.y;
                }
                const float gs = group_sum<GV>(vs);
                const bool leader = (j % GV) == 0;
                if (leader && g < G) {
                    gmax[g] = gm;
                    gsum[g] = gs;
                }
                // draft: fold the group into the running statistics
                if (!shape.on) {
                    RawMax<D> rd;
                    rd.add(wd);
                    const float gmd = group_max_nan<GV>(rd.get());
                    float vd = 0.f;
                    if (gmd != -INFINITY) {
                        const float2 a = exp_sum<D>(wd, c, gmd * c, make_float2(0.f, 0.f));
                        vd = a.x + a.y;
                    }
                    const float gsd = group_sum<GV>(vd);
                    if (leader && gmd != -INFINITY) st_d = stat_merge(st_d, Stat{gmd * c, gsd});
                    if (leader && gmd != gmd) st_d = Stat{NAN, NAN};
                } else {
                    float z[VEC];
                    decode_vec<D>(wd, z);
                    const int e0 = (h.chunk * GPC_PAIR) * kGroupTokens + j * VEC;
                    float x[VEC];
                    float xm = -INFINITY;
#pragma unroll
                    for (int i = 0; i < VEC; ++i) {
                        x[i] = z[i] * c + draft_bias(shape, z[i], e0 + i);
                        xm = fmax_nan(xm, x[i]);
                    }
                    const float gxm = group_max_nan<GV>(xm);
                    float vd = 0.f;
                    if (gxm != -INFINITY) {
#pragma unroll
                        for (int i = 0; i < VEC; ++i) vd += ex2(x[i] - gxm);
                    }
                    const float gsd = group_sum<GV>(vd);
                    if (leader && gxm != -INFINITY) st_d = stat_merge(st_d, Stat{gxm, gsd});
                    if (leader && gxm != gxm) st_d = Stat{NAN, NAN};
                }
            } else if (h.pass == kPassStats) {
                // one row: sampled row K (max + mass) or greedy (max, drafted token excluded)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int j = tid + half * kCT;
                    const bool ok = j < h.nvec;
                    uint4 w = ok ? *reinterpret_cast<const uint4 *>(st + 16 * j) : neg_inf_vec<D>();
                    const int e0 = h.chunk * GPC_ONE * kGroupTokens + j * VEC;
                    if (static_cast<unsigned>(xmask - e0) < static_cast<unsigned>(VEC))
                        mask_vec<D>(w, e0, 0, V, xmask);
                    const int g = h.chunk * GPC_ONE + j / GV;
                    RawMax<D> rm;
                    rm.add(w);
                    const float gm = group_max_nan<GV>(rm.get());
                    float gs = 0.f;
                    if (sampled) {
                        float vs = 0.f;
                        if (gm != -INFINITY) {
                            const float2 a = exp_sum<D>(w, c, gm * c, make_float2(0.f, 0.f));
                            vs = a.x + a.y;
                        }
                        gs = group_sum<GV>(vs);
                    }
                    if ((j % GV) == 0 && g < G) {
                        gmax[g] = gm;
                        gsum[g] = gs;
                    }
                }
            } else {
                // pass 2 (pair): residual masses and maxima per group
                const int j = tid;
                const bool ok = j < h.nvec;
                const uint4 wt = ok ? *reinterpret_cast<const uint4 *>(st + 16 * j) : neg_inf_vec<D>();
                const uint4 wd = ok ? *reinterpret_cast<const uint4 *>(st + kHalfBytes + 16 * j)
                                    : neg_inf_vec<D>();
                float zt[VEC], zd[VEC];
                decode_vec<D>(wt, zt);
                decode_vec<D>(wd, zd);
                const int e0 = (h.chunk * GPC_PAIR) * kGroupTokens + j * VEC;
                float2 acc = make_float2(0.f, 0.f);
                float mx = 0.f;
#pragma unroll
                for (int i = 0; i < VEC; i += 2) {
                    const float w0 = resid1(zt[i], zd[i], e0 + i);
                    const float w1 = resid1(zt[i + 1], zd[i + 1], e0 + i + 1);
                    acc = __fadd2_rn(acc, make_float2(w0, w1));
                    mx = fmaxf(mx, fmaxf(w0, w1));
                }
                const float gs = group_sum<GV>(acc.x + acc.y);
                float gm = mx;
#pragma unroll
                for (int o = 1; o < GV; o <<= 1) gm = fmaxf(gm, __shfl_xor_sync(kFull, gm, o));
                const int g = h.chunk * GPC_PAIR + j / GV;
                if ((j % GV) == 0 && g < G) {
                    gmax[g] = gm;
                    gsum[g] = gs;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        ++n;
        if (!h.last) continue;

        // ---- end of a pass: the unit's tail ----------------------------------
        cbar();  // group arrays complete
        rec.flags = flags;
        const bool want_p2 = pair && (do_verify || Fk > 0);
        if (!active) {
            // an inactive pair still receives its second pass; finish after it
            if (h.pass == kPassResid || !want_p2) finish_unit();
            continue;
        }
        if (h.pass == kPassStats && sampled) {
            gT = target_stats();
            if (pair) gD = c_stat(st_d, sc);
            const bool okT = (gT.m < INFINITY) && (gT.S > 0.f) && (gT.S < INFINITY);
            const bool okD = !pair || ((gD.m < INFINITY) && (gD.S > 0.f) && (gD.S < INFINITY));
            if (!okT || !okD) {
                flags |= SSD_DEV_NONFINITE;
                rec.flags = flags;
                active = false;
                if (!want_p2) finish_unit();
                continue;  // a pair's second pass is still streamed and consumed
            }
            LT = gT.m + lg2(gT.S);
            LD = pair ? gD.m + lg2(gD.S) : 0.f;
            if (pair && tid == 0) {
                const float p = ex2(ztx * c - gT.m) / gT.S;
                const float q = ex2(zdx * c + draft_bias(shape, zdx, xt) - gD.m) / gD.S;
                rec.p_tok = p;
                rec.q_tok = q;
                rec.accept = (u_k * q < p) ? 1 : 0;
            }
            if (pair) {
                if (!want_p2) finish_unit();
                continue;  // pass 2 follows
            }
            // sampled row K: cache from raw maxima, bonus from p_K
            if (Fk > 0) top_f();
            if (do_verify) crossing(true, gT.m);
            finish_unit();
            continue;
        }
        if (h.pass == kPassStats && greedy) {
            // argmax: the best group (lowest index on ties), then the lowest id in it
            uint64_t gk = 0;
            for (int g = tid; g < G; g += kCT) {
                const uint64_t key = (static_cast<uint64_t>(ordered_bits(gmax[g])) << 32) |
                                     static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(g));
                gk = key > gk ? key : gk;
            }
            const uint64_t best = c_max_u64(gk, sc);
            const float M = value_of_ordered(static_cast<uint32_t>(best >> 32));
            const int gbest = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFu));
            if (M != M) {
                flags |= SSD_DEV_NONFINITE;
                rec.flags = flags;
                finish_unit();
                continue;
            }
            if (warp == 0) {
                const int e = gbest * kGroupTokens + lane;
                bool m = false;
                if (e < V && e != xmask) m = load_logit<D>(trow, e) == M;
                const uint32_t who = __ballot_sync(kFull, m);
                const int id = who ? gbest * kGroupTokens + __ffs(who) - 1 : gbest * kGroupTokens;
                if (lane == 0) {
                    sc.bkey = make_key(M, id);
                    sc.bid = id;
                }
            }
            cbar();
            const uint64_t gkey = sc.bkey;
            if (tid == 0) {
                rec.tk = sc.bid;
                if (!rowK) {
                    rec.accept = make_key(ztx, xt) > gkey ? 1 : 0;
                    rec.p_tok = rec.accept ? 1.f : 0.f;
                    rec.q_tok = 1.f;
                }
            }
            cbar();
            if (Fk > 0) top_f();
            finish_unit();
            continue;
        }
        // end of pass 2 (pair): residual mass, cache, bonus
        {
            float zs = 0.f;
            for (int g = tid; g < G; g += kCT) zs += gsum[g];
            const float Z = c_sum_f32(zs, sc);
            if (Fk > 0) top_f();
            if (do_verify) {
                if (Z > 0.f) {
                    crossing(false, 0.f);
                } else {
                    // no residual mass: draw from p at this row (group p-masses again)
                    for (int g = tid; g < G; g += kCT) {
                        float m = -INFINITY;
                        for (int i = 0; i < kGroupTokens; ++i) {
                            const int e = g * kGroupTokens + i;
                            if (e < V) m = fmaxf(m, load_logit<D>(trow, e));
                        }
                        float s2 = 0.f;
                        for (int i = 0; i < kGroupTokens; ++i) {
                            const int e = g * kGroupTokens + i;
                            if (e < V) s2 += ex2(load_logit<D>(trow, e) * c - m * c);
                        }
                        gmax[g] = m;
                        gsum[g] = s2;
                    }
                    cbar();
                    crossing(true, gT.m);
                }
            }
            finish_unit();
        }
    }

    // consumers done: the last CTA to finish resets the unit scheduler
    cbar();
    if (tid == 0) {
        __threadfence();
        const uint32_t done = atomicAdd(P.exit_counter, 1u);
        if (done == gridDim.x - 1) {
            *P.unit_counter = 0;
            *P.exit_counter = 0;
        }
    }
}

int stream_setup(int dtype, size_t optin, size_t *max_dyn) {
    bool dummy = true;
    return dtype == SSD_F32 ? setup_kernel(ssd_stream_kernel<F32Tag>, optin, max_dyn, &dummy)
                            : setup_kernel(ssd_stream_kernel<BF16Tag>, optin, max_dyn, &dummy);
}

int stream_launch(int dtype, const UnitParams &P, int grid, size_t dyn, void *stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.numAttrs = 0;
    const cudaError_t e = dtype == SSD_F32 ? cudaLaunchKernelEx(&cfg, ssd_stream_kernel<F32Tag>, P)
                                           : cudaLaunchKernelEx(&cfg, ssd_stream_kernel<BF16Tag>, P);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SSD_ERR_CUDA;
    }
    return SSD_OK;
}

}  // namespace ssd
