// ssd_stream.cu -- persistent, warp-specialised streaming form of the fused
// verify / cache-build / lookup kernel (sm_103a).
//
// One CTA per SM, four roles:
//   * two producer warps (one elected lane each), one per consumer group: each
//     takes units (sequence b, position k) from a global counter and streams
//     their logit rows with cp.async.bulk into its group's 4-stage shared-memory
//     ring, each stage guarded by a full/empty mbarrier pair.  Units whose
//     sequence samples (temperature > 0) and whose position is below K -- the
//     two-row, two-pass units -- are handed out first, single rows last, so the
//     grid ends on short units;
//   * two consumer groups of 8 warps each, every group working through its
//     own units:
//       pass 1 (HBM)  per 32-token group: the raw maximum and, for sampled
//                     rows, the base-2 mass sum 2^(z c - gmax c) (c = log2 e / tau);
//                     greedy rows keep only group maxima (drafted token
//                     excluded); the draft row of a pair folds into running
//                     statistics;
//       pass 2 (L2)   pair units (sampled, k < K) stream both rows again (they
//                     were just read, so they hit L2): per group the residual
//                     mass sum max(0, p - q) and the largest residual;
//       tail          normalisers, accept test ([SD] step 3), greedy argmax,
//                     cache top-F_k (groups whose maximum reaches the F-th
//                     largest per-thread maximum are expanded into (value, id)
//                     keys), inverse-CDF bonus t_k at u_K;
//   * a finisher warp that takes each unit's record from the groups through a
//     small shared-memory queue, publishes it, counts the sequence's finished
//     units and, for the last unit of a sequence, runs the epilogue (scan -> a,
//     bonus t_a, outputs, cache lookup) with its 32 lanes loading in parallel;
//     the consumer groups never wait on global-memory round trips.
// A thread owns whole 32-token groups (bf16) or halves/quarters of them (fp32,
// second pass), so group reductions need at most two shuffles.
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

constexpr int kGW = kStreamGroupWarps;  // warps per consumer group
constexpr int kGT = kGW * 32;           // threads per consumer group
constexpr int kNG = kStreamGroups;      // consumer groups
constexpr int kRS = kStreamRingStages;  // stages per ring
constexpr int kSB = kStreamStageBytes;  // bytes per stage
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kCandGroupsCap = 512;

enum : int { kPassStats = 1, kPassResid = 2, kPassSkip = 3, kPassStop = 4 };

struct __align__(16) Hdr {
    int unit;   // unit index (changes at every unit)
    int pass;   // kPass*
    int chunk;  // chunk index within the pass
    int nvec;   // 16-byte vectors per row in this stage
    int last;   // last chunk of the pass
    int b, k;   // sequence and position of the unit
    int pair;   // stage layout: 1 = target and draft halves, 0 = one row
};

// A finished unit on its way from a consumer group to the finisher warp.
struct FinEntry {
    UnitRecord rec;
    int b, k;
    int stop;  // 1: the group has no more units
    int pad;
};

constexpr int kFinQ = 4;          // finisher queue entries per consumer group
constexpr int kSchedCap = 2048;   // largest batch ordered by unit kind

struct DraftShape {
    bool on;
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

// Loads the VPT vectors [vbase, vbase + VPT) of a staged row (vectors at or
// past nvec read as -inf), rotated by `rot` so that neighbouring threads hit
// different shared-memory banks.
template <class D, int VPT>
__device__ __forceinline__ void load_vecs(const unsigned char *row, int vbase, int nvec, int rot,
                                          uint4 (&w)[VPT]) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = vbase + ((k + rot) & (VPT - 1));
        w[k] = v < nvec ? *reinterpret_cast<const uint4 *>(row + 16 * v) : neg_inf_vec<D>();
    }
}

template <class D, int VPT>
__device__ __forceinline__ float vecs_max(const uint4 (&w)[VPT]) {
    RawMax<D> rm;
#pragma unroll
    for (int k = 0; k < VPT; ++k) rm.add(w[k]);
    return rm.get();
}

template <class D, int VPT>
__device__ __forceinline__ float vecs_expsum(const uint4 (&w)[VPT], float c, float mc) {
    float2 a = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) a = exp_sum<D>(w[k], c, mc, a);
    return a.x + a.y;
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

// ---- group-wide reductions (one consumer group, named barrier 1 + group) ----
struct Scratch {
    uint32_t u[kGW];
    float f[kGW];
    double d[kGW];
    uint64_t k[kGW];
    Stat st[kGW];
    int i[4];
    double cut;
    uint64_t bkey;
    int bid;
};

struct GroupCtx {
    int bar_id;  // named barrier of the group
    int t;       // thread index within the group
    int lane, warp;
};

__device__ __forceinline__ void gbar(const GroupCtx &g) {
    asm volatile("bar.sync %0, %1;" ::"r"(g.bar_id), "r"(kGT) : "memory");
}

__device__ uint32_t g_max_u32(const GroupCtx &g, uint32_t v, Scratch &s) {
    v = __reduce_max_sync(kFull, v);
    gbar(g);
    if (g.lane == 0) s.u[g.warp] = v;
    gbar(g);
    uint32_t r = s.u[0];
    for (int w = 1; w < kGW; ++w) r = s.u[w] > r ? s.u[w] : r;
    return r;
}

__device__ uint64_t g_max_u64(const GroupCtx &g, uint64_t v, Scratch &s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t x = __shfl_xor_sync(kFull, v, o);
        v = x > v ? x : v;
    }
    gbar(g);
    if (g.lane == 0) s.k[g.warp] = v;
    gbar(g);
    uint64_t r = s.k[0];
    for (int w = 1; w < kGW; ++w) r = s.k[w] > r ? s.k[w] : r;
    return r;
}

__device__ float g_sum_f32(const GroupCtx &g, float v, Scratch &s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    gbar(g);
    if (g.lane == 0) s.f[g.warp] = v;
    gbar(g);
    float r = s.f[0];
    for (int w = 1; w < kGW; ++w) r += s.f[w];
    return r;
}

__device__ Stat g_stat(const GroupCtx &g, Stat st, Scratch &s) {
    const uint32_t mo = __reduce_max_sync(kFull, ordered_bits(st.m));
    const float M = value_of_ordered(mo);
    float S = (st.m == -INFINITY) ? 0.f : st.S * ex2(st.m - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(kFull, S, o);
    gbar(g);
    if (g.lane == 0) s.st[g.warp] = {M, M == -INFINITY ? 0.f : S};
    gbar(g);
    Stat r = s.st[0];
    for (int w = 1; w < kGW; ++w) r = stat_merge(r, s.st[w]);
    return r;
}

// F-th largest (with multiplicity) of the per-thread values v of the group
// (ordered bits; 0 = none).  tops: kGW * 32 words.
__device__ uint32_t g_fth_largest(const GroupCtx &g, uint32_t v, int F, uint32_t *tops, Scratch &s) {
    const int Fw = F < 32 ? F : 32;
    gbar(g);
    for (int it = 0; it < Fw; ++it) {
        const uint32_t mx = __reduce_max_sync(kFull, v);
        const uint32_t who = __ballot_sync(kFull, v == mx);
        if (g.lane == __ffs(who) - 1) v = 0;
        if (g.lane == 0) tops[g.warp * 32 + it] = mx;
    }
    gbar(g);
    if (g.warp == 0) {
        uint32_t vals[kGW];
        const int nq = kGW * Fw;
#pragma unroll
        for (int i = 0; i < kGW; ++i) {
            const int q = g.lane + 32 * i;
            vals[i] = q < nq ? tops[(q / Fw) * 32 + (q % Fw)] : 0u;
        }
        uint32_t mx = 0;
        for (int it = 0; it < F; ++it) {
            uint32_t lm = vals[0];
#pragma unroll
            for (int i = 1; i < kGW; ++i) lm = vals[i] > lm ? vals[i] : lm;
            mx = __reduce_max_sync(kFull, lm);
            const uint32_t who = __ballot_sync(kFull, lm == mx);
            if (g.lane == __ffs(who) - 1) {
                bool done = false;
#pragma unroll
                for (int i = 0; i < kGW; ++i)
                    if (!done && vals[i] == mx) {
                        vals[i] = 0;
                        done = true;
                    }
            }
        }
        if (g.lane == 0) s.u[0] = mx;
    }
    gbar(g);
    const uint32_t r = s.u[0];
    gbar(g);
    return r;
}

// Per consumer group shared state.
struct GroupShared {
    uint64_t full_bar[kRS];
    uint64_t empty_bar[kRS];
    uint64_t fin_full[kFinQ];
    uint64_t fin_empty[kFinQ];
    Hdr hdr[kRS];
    FinEntry fin[kFinQ];
    Scratch sc;
    uint64_t cand[kCandCap];
    int cgroups[kCandGroupsCap];
    uint32_t tops[kGW * 32];
};

}  // namespace

template <class D>
__global__ void __launch_bounds__(kStreamThreads, 1)
    ssd_stream_kernel(const __grid_constant__ UnitParams P) {
    constexpr int VEC = D::kVec, S = D::kBytes;
    constexpr int GV = kGroupTokens / VEC;        // vectors per 32-token group
    constexpr int HALF = kSB / 2;                 // bytes per row in a pair stage
    constexpr int GPR = HALF / 16 / GV;           // groups per row in a pair stage
    constexpr int GPS = kSB / 16 / GV;            // groups in a single-row stage
    constexpr int TPG1 = (kGT / 2) / GPR;         // pass 1 pair: threads per group (per row)
    constexpr int TPGS = kGT / GPS;               // pass 1 single: threads per group
    constexpr int TPG2 = kGT / GPR;               // pass 2: threads per group
    constexpr int VPT1 = GV / TPG1, VPTS = GV / TPGS, VPT2 = GV / TPG2;
    static_assert(VPT1 == 4 && VPTS == 4 && VPT2 == 2, "stage geometry");

    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ GroupShared gsh[kNG];
    __shared__ int s_abort;
    __shared__ int s_nS;
    __shared__ int s_cnt[kSchedCap / 32];
    __shared__ uint16_t sched[kSchedCap];  // sampled sequences, then the others

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = P.B, K = P.K, V = P.V;
    const int G = (V + kGroupTokens - 1) / kGroupTokens;
    const int Gp = (G + 31) & ~31;
    const bool do_verify = (P.mode & kModeVerify) != 0;
    const bool do_cache = (P.mode & kModeCache) != 0;
    const int nunits = B * (K + 1);
    const int64_t row_bytes = static_cast<int64_t>(V) * S;

    if (tid == 0) {
        for (int g = 0; g < kNG; ++g) {
            for (int i = 0; i < kRS; ++i) {
                mbar_init(&gsh[g].full_bar[i], 1);
                mbar_init(&gsh[g].empty_bar[i], kGW);
            }
            for (int i = 0; i < kFinQ; ++i) {
                mbar_init(&gsh[g].fin_full[i], 1);
                mbar_init(&gsh[g].fin_empty[i], 1);
            }
        }
        s_abort = 0;
        s_nS = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Unit order: pair units (sampled sequence, k < K) first, then the sampled
    // rows K, then the other sequences' rows.  Every CTA maps the shared unit
    // counter through this list, so it is built the same way everywhere: a
    // stable compaction in ascending b (per-32 ballots, then chunk prefixes).
    const bool use_list = B <= kSchedCap;
    if (use_list) {
        constexpr int kWarps = kStreamThreads / 32;
        constexpr int kMaxIt = (kSchedCap / 32 + kWarps - 1) / kWarps;
        const int nchunks = (B + 31) / 32;
        uint32_t masks[kMaxIt];
#pragma unroll
        for (int i = 0; i < kMaxIt; ++i) {
            const int c = warp + i * kWarps;
            masks[i] = 0;
            if (c < nchunks) {
                const int b = c * 32 + lane;
                bool smp = false;
                if (b < B) {
                    const float tau = P.temperature[b];
                    smp = tau > 0.f && tau < INFINITY;
                }
                masks[i] = __ballot_sync(kFull, smp);
                if (lane == 0) s_cnt[c] = __popc(masks[i]);
            }
        }
        __syncthreads();
        int tot = 0;
        for (int j = lane; j < nchunks; j += 32) tot += s_cnt[j];
        tot = __reduce_add_sync(kFull, tot);
        if (tid == 0) s_nS = tot;
#pragma unroll
        for (int i = 0; i < kMaxIt; ++i) {
            const int c = warp + i * kWarps;
            if (c < nchunks) {
                int pre = 0;
                for (int j = lane; j < c; j += 32) pre += s_cnt[j];
                pre = __reduce_add_sync(kFull, pre);
                const int b = c * 32 + lane;
                if (b < B) {
                    const int below = __popc(masks[i] & ((1u << lane) - 1u));
                    if ((masks[i] >> lane) & 1u)
                        sched[pre + below] = static_cast<uint16_t>(b);
                    else
                        sched[tot + (c * 32 - pre) + (lane - below)] = static_cast<uint16_t>(b);
                }
            }
        }
    }
    __syncthreads();

    // =========================== producers ==================================
    if (warp >= kNG * kGW && warp < kNG * kGW + kNG) {
        if (lane != 0) return;
        const int rg = warp - kNG * kGW;  // ring served by this producer
        GroupShared &gq = gsh[rg];
        unsigned char *ring = dyn_smem + rg * kRS * kSB;
        const uint64_t pol = policy_evict_first();
        const int nS = s_nS;
        const int nG = B - nS;
        auto unit_bk = [&](int u, int &b, int &k) {
            if (use_list) {
                const int np = nS * K;
                if (u < np) {
                    k = u / nS;
                    b = sched[u - k * nS];
                    return;
                }
                int v = u - np;
                if (v < nS) {
                    k = K;
                    b = sched[v];
                    return;
                }
                v -= nS;
                k = v / nG;
                b = sched[nS + v - k * nG];
            } else {
                k = u / B;
                b = static_cast<int>((static_cast<int64_t>(u - k * B) * P.perm_mul) % B);
            }
        };
        // The next unit is claimed and its metadata loaded while the current
        // unit's last stages are issued, so neither round trip stalls the ring.
        int pf_state = 0, pf_u = 0, pf_b = 0, pf_k = 0;
        float pf_tau = 0.f;
        uint32_t pf_rej = 0;
        auto pf_step = [&]() {
            if (pf_state == 0) {
                pf_u = static_cast<int>(atomicAdd(P.unit_counter, 1u));
                pf_state = 1;
            } else if (pf_state == 1) {
                if (pf_u < nunits) {
                    unit_bk(pf_u, pf_b, pf_k);
                    pf_tau = P.temperature[pf_b];
                    pf_rej = (P.mode & kModeEarlyExit) ? __ldcg(P.seq_reject + pf_b) : 0u;
                }
                pf_state = 2;
            }
        };
        uint32_t n = 0;  // stages pushed
        bool ok = true;
        for (;;) {
            while (pf_state < 2) pf_step();
            pf_state = 0;
            const int u = pf_u;
            if (u >= nunits) {
                const int s = static_cast<int>(n % kRS);
                if (!mbar_wait_bounded(&gq.empty_bar[s], ((n / kRS) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                gq.hdr[s] = Hdr{-1, kPassStop, 0, 0, 1, 0, 0, 0};
                mbar_arrive_expect_tx(&gq.full_bar[s], 0);
                break;
            }
            const int b = pf_b, k = pf_k;
            const float tau = pf_tau;
            const bool sampled = (tau > 0.f) && (tau < INFINITY);
            const bool pair = sampled && k < K;
            const bool p2 = pair && (do_verify || (do_cache && P.F[k] > 0));
            const uint32_t mask = (k >= 32) ? 0xFFFFFFFFu : ((1u << k) - 1u);
            const bool skip = (P.mode & kModeEarlyExit) && k > 0 && (pf_rej & mask) != 0;
            const unsigned char *trow = static_cast<const unsigned char *>(P.tgt) +
                                        (static_cast<int64_t>(b) * P.tgt_seq_stride + static_cast<int64_t>(k) * V) * S;
            const unsigned char *drow =
                pair ? static_cast<const unsigned char *>(P.drf) +
                           (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * V) * S
                     : nullptr;
            const int cb = pair ? HALF : kSB;
            const int nch = static_cast<int>((row_bytes + cb - 1) / cb);
            const int total = skip ? 1 : nch * (p2 ? 2 : 1);
            for (int i = 0; i < total; ++i) {
                const int s = static_cast<int>(n % kRS);
                if (!mbar_wait_bounded(&gq.empty_bar[s], ((n / kRS) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                if (skip) {
                    gq.hdr[s] = Hdr{u, kPassSkip, 0, 0, 1, b, k, 0};
                    mbar_arrive_expect_tx(&gq.full_bar[s], 0);
                } else {
                    const bool second = i >= nch;
                    const int chunk = second ? i - nch : i;
                    const int64_t off = static_cast<int64_t>(chunk) * cb;
                    const uint32_t bytes = static_cast<uint32_t>(row_bytes - off < cb ? row_bytes - off : cb);
                    gq.hdr[s] = Hdr{u, second ? kPassResid : kPassStats, chunk, static_cast<int>(bytes / 16),
                                    chunk == nch - 1, b, k, pair ? 1 : 0};
                    unsigned char *dst = ring + s * kSB;
                    mbar_arrive_expect_tx(&gq.full_bar[s], bytes * (pair ? 2u : 1u));
                    if (!pair || second) {  // not read again
                        bulk_copy_hint(dst, trow + off, bytes, &gq.full_bar[s], pol);
                        if (pair) bulk_copy_hint(dst + HALF, drow + off, bytes, &gq.full_bar[s], pol);
                    } else {
                        bulk_copy_g2s(dst, trow + off, bytes, &gq.full_bar[s]);
                        bulk_copy_g2s(dst + HALF, drow + off, bytes, &gq.full_bar[s]);
                    }
                }
                ++n;
                if (total - i <= 3) pf_step();
            }
            if (!ok) break;
        }
        if (!ok) {
            atomicOr(&s_abort, 1);
            if (P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
        }
        return;
    }

    // =========================== finisher ===================================
    if (warp == kNG * kGW + kNG) {
        uint32_t nf[kNG];
        bool stopped[kNG];
#pragma unroll
        for (int g = 0; g < kNG; ++g) {
            nf[g] = 0;
            stopped[g] = false;
        }
        int idle = 0;
        for (;;) {
            bool all = true, progress = false;
#pragma unroll
            for (int g = 0; g < kNG; ++g) {
                if (stopped[g]) continue;
                all = false;
                const uint32_t qi = nf[g] % kFinQ;
                const uint32_t par = (nf[g] / kFinQ) & 1;
                const bool ready = __all_sync(kFull, mbar_test_wait(&gsh[g].fin_full[qi], par));
                if (!ready) continue;
                progress = true;
                const FinEntry E = gsh[g].fin[qi];
                __syncwarp();
                if (lane == 0) mbar_arrive(&gsh[g].fin_empty[qi]);
                ++nf[g];
                if (E.stop) {
                    stopped[g] = true;
                    continue;
                }
                const int b = E.b, k = E.k;
                if (lane == 0) {
                    UnitRecord *R = P.rec + static_cast<int64_t>(b) * (K + 1) + k;
                    *R = E.rec;
                    if (E.rec.flags == 0 && E.rec.state == 1 && k < K && !E.rec.accept &&
                        (P.mode & kModeEarlyExit))
                        atomicOr(P.seq_reject + b, 1u << k);
                }
                // The record and the group's cache writes (ordered before the
                // queue entry) become visible before the unit is counted.
                __threadfence();
                uint32_t done = 0;
                if (lane == 0) done = atomicAdd(P.seq_count + b, 1u);
                done = __shfl_sync(kFull, done, 0);
                if (done != static_cast<uint32_t>(K)) continue;
                // last unit of sequence b: the epilogue, lanes loading in parallel
                __threadfence();
                const UnitRecord *RR = P.rec + static_cast<int64_t>(b) * (K + 1);
                int fl = 0, acc = 1, tk = -1;
                float pt = NAN, qt = NAN;
                if (lane < K) {
                    fl = __ldcg(&RR[lane].flags);
                    acc = __ldcg(&RR[lane].accept);
                    tk = __ldcg(&RR[lane].tk);
                    pt = __ldcg(&RR[lane].p_tok);
                    qt = __ldcg(&RR[lane].q_tok);
                }
                const int flK = __ldcg(&RR[K].flags);
                const int tkK = __ldcg(&RR[K].tk);
                fl = static_cast<int>(__reduce_or_sync(kFull, static_cast<unsigned>(fl))) | flK;
                const uint32_t rej = __ballot_sync(kFull, lane < K && acc == 0);
                const int a = rej ? __ffs(rej) - 1 : K;
                const int tsh = __shfl_sync(kFull, tk, a & 31);
                const int tstar = a == K ? tkK : tsh;
                const bool bad = fl != 0 || tstar < 0;
                if (do_verify) {
                    if (lane == 0) {
                        P.accept_len[b] = bad ? -1 : a;
                        P.bonus[b] = bad ? -1 : tstar;
                    }
                    if (P.p_tok && lane < K) {
                        const bool keep = !bad && lane <= a;
                        P.p_tok[static_cast<int64_t>(b) * K + lane] = keep ? pt : NAN;
                        P.q_tok[static_cast<int64_t>(b) * K + lane] = keep ? qt : NAN;
                    }
                    if (P.mode & kModeLookup) {
                        int slot = -1;
                        if (!bad) {
                            const int32_t *row = P.cache_tok + static_cast<int64_t>(b) * P.budget;
                            for (int j0 = P.off[a]; j0 < P.off[a + 1] && slot < 0; j0 += 32) {
                                const int j = j0 + lane;
                                const bool m = j < P.off[a + 1] && __ldcg(row + j) == tstar;
                                const uint32_t mm = __ballot_sync(kFull, m);
                                if (mm) slot = j0 + __ffs(mm) - 1;
                            }
                        }
                        if (lane == 0) {
                            P.hit[b] = slot >= 0 ? 1 : 0;
                            P.slot[b] = slot;
                        }
                    }
                }
                if (lane == 0) {
                    if (fl && P.dev_status) atomicOr(P.dev_status, fl);
                    P.seq_count[b] = 0;
                    P.seq_reject[b] = 0;
                }
            }
            if (all) break;
            if (progress) {
                idle = 0;
            } else {
                if (++idle > (1 << 24)) {
                    if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
                    break;
                }
                __nanosleep(64);
            }
        }
        // this CTA is done; the last CTA of the grid resets the unit scheduler
        if (lane == 0) {
            __threadfence();
            const uint32_t done = atomicAdd(P.exit_counter, 1u);
            if (done == gridDim.x - 1) {
                *P.unit_counter = 0;
                *P.exit_counter = 0;
            }
        }
        return;
    }

    // =========================== consumers ==================================
    const int grp = warp / kGW;
    GroupShared &gs = gsh[grp];
    Scratch &sc = gs.sc;
    GroupCtx gc{1 + grp, tid - grp * kGT, lane, warp - grp * kGW};
    const int t = gc.t;
    unsigned char *ring = dyn_smem + grp * kRS * kSB;
    float *gmax = reinterpret_cast<float *>(dyn_smem + kNG * kRS * kSB) + grp * 2 * Gp;
    float *gsum = gmax + Gp;

    int64_t n = 0;  // stages consumed
    int cur = -1;
    int b = 0, k = 0, xt = -1, flags = 0, Fk = 0, xmask = -1;
    bool greedy = false, sampled = false, pair = false, rowK = false, active = false;
    float c = 0.f;
    DraftShape shape{false, 0.f, 0, 0.f};
    const unsigned char *trow = nullptr, *drow = nullptr;
    Stat st_d{-INFINITY, 0.f};
    Stat gT{-INFINITY, 0.f}, gD{-INFINITY, 0.f};
    float LT = 0.f, LD = 0.f;
    float ztx = 0.f, zdx = 0.f, u_k = 0.f;
    UnitRecord rec{};

    auto resid_e = [&](float zp, float zq, int e) -> float {
        return resid_of(zp, zq, c, -LT, draft_bias(shape, zq, e) - LD);
    };

    // normaliser of the target row from the group arrays
    auto target_stats = [&]() -> Stat {
        uint32_t mo = 0;
        for (int g = t; g < G; g += kGT) {
            const uint32_t o = ordered_bits(gmax[g]);
            mo = o > mo ? o : mo;
        }
        const float M = value_of_ordered(g_max_u32(gc, mo, sc));
        const float Mc = M * c;
        float s = 0.f;
        if (M == M && M != -INFINITY) {
            for (int g = t; g < G; g += kGT) {
                const float gm = gmax[g];
                if (gm != -INFINITY) s += gsum[g] * ex2(gm * c - Mc);
            }
        }
        return Stat{Mc, g_sum_f32(gc, s, sc)};
    };

    // top-F_k of the unit into its cache segment (gmax: per-group maxima of the
    // scores -- residuals for pairs, raw logits otherwise)
    auto top_f = [&]() {
        uint32_t tv = 0;
        for (int g = t; g < G; g += kGT) {
            const uint32_t o = ordered_bits(gmax[g]);
            tv = o > tv ? o : tv;
        }
        const uint32_t theta_u0 = g_fth_largest(gc, tv, Fk, gs.tops, sc);
        uint64_t theta = static_cast<uint64_t>(theta_u0) << 32;
        if (t == 0) {
            sc.i[0] = 0;
            sc.i[1] = 0;
        }
        gbar(gc);
        for (int g = t; g < G; g += kGT) {
            if (ordered_bits(gmax[g]) >= theta_u0) {
                const int idx = atomicAdd(&sc.i[0], 1);
                if (idx < kCandGroupsCap) gs.cgroups[idx] = g;
            }
        }
        gbar(gc);
        const int ncg = sc.i[0];
        const bool all_groups = ncg > kCandGroupsCap;
        const int ngroups = all_groups ? G : ncg;
        int count = 0;
        for (int round = 0; round < 64; ++round) {
            for (int q = gc.warp; q < ngroups; q += kGW) {
                const int g = all_groups ? q : gs.cgroups[q];
                const int e = g * kGroupTokens + lane;
                bool has = false;
                uint64_t key = 0;
                if (e < V) {
                    const float zt = load_logit<D>(trow, e);
                    if (pair)
                        key = make_key(resid_e(zt, load_logit<D>(drow, e), e), e);
                    else
                        key = (e == xmask) ? excluded_key(e) : make_key(zt, e);
                    has = key >= theta;
                }
                if (has) {
                    const int idx = atomicAdd(&sc.i[1], 1);
                    if (idx < kCandCap) gs.cand[idx] = key;
                }
            }
            gbar(gc);
            count = sc.i[1];
            if (count <= kCandCap) break;
            // overflow: raise theta to the F-th largest of the stored keys
            for (int kk = 2; kk <= kCandCap; kk <<= 1) {
                for (int j = kk >> 1; j > 0; j >>= 1) {
                    for (int i = t; i < kCandCap; i += kGT) {
                        const int ixj = i ^ j;
                        if (ixj > i) {
                            const uint64_t a = gs.cand[i], cc2 = gs.cand[ixj];
                            const bool desc = (i & kk) == 0;
                            if (desc ? (a < cc2) : (a > cc2)) {
                                gs.cand[i] = cc2;
                                gs.cand[ixj] = a;
                            }
                        }
                    }
                    gbar(gc);
                }
            }
            theta = gs.cand[Fk - 1];
            gbar(gc);
            if (t == 0) sc.i[1] = 0;
            gbar(gc);
        }
        if (count > kCandCap) count = kCandCap;
        // rank by counting; ranks below F go straight to the cache row
        for (int i = t; i < count; i += kGT) {
            const uint64_t key = gs.cand[i];
            int rr = 0;
            for (int j = 0; j < count; ++j) rr += gs.cand[j] > key ? 1 : 0;
            if (rr < Fk) {
                P.cache_tok[static_cast<int64_t>(b) * P.budget + P.off[k] + rr] = key_id(key);
            }
        }
        gbar(gc);
    };

    // inverse-CDF bonus at u_K over ascending token id; per-group weights from
    // gsum (residual masses) or, when `pmode`, p-masses gsum * 2^(gmax c - Mc)
    auto crossing = [&](bool pmode, float Mc) {
        const int R = (G + kGT - 1) / kGT;
        const int g0 = min(G, t * R), g1 = min(G, g0 + R);
        auto gweight = [&](int g) -> float {
            if (!pmode) return gsum[g];
            const float gm = gmax[g];
            return (gm == -INFINITY) ? 0.f : gsum[g] * ex2(gm * c - Mc);
        };
        float run = 0.f;
        for (int g = g0; g < g1; ++g) run += gweight(g);
        double incl = static_cast<double>(run);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        gbar(gc);
        if (lane == 31) sc.d[gc.warp] = incl;
        if (t == 0) sc.i[2] = kGT;
        gbar(gc);
        double base = 0.0, tot = 0.0;
        for (int w = 0; w < kGW; ++w) {
            if (w < gc.warp) base += sc.d[w];
            tot += sc.d[w];
        }
        const double T = static_cast<double>(P.uniforms[static_cast<int64_t>(b) * (K + 1) + K]) * tot;
        const double before = base + incl - static_cast<double>(run);
        if (run > 0.f && before + static_cast<double>(run) > T) atomicMin(&sc.i[2], t);
        gbar(gc);
        const int tstar = sc.i[2];
        if (t == tstar) {
            double acc = before;
            int gstar = g1 - 1;
            double cut = 0.0;
            for (int g = g0; g < g1; ++g) {
                const float wg = gweight(g);
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
        if (tstar == kGT) {  // past the total only through rounding: last group with mass
            uint32_t lastg = 0;
            for (int g = t; g < G; g += kGT)
                if (gweight(g) > 0.f) lastg = static_cast<uint32_t>(g + 1);
            const uint32_t lg = g_max_u32(gc, lastg, sc);
            if (t == 0) {
                sc.i[3] = lg > 0 ? static_cast<int>(lg) - 1 : 0;
                sc.cut = 1e300;
            }
        }
        gbar(gc);
        if (gc.warp == 0) {
            const int g = sc.i[3];
            const double cut = sc.cut;
            const int e = g * kGroupTokens + lane;
            float w = 0.f;
            if (e < V) {
                const float zt = load_logit<D>(trow, e);
                w = pmode ? ex2(fmaf(zt, c, -Mc)) : resid_e(zt, load_logit<D>(drow, e), e);
            }
            double cum = static_cast<double>(w);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(kFull, cum, o);
                if (lane >= o) cum += y;
            }
            const uint32_t over = __ballot_sync(kFull, cum > cut && e < V);
            const uint32_t pos = __ballot_sync(kFull, w > 0.f && e < V);
            int pick;
            if (over)
                pick = g * kGroupTokens + __ffs(over) - 1;
            else if (pos)
                pick = g * kGroupTokens + 31 - __clz(pos);
            else
                pick = g * kGroupTokens;
            if (lane == 0) sc.bid = pick;
        }
        gbar(gc);
        if (t == 0) rec.tk = sc.bid;
    };

    uint32_t nfin = 0;  // entries handed to the finisher (uniform in the group)
    auto push_fin = [&](int stop) {
        if (t == 0) {
            const uint32_t qi = nfin % kFinQ;
            if (mbar_wait_bounded(&gs.fin_empty[qi], ((nfin / kFinQ) & 1) ^ 1)) {
                FinEntry &E = gs.fin[qi];
                E.rec = rec;
                E.b = b;
                E.k = k;
                E.stop = stop;
                mbar_arrive(&gs.fin_full[qi]);
            } else {
                atomicOr(&s_abort, 1);
                if (P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
            }
        }
        ++nfin;
    };
    // the unit is complete: hand its record to the finisher (the barrier orders
    // every thread's cache writes before the hand-off)
    auto finish_unit = [&]() {
        gbar(gc);
        push_fin(0);
    };

    for (;;) {
        const int s = static_cast<int>(n % kRS);
        const uint32_t par = static_cast<uint32_t>((n / kRS) & 1);
        if (!mbar_wait_bounded(&gs.full_bar[s], par)) {
            atomicOr(&s_abort, 1);
            if (t == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
            break;
        }
        const Hdr h = gs.hdr[s];
        if (h.pass == kPassStop) break;
        if (h.unit != cur) {
            // a new unit: per-unit constants (identical in every thread of the group)
            cur = h.unit;
            k = h.k;
            b = h.b;
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
            xmask = (greedy && !rowK) ? xt : -1;
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
            if (t == 0 && active && !rowK) {
                ztx = load_logit<D>(trow, xt);
                if (pair) {
                    zdx = load_logit<D>(drow, xt);
                    u_k = P.uniforms ? P.uniforms[static_cast<int64_t>(b) * (K + 1) + k] : 0.f;
                }
            }
        }
        const unsigned char *st = ring + s * kSB;
        if (h.pass == kPassSkip) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&gs.empty_bar[s]);
            ++n;
            rec.state = 2;
            rec.flags = flags;
            finish_unit();
            continue;
        }

        // ---- stage processing -----------------------------------------------
        if (active) {
            if (h.pass == kPassStats && h.pair) {
                // threads [0, kGT/2) take target groups, the rest draft groups
                const int row = t / (kGT / 2);
                const int tr = t - row * (kGT / 2);
                const int gl = tr / TPG1, part = tr % TPG1;
                uint4 w[VPT1];
                load_vecs<D, VPT1>(st + row * HALF, gl * GV + part * VPT1, h.nvec, (tr >> 1) & 3, w);
                const int g = h.chunk * GPR + gl;
                if (row == 0 || !shape.on) {
                    const float gm = tpg_max_nan<TPG1>(vecs_max<D, VPT1>(w));
                    float vs = 0.f;
                    if (gm != -INFINITY) vs = vecs_expsum<D, VPT1>(w, c, gm * c);
                    const float gsv = tpg_sum<TPG1>(vs);
                    if (part == 0) {
                        if (row == 0) {
                            if (g < G) {
                                gmax[g] = gm;
                                gsum[g] = gsv;
                            }
                        } else if (gm != -INFINITY) {
                            st_d = (gm == gm) ? stat_merge(st_d, Stat{gm * c, gsv}) : Stat{NAN, NAN};
                        }
                    }
                } else {
                    // reshaped draft: weights 2^(z c + log2 c_t), maximum over weighted values
                    const int e0 = h.chunk * GPR * kGroupTokens + (gl * GV + part * VPT1) * VEC;
                    float x[VPT1][VEC];
                    float xm = -INFINITY;
#pragma unroll
                    for (int kk = 0; kk < VPT1; ++kk) {
                        float z[VEC];
                        decode_vec<D>(w[kk], z);
                        const int ev = e0 + ((kk + ((tr >> 1) & 3)) & (VPT1 - 1)) * VEC;
#pragma unroll
                        for (int i = 0; i < VEC; ++i) {
                            x[kk][i] = z[i] * c + draft_bias(shape, z[i], ev + i);
                            xm = fmax_nan(xm, x[kk][i]);
                        }
                    }
                    const float gxm = tpg_max_nan<TPG1>(xm);
                    float vs = 0.f;
                    if (gxm != -INFINITY) {
#pragma unroll
                        for (int kk = 0; kk < VPT1; ++kk)
#pragma unroll
                            for (int i = 0; i < VEC; ++i) vs += ex2(x[kk][i] - gxm);
                    }
                    const float gsv = tpg_sum<TPG1>(vs);
                    if (part == 0 && gxm != -INFINITY)
                        st_d = (gxm == gxm) ? stat_merge(st_d, Stat{gxm, gsv}) : Stat{NAN, NAN};
                }
            } else if (h.pass == kPassStats) {
                // one row: sampled row K (max + mass) or greedy (max, drafted token excluded)
                const int gl = t / TPGS, part = t % TPGS;
                const int vbase = gl * GV + part * VPTS;
                uint4 w[VPTS];
                load_vecs<D, VPTS>(st, vbase, h.nvec, (t >> 1) & 3, w);
                const int e0 = h.chunk * GPS * kGroupTokens + vbase * VEC;
                if (static_cast<unsigned>(xmask - e0) < static_cast<unsigned>(VPTS * VEC)) {
#pragma unroll
                    for (int kk = 0; kk < VPTS; ++kk) {
                        const int ev = e0 + ((kk + ((t >> 1) & 3)) & (VPTS - 1)) * VEC;
                        if (static_cast<unsigned>(xmask - ev) < static_cast<unsigned>(VEC))
                            mask_vec<D>(w[kk], ev, 0, V, xmask);
                    }
                }
                const float gm = tpg_max_nan<TPGS>(vecs_max<D, VPTS>(w));
                float gsv = 0.f;
                if (sampled) {
                    float vs = 0.f;
                    if (gm != -INFINITY) vs = vecs_expsum<D, VPTS>(w, c, gm * c);
                    gsv = tpg_sum<TPGS>(vs);
                }
                const int g = h.chunk * GPS + gl;
                if (part == 0 && g < G) {
                    gmax[g] = gm;
                    gsum[g] = gsv;
                }
            } else {
                // pass 2 (pair): residual masses and maxima per group
                const int gl = t / TPG2, part = t % TPG2;
                const int vbase = gl * GV + part * VPT2;
                const int rot = (t >> 2) & 1;
                uint4 wt[VPT2], wd[VPT2];
                load_vecs<D, VPT2>(st, vbase, h.nvec, rot, wt);
                load_vecs<D, VPT2>(st + HALF, vbase, h.nvec, rot, wd);
                float2 acc = make_float2(0.f, 0.f);
                float mx = 0.f;
                if (!shape.on) {
                    const float2 cc = make_float2(c, c), nl = make_float2(-LT, -LD);
#pragma unroll
                    for (int kk = 0; kk < VPT2; ++kk) {
                        float zt[VEC], zd[VEC];
                        decode_vec<D>(wt[kk], zt);
                        decode_vec<D>(wd[kk], zd);
#pragma unroll
                        for (int i = 0; i < VEC; i += 2) {
                            const float2 x0 = __ffma2_rn(make_float2(zt[i], zd[i]), cc, nl);
                            const float2 x1 = __ffma2_rn(make_float2(zt[i + 1], zd[i + 1]), cc, nl);
                            const float2 d = __ffma2_rn(make_float2(ex2(x0.y), ex2(x1.y)),
                                                        make_float2(-1.f, -1.f),
                                                        make_float2(ex2(x0.x), ex2(x1.x)));
                            const float w0 = fmaxf(d.x, 0.f), w1 = fmaxf(d.y, 0.f);
                            acc = __fadd2_rn(acc, make_float2(w0, w1));
                            mx = fmaxf(mx, fmaxf(w0, w1));
                        }
                    }
                } else {
                    const int e0 = h.chunk * GPR * kGroupTokens + vbase * VEC;
#pragma unroll
                    for (int kk = 0; kk < VPT2; ++kk) {
                        float zt[VEC], zd[VEC];
                        decode_vec<D>(wt[kk], zt);
                        decode_vec<D>(wd[kk], zd);
                        const int ev = e0 + ((kk + rot) & (VPT2 - 1)) * VEC;
#pragma unroll
                        for (int i = 0; i < VEC; ++i) {
                            const float wv = resid_e(zt[i], zd[i], ev + i);
                            acc.x += wv;
                            mx = fmaxf(mx, wv);
                        }
                    }
                }
                const float gsv = tpg_sum<TPG2>(acc.x + acc.y);
                const float gm = tpg_max<TPG2>(mx);
                const int g = h.chunk * GPR + gl;
                if (part == 0 && g < G) {
                    gmax[g] = gm;
                    gsum[g] = gsv;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&gs.empty_bar[s]);
        ++n;
        if (!h.last) continue;

        // ---- end of a pass: the unit's tail ----------------------------------
        gbar(gc);  // group arrays complete
        rec.flags = flags;
        const bool want_p2 = pair && (do_verify || Fk > 0);
        if (!active) {
            if (h.pass == kPassResid || !want_p2) finish_unit();
            continue;
        }
        if (h.pass == kPassStats && sampled) {
            gT = target_stats();
            if (pair) gD = g_stat(gc, st_d, sc);
            const bool okT = (gT.m < INFINITY) && (gT.S > 0.f) && (gT.S < INFINITY);
            const bool okD = !pair || ((gD.m < INFINITY) && (gD.S > 0.f) && (gD.S < INFINITY));
            if (!okT || !okD) {
                flags |= SSD_DEV_NONFINITE;
                rec.flags = flags;
                active = false;
                if (!want_p2) finish_unit();
                continue;
            }
            LT = gT.m + lg2(gT.S);
            LD = pair ? gD.m + lg2(gD.S) : 0.f;
            if (pair && t == 0) {
                const float p = ex2(ztx * c - gT.m) / gT.S;
                const float q = ex2(zdx * c + draft_bias(shape, zdx, xt) - gD.m) / gD.S;
                rec.p_tok = p;
                rec.q_tok = q;
                rec.accept = (u_k * q < p) ? 1 : 0;
            }
            if (pair) {
                if (!want_p2) finish_unit();
                continue;
            }
            if (Fk > 0) top_f();
            if (do_verify) crossing(true, gT.m);
            finish_unit();
            continue;
        }
        if (h.pass == kPassStats && greedy) {
            uint64_t gk = 0;
            for (int g = t; g < G; g += kGT) {
                const uint64_t key = (static_cast<uint64_t>(ordered_bits(gmax[g])) << 32) |
                                     static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(g));
                gk = key > gk ? key : gk;
            }
            const uint64_t best = g_max_u64(gc, gk, sc);
            const float M = value_of_ordered(static_cast<uint32_t>(best >> 32));
            const int gbest = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFu));
            if (M != M) {
                flags |= SSD_DEV_NONFINITE;
                rec.flags = flags;
                finish_unit();
                continue;
            }
            if (gc.warp == 0) {
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
            gbar(gc);
            if (t == 0) {
                rec.tk = sc.bid;
                if (!rowK) {
                    rec.accept = make_key(ztx, xt) > sc.bkey ? 1 : 0;
                    rec.p_tok = rec.accept ? 1.f : 0.f;
                    rec.q_tok = 1.f;
                }
            }
            if (Fk > 0) top_f();
            finish_unit();
            continue;
        }
        // end of pass 2 (pair): residual mass, cache, bonus
        {
            float zs = 0.f;
            for (int g = t; g < G; g += kGT) zs += gsum[g];
            const float Z = g_sum_f32(gc, zs, sc);
            if (Fk > 0) top_f();
            if (do_verify) {
                if (Z > 0.f) {
                    crossing(false, 0.f);
                } else {
                    // no residual mass: draw from p at this row (group p-masses again)
                    for (int g = t; g < G; g += kGT) {
                        float m = -INFINITY;
                        for (int i = 0; i < kGroupTokens; ++i) {
                            const int e = g * kGroupTokens + i;
                            if (e < V) m = fmaxf(m, load_logit<D>(trow, e));
                        }
                        float s2 = 0.f;
                        for (int i = 0; i < kGroupTokens; ++i) {
                            const int e = g * kGroupTokens + i;
                            if (e < V) s2 += ex2(fmaf(load_logit<D>(trow, e), c, -m * c));
                        }
                        gmax[g] = m;
                        gsum[g] = s2;
                    }
                    gbar(gc);
                    crossing(true, gT.m);
                }
            }
            finish_unit();
        }
    }

    // this group is done
    gbar(gc);
    push_fin(1);
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
