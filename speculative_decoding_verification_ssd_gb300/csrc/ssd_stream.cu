// ssd_stream.cu -- persistent, warp-specialised streaming form of the fused
// verify / cache-build / lookup kernel (sm_103a).
//
// One CTA per SM, three roles, each present once per work lane g = 0, 1:
//   * producer warp g (one elected lane) takes units (sequence b, position k)
//     from a global counter and streams their logit rows with cp.async.bulk
//     into ring g (4 stages of 16 KB, each guarded by a full/empty mbarrier
//     pair).  The two-row, two-pass units (sampled sequence, position below
//     K) go before the greedy rows, so the grid ends on short units (a cache
//     build puts the sampled rows K first: unit_bk below);
//   * consumer group g (8 warps) only streams:
//       pass 1 (HBM)  sampled rows fold every element into per-thread online
//                     softmax statistics (base 2: m = max z c, S = sum 2^(z c - m),
//                     c = log2 e / tau); single rows also store per 64-token
//                     group the raw maximum (greedy rows: drafted token
//                     excluded) and, when sampled, the mass 2^(z c - gmax c);
//                     A pair unit that builds a cache also keeps the raw
//                     64-token group maxima of both rows;
//       between       a pair unit reduces its two statistics to the
//                     normalisers L_T, L_D and takes the accept test ([SD]
//                     step 3).  Only a rejected position's residual can be
//                     sampled; at an accepted one the residual serves the
//                     cache top-F_k alone, and a group can hold one of those
//                     only if its upper bound p(max z_p) reaches the F-th
//                     largest lower bound p(max z_p) - q(max z_q) (found with
//                     barrier counts over the threads' largest bounds);
//       pass 2        the pair's rows stream again, from the row's end back to
//                     its start (the chunks read last are still in L2): per
//                     group the residual mass sum max(0, p - q) and the largest
//                     residual, at an accepted position for those groups only
//                     (the rest read as 0).  The producer streams the first
//                     kRS stages of the pass unasked and the rest only for the
//                     chunks the consumers list after the accept test;
//     then hands the unit's group arrays (double-buffered) to
//   * tail warp g, which, without block barriers: selects the cache top-F_k
//     (groups whose maximum reaches the F-th largest of the lanes' two
//     largest group maxima are re-read and ranked as (value, id) keys, with
//     a bisection over the maxima for F_k above 64), draws the bonus t_k (at a
//     rejected position, or from p_K) at u_K by
//     inverse CDF over ascending token id (group prefix, then the crossing
//     group re-read), takes the greedy argmax, publishes the unit's record,
//     counts the sequence's finished units and, for the last one, runs the
//     epilogue (scan -> a, bonus t_a, outputs, cache lookup).
// The consumer groups never wait on a global-memory round trip, except in the
// kernel form that finds sigma_{F,C} in the pass (kSig), where a pair's draft
// top-F set is selected between its two passes (sigma_fuse).
//
// Operation sources: [SD] "Speculative decoding" (brentwoodlivery.com), "The
// Algorithm (Step-by-Step)" and "Temperature and Sampling"; [WHY] "Why does
// speculative decoding exist?", "How it works"; [SSD] "Speculative Speculative
// Decoding" notes (papernotes.org), "关键设计" items 1-2 and "整体框架".
#include <algorithm>

#include "ssd_device.cuh"
#include "ssd_launch.cuh"
#include "ssd_stream.cuh"
#include "ssd_stream_ops.cuh"
#include "ssd_unit.cuh"
#include "ssd_vec.cuh"

namespace ssd {
namespace {

constexpr int kGW = kStreamGroupWarps;  // warps per consumer group
constexpr int kGT = kGW * 32;           // threads per consumer group
constexpr int kNG = kStreamGroups;      // consumer groups (= rings = tail warps)
// A ring of kStreamRingStages x 16 KB is cut into slots of kSubs stages of the consumers'
// 16 KB geometry (one wait, header and release per slot; a pair slot is [target row part |
// draft row part]).  kSubs is set per kernel form: 2 for the wide form without the fused
// sigma selection (c4 105.2 -> 99.7 us, c2 37.7 -> 36.3), 1 for the others (c5 unchanged at
// 2, c3 80.4 -> 82.6).
constexpr int kSubB = kStreamStageBytes;   // bytes per stage (processing geometry)
constexpr int kRSMax = kStreamRingStages;  // slots per ring at one stage per slot
constexpr int kGTok = kGroupTokens;     // tokens per group of the group arrays
constexpr int kNBuf = kStreamBuffers;   // group-array buffers per consumer group
constexpr int kProducerWarp0 = kNG * kGW;
constexpr int kTailWarp0 = kProducerWarp0 + kNG;
constexpr int kCandGroupsCap = 512;
constexpr int kConsCandCap = 256;  // candidate groups an accepted pair resolves by direct loads
constexpr int kDecWords = 4;  // chunk bitmap of a second pass (128 chunks)
constexpr int kSchedCap = 2048;  // largest batch ordered by unit kind
static_assert(kStreamSigKeys == kCandCap && kGT == kThreads, "fused sigma selection geometry");

static_assert(kTailWarp0 + kNG == kStreamThreads / 32, "warp roles");

enum : int { kPassStats = 1, kPassResid = 2, kPassSkip = 3, kPassStop = 4 };
enum : int { kKindStop = 0, kKindPair = 1, kKindGreedy = 2, kKindSampled = 3, kKindPass = 4 };

// Stage header written by the producer: code = pass | last << 4 | pair << 5.
struct __align__(16) Hdr {
    int unit;
    int code;
    int chunk;  // chunk index within the pass
    int nvec;   // 16-byte vectors per row in this stage
    int b, k;   // sequence and position of the unit
    int tau;    // the sequence's temperature (float bits), loaded with the unit's claim
    int xt;     // drafted token x~_k (k < K), likewise
};

// A finished unit's hand-off from a consumer group to its tail warp.
struct TailDesc {
    int kind, b, k, flags;
    int state, accept, xt;
    int notfirst;  // pair: rejected after an earlier rejection of the sequence (bonus unused)
    float c;       // log2 e / tau
    float M, S;    // sampled single row: target statistics (base 2)
    float LT, LD;  // pair: normalisers (base 2)
    float p_tok, q_tok;
    float ztx;  // target logit of the drafted token (k < K)
    float tlo;  // pair: a score at least F_k tokens reach (-inf when none is known)
    DraftShape shape;
};

struct GroupShared {
    uint64_t full_bar[kRSMax];
    uint64_t empty_bar[kRSMax];
    uint64_t tail_full[kNBuf];
    uint64_t tail_empty[kNBuf];
    uint64_t dec_bar;         // consumer thread 0 -> producer: the chunks a second pass needs
    uint32_t dec_mask[kDecWords];
    Hdr hdr[kRSMax];
    TailDesc desc[kNBuf];
    Stat red[kGW];
    // tail-warp scratch
    uint64_t cand[kCandCap];
    int cgroups[kCandGroupsCap];
    int cnt[2];
    int scnt;  // consumer group: candidate count of the fused sigma selection
    // consumer group: an accepted pair's candidate groups (their largest residual is
    // computed from direct loads instead of a second pass over their chunks)
    uint16_t ccg[kConsCandCap];
    int ccnt;
    int rnf;  // consumer group: thread 0's answer whether the sequence rejected earlier
};

// sigma_{F,C} of one draft row found in the streaming pass ([SSD] item 2): the
// consumer group (kGT threads, named barrier bar_id) finds the row's top-F
// keys from its raw 64-token group maxima gmax[0, G) (written in pass 1).
// Each thread takes the largest of its groups' maxima; the F-th largest of
// those (found bit by bit with barrier counts) bounds the F-th largest logit
// from below; the groups at or above it are re-read from global memory (just
// streamed, so they hit L2) by whole warps, and the tokens at or above it are
// gathered and sorted (by one warp when at most 32 qualify, else by the group).
// The reshaped normaliser comes from the row's plain statistics gD = (m, S) at
// c: sum_t c_t 2^(x_t - m) = S - (1 - C) * (members' mass), whose rounding stays
// within 8 ulps of S when C >= 1/8 or the result is at least S/8; otherwise the
// non-members are summed afresh from the row (online, shifted by their own
// maximum).  On return (every thread): the descriptor, and
// q(t) = c_t 2^(z_t c - qm) / qS.
struct SigResult {
    DraftShape shape;
    float qm, qS;
};

template <class D>
__device__ __noinline__ SigResult sigma_fuse(const unsigned char *drow, const float *gmax, int G, int V,
                                             int F, float C, float c, Stat gD, uint64_t *keys, int *cnt,
                                             float *red, int t, int bar_id) {
    constexpr int VEC = D::kVec;
    const auto bar = [bar_id]() { asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(kGT) : "memory"); };
    const int lane = t & 31, w = t >> 5;
    float bm = -INFINITY;
    for (int g = t; g < G; g += kGT) bm = fmaxf(bm, gmax[g]);
    // F-th largest thread maximum, bit by bit over the upper 16 bits of the
    // ordered value (all of a bf16 value's; for fp32 the bound is the bottom of
    // its 2^-7-wide bucket), so T is at or below it
    const uint32_t ob = ordered_bits_nz(bm);
    uint32_t T = 0;
    for (int bit = 31; bit >= 16; --bit) {
        const uint32_t cand = T | (1u << bit);
        if (group_count(bar_id, kGT, ob >= cand) >= F) T = cand;
    }
    // id V ranks below every token of that value: a lower bound on the F-th key
    const uint64_t theta = (static_cast<uint64_t>(T) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(V));
    const float tv = value_of_ordered(T);
    auto visit = [&](uint64_t th, float thv, auto emit) {
        for (int g0 = w * 32; g0 < G; g0 += kGW * 32) {
            const int g = g0 + lane;
            uint32_t m = __ballot_sync(kFull, g < G && gmax[g] >= thv);
            while (m) {
                const int gg = g0 + __ffs(m) - 1;
                m &= m - 1;
                const int e = gg * kGTok + 2 * lane;  // the warp reads the group's 64 tokens
                if (e < V) {
                    const uint64_t k0 = make_key(load_logit<D>(drow, e), e);
                    if (k0 >= th) emit(k0);
                }
                if (e + 1 < V) {
                    const uint64_t k1 = make_key(load_logit<D>(drow, e + 1), e + 1);
                    if (k1 >= th) emit(k1);
                }
            }
        }
    };
    if (t == 0) *cnt = 0;
    bar();
    visit(theta, tv, [&](uint64_t key) {
        const int idx = atomicAdd(cnt, 1);
        if (idx < kCandCap) keys[idx] = key;
    });
    bar();
    const int count = *cnt;
    float top = 0.f;
    if (count <= 32) {
        // one warp sorts and sums the members (F <= count <= 32)
        if (w == 0) {
            uint64_t v = lane < count ? keys[lane] : 0;
            v = warp_sort_desc(v, lane);
            keys[lane] = v;
            float sm = lane < F ? ex2(fmaf(key_value(v), c, -gD.m)) : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(kFull, sm, o);
            if (lane == 0) red[0] = sm;
        }
        bar();
        top = red[0];
    } else {
        // many candidates (F above 32, or ties): the group's top-F selection
        const uint64_t tb = make_key(bm, V);
        group_topf(
            F, tb,
            [&](uint64_t th, auto emit) { visit(th, th ? key_value(th) : -INFINITY, emit); },
            keys, cnt, t, bar);
        float sm = t < F ? ex2(fmaf(key_value(keys[t]), c, -gD.m)) : 0.f;  // F <= kGT
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(kFull, sm, o);
        if (lane == 0) red[w] = sm;
        bar();
#pragma unroll
        for (int i = 0; i < kGW; ++i) top += red[i];
    }
    const uint64_t thr = keys[F - 1];
    bar();  // keys and red are free again
    SigResult r;
    r.shape.on = 1;
    r.shape.thr = key_value(thr);
    r.shape.thr_id = key_id(thr);
    r.shape.l2C = C > 0.f ? (C == 1.f ? 0.f : lg2(C)) : -INFINITY;
    const float Sp = gD.S - (1.f - C) * top;
    if (C >= 0.125f || Sp >= 0.125f * gD.S) {
        r.qm = gD.m;
        r.qS = Sp;
        return r;
    }
    // the members hold nearly all of the mass and C is small: sum the rest afresh
    Stat sn{-INFINITY, 0.f};
    const int nvec = (V + VEC - 1) / VEC;
    for (int v = t; v < nvec; v += kGT) {
        float z[VEC];
        decode_vec<D>(__ldg(reinterpret_cast<const uint4 *>(drow) + v), z);
        float x[VEC];
        float xm = -INFINITY;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const int e = v * VEC + i;
            const bool mem = z[i] > r.shape.thr || (z[i] == r.shape.thr && e <= r.shape.thr_id);
            x[i] = (mem || e >= V) ? -INFINITY : z[i] * c;
            xm = fmaxf(xm, x[i]);
        }
        stat_fold(sn, xm, [&](float mn) {
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < VEC; ++i) a += ex2(x[i] - mn);
            return a;
        });
    }
    const Stat ws = warp_stat(sn);
    if (lane == 0) {
        red[2 * w] = ws.m;
        red[2 * w + 1] = ws.S;
    }
    bar();
    Stat tot{-INFINITY, 0.f};
#pragma unroll
    for (int i = 0; i < kGW; ++i) tot = stat_merge_nan(tot, Stat{red[2 * i], red[2 * i + 1]});
    bar();
    // log2 of C * top * 2^m + S_non * 2^m_non, the larger term factored out
    const float a = (C > 0.f && top > 0.f) ? gD.m + lg2(C * top) : -INFINITY;
    const float bb = tot.S > 0.f ? tot.m + lg2(tot.S) : -INFINITY;
    const float hi = fmaxf(a, bb), lo = fminf(a, bb);
    r.qm = hi + lg2(1.f + ex2(lo - hi));
    r.qS = 1.f;
    return r;
}

}  // namespace

// kSig: sigma_{F,C} found in the pass.  kTail: rows are not whole 16-byte
// vectors (a row stride longer than V), so each row's last vector is masked; the
// common form carries none of that code.  kWide: both consumer groups work on
// each unit (instantiated in its own translation unit, ssd_stream_wide.cu, for
// rows of whole vectors; the one-group forms carry none of its code).
template <class D, bool kSig, bool kTail, bool kWide>
__global__ void __launch_bounds__(kStreamThreads, 1)
    ssd_stream_kernel(const __grid_constant__ UnitParams P) {
    constexpr int VEC = D::kVec, S = D::kBytes;
    constexpr int GV = kGTok / VEC;        // vectors per group
    constexpr int kSubs = (kWide && !kSig) ? 2 : 1;   // stages per ring slot
    constexpr int kRS = kStreamRingStages / kSubs;     // slots per ring
    constexpr int kSB = kStreamStageBytes * kSubs;     // bytes per slot
    static_assert(kRS * kSB == kStreamRingStages * kStreamStageBytes, "ring bytes");
    constexpr int HALF = kSubB / 2;        // bytes per row in a pair stage
    constexpr int DOFF = kSB / 2;          // the draft row part's offset in a pair slot
    constexpr int FULL_PAIR = HALF / 16;   // vectors per row in a full pair stage
    constexpr int FULL_ONE = kSubB / 16;   // vectors in a full single-row stage
    constexpr int GPR = FULL_PAIR / GV;    // groups per row in a pair stage
    constexpr int GPS = FULL_ONE / GV;     // groups in a single-row stage
    constexpr int TPGS = kGT / GPS;        // single rows: threads per group
    constexpr int TPG2 = kGT / GPR;        // pass 2: threads per group
    constexpr int VPT1 = FULL_PAIR / (kGT / 2), VPTS = GV / TPGS, VPT2 = GV / TPG2;
    constexpr int TPG1 = GV / VPT1;        // pass 1 of a pair: threads per group of one row
    static_assert(VPT1 == 4 && VPTS == 4 && VPT2 == 2, "stage geometry");
    static_assert((kStreamMaxGroups + GPR * kSubs - 1) / (GPR * kSubs) <= kDecWords * 32, "second-pass chunk list");
    constexpr int LPG = GV < 32 ? GV : 32;  // tail: lanes per group re-read (one vector each)
    constexpr int GPI = 32 / LPG;           // tail: groups per warp iteration
    constexpr int VPL = GV / LPG;           // tail: vectors per lane per group
    constexpr int TPL = kGTok / 32;         // tail: tokens per lane of one group
    constexpr int kBatch = 2;               // tail: vectors in flight per lane when re-reading
    constexpr int kMaskWords = kStreamMaxGroups / (32 * 32);  // tail: candidate mask words per lane (4 bits per strip)
    static_assert(32 % LPG == 0 && TPL >= 1 && kBatch % VPL == 0, "tail geometry");

    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ GroupShared gsh[kNG];
    __shared__ int s_abort;
    __shared__ int s_nS;
    __shared__ uint64_t s_ubar;  // wide: one arrival per consumer group at each shared step of a unit
    // wide: what group 0 finds between a pair's passes, for group 1
    __shared__ struct {
        float cthr, LD;
        DraftShape shape;
    } s_pub;
    __shared__ float s_wscr[kGW];  // wide: group 0's scratch for the fused sigma selection
    __shared__ int s_cnt[kSchedCap / 32];
    __shared__ uint16_t sched[kSchedCap];  // sampled sequences, then the others

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = P.B, K = P.K, V = P.V;
    const int G = (V + kGTok - 1) / kGTok;
    const int Gp = (G + 127) & ~127;  // group arrays padded to whole strips of 4 x 32 groups
    const bool do_verify = (P.mode & kModeVerify) != 0;
    const bool do_cache = (P.mode & kModeCache) != 0;
    const int nunits = B * (K + 1);
    // a row is streamed as whole 16-byte vectors: with a row stride longer than V
    // the last vector carries V % VEC tokens and the rest is masked on arrival
    const int nvec_row = (V + VEC - 1) / VEC;
    const int vtail = kTail ? V % VEC : 0;
    const int64_t row_bytes = static_cast<int64_t>(nvec_row) * 16;

    // the next launch on the stream may be scheduled now (it waits below for this one)
    asm volatile("griddepcontrol.launch_dependents;");
    if (tid == 0) {
        for (int g = 0; g < kNG; ++g) {
            for (int i = 0; i < kRS; ++i) {
                mbar_init(&gsh[g].full_bar[i], 1);
                mbar_init(&gsh[g].empty_bar[i], kGW);
            }
            for (int i = 0; i < kNBuf; ++i) {
                mbar_init(&gsh[g].tail_full[i], 1);
                mbar_init(&gsh[g].tail_empty[i], 1);
            }
            mbar_init(&gsh[g].dec_bar, 1);
        }
        mbar_init(&s_ubar, kNG);
        s_abort = 0;
        s_nS = 0;
        fence_mbar_init();
    }
    // Launched right behind another kernel (programmatic dependent launch), this
    // grid may get here while that kernel still runs: only shared memory is set
    // up above.  Global memory -- the inputs, which the previous kernel may have
    // written, and the workspace, which the previous round's last block resets --
    // is read only after that grid has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    // Sequence list of the unit order (unit_bk, below): the sampled sequences
    // first, then the others.  Every CTA maps the shared unit
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
    if (warp >= kProducerWarp0 && warp < kTailWarp0) {
        if (lane != 0) return;
        const int rg = warp - kProducerWarp0;  // ring served by this producer
        if (kWide && rg == 1) return;          // wide: producer 0 serves both rings
        GroupShared &gq = gsh[rg];
        unsigned char *ring = dyn_smem + rg * kRS * kSB;
        const uint64_t pol = policy_evict_first();
        const int nS = s_nS;
        const int nG = B - nS;
        auto unit_bk = [&](int u, int &b, int &k) {
            if (use_list && do_cache) {
                // A cache build streams every row: the sampled rows K go first (their short
                // units stagger the pairs, so that fewer groups finish a first pass at once;
                // c5 109.8 -> 108.9 us), then the pairs, then the greedy rows.
                if (u < nS) {
                    k = K;
                    b = sched[u];
                    return;
                }
                int v = u - nS;
                const int np = nS * K;
                if (v < np) {
                    k = v / nS;
                    b = sched[v - k * nS];
                    return;
                }
                v -= np;
                k = v / nG;
                b = sched[nS + v - k * nG];
                return;
            }
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
        int pf_state = 0, pf_u = 0, pf_b = 0, pf_k = 0, pf_xt = -1;
        float pf_tau = 0.f;
        uint32_t pf_rej = 0;
        // Every ring takes units from the front of the order (a shared counter; the
        // 64-bit word's high half is unused).  Starting ring 1 with a single row
        // from the back, to put the two groups' pairs out of phase, paid while every
        // pair streamed a long second pass; with short second passes it cost 2.4 us
        // at c5 (112.8 against 110.4).
        auto pf_step = [&]() {
            if (pf_state == 0) {
                const unsigned long long old = atomicAdd(P.unit_ends, 1ull);
                const uint32_t f = static_cast<uint32_t>(old);
                pf_u = f < static_cast<uint32_t>(nunits) ? static_cast<int>(f) : nunits;
                pf_state = 1;
            } else if (pf_state == 1) {
                if (pf_u < nunits) {
                    unit_bk(pf_u, pf_b, pf_k);
                    pf_tau = P.temperature[pf_b];
                    pf_xt = pf_k < K ? P.tokens[static_cast<int64_t>(pf_b) * K + pf_k] : -1;
                    pf_rej = (P.mode & kModeEarlyExit) ? __ldcg(P.seq_reject + pf_b) : 0u;
                }
                pf_state = 2;
            }
        };
        uint32_t n = 0;     // stages pushed
        uint32_t ndec = 0;  // second-pass chunk lists received
        bool ok = true;
        // Stages of a second pass streamed before the consumers' chunk list arrives: a
        // ring's worth (per ring), also in verification alone, where only a rejected pair
        // uses them -- they hide the decision's latency on the first rejection of a
        // sequence, which bounds the launch (c3 with none: 85.5 against 82.5 us).
        const int unasked = kRS;
        if constexpr (kWide) {
            // Both consumer groups share each unit: its chunk stages alternate between
            // ring 0 and ring 1 (every pass puts its last chunk on each ring with the
            // end bit, or a header-only end stage on a ring that got no chunk), and a
            // second pass longer than both rings follows group 0's chunk list.
            uint32_t nr1 = 0;  // stages pushed to ring 1 (n counts ring 0's)
            auto push = [&](int r, Hdr hd, const unsigned char *src_t, const unsigned char *src_d,
                            uint32_t bytes) -> bool {
                const uint32_t nn = r ? nr1 : n;
                const int s = static_cast<int>(nn % kRS);
                if (!mbar_wait_suspend(&gsh[r].empty_bar[s], ((nn / kRS) & 1) ^ 1)) return false;
                gsh[r].hdr[s] = hd;
                unsigned char *dst = dyn_smem + (r * kRS + s) * kSB;
                mbar_arrive_expect_tx(&gsh[r].full_bar[s], src_t ? bytes * (src_d ? 2u : 1u) : 0u);
                if (src_t) {
                    bulk_copy_hint(dst, src_t, bytes, &gsh[r].full_bar[s], pol);
                    if (src_d) bulk_copy_hint(dst + DOFF, src_d, bytes, &gsh[r].full_bar[s], pol);
                }
                if (r) ++nr1; else ++n;
                return true;
            };
            for (;;) {
                while (pf_state < 2) pf_step();
                pf_state = 0;
                const int u = pf_u;
                if (u >= nunits) {
                    const Hdr stop{-1, kPassStop | (1 << 4), 0, 0, 0, 0, 0, 0};
                    ok = push(0, stop, nullptr, nullptr, 0) && push(1, stop, nullptr, nullptr, 0);
                    break;
                }
                const int b = pf_b, k = pf_k, xt = pf_xt;
                const float tau = pf_tau;
                const int taub = __float_as_int(tau);
                const bool sampled = (tau > 0.f) && (tau < INFINITY);
                const bool pair = sampled && k < K;
                const bool p2 = pair && (do_verify || (do_cache && P.F[k] > 0));
                const uint32_t mask = (k >= 32) ? 0xFFFFFFFFu : ((1u << k) - 1u);
                if ((P.mode & kModeEarlyExit) && k > 0 && (pf_rej & mask) != 0) {
                    const Hdr sk{u, kPassSkip | (1 << 4), 0, 0, b, k, taub, xt};
                    ok = push(0, sk, nullptr, nullptr, 0) && push(1, sk, nullptr, nullptr, 0);
                    if (!ok) break;
                    continue;
                }
                const unsigned char *trow = static_cast<const unsigned char *>(P.tgt) +
                                            (static_cast<int64_t>(b) * P.tgt_seq_stride + static_cast<int64_t>(k) * P.ld) * S;
                const unsigned char *drow =
                    pair ? static_cast<const unsigned char *>(P.drf) +
                               (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * P.ld) * S
                         : nullptr;
                const int cb = pair ? DOFF : kSB;
                const int nch = static_cast<int>((row_bytes + cb - 1) / cb);
                const int pbit = (pair ? 1 : 0) << 5;
                auto chunk_stage = [&](int r, int pass, int chunk, bool last) -> bool {
                    const int64_t off = static_cast<int64_t>(chunk) * cb;
                    const uint32_t bytes = static_cast<uint32_t>(row_bytes - off < cb ? row_bytes - off : cb);
                    const Hdr hd{u, pass | ((last ? 1 : 0) << 4) | pbit, chunk, static_cast<int>(bytes / 16), b, k, taub, xt};
                    return push(r, hd, trow + off, drow ? drow + off : nullptr, bytes);
                };
                auto end_stage = [&](int r, int pass) -> bool {
                    const Hdr hd{u, pass | (1 << 4) | pbit, -1, 0, b, k, taub, xt};
                    return push(r, hd, nullptr, nullptr, 0);
                };
                for (int c = 0; c < nch && ok; ++c) {
                    ok = chunk_stage(c & 1, kPassStats, c, c >= nch - 2);
                    if (!p2 && nch - c <= 3) pf_step();
                }
                if (ok && nch == 1) ok = end_stage(1, kPassStats);
                if (ok && p2) {
                    // from the row's end back to its start, as in the one-ring form
                    if (nch <= 2 * unasked) {
                        for (int i = 0; i < nch && ok; ++i) {
                            ok = chunk_stage(i & 1, kPassResid, nch - 1 - i, i >= nch - 2);
                            if (nch - i <= 3) pf_step();
                        }
                        if (ok && nch == 1) ok = end_stage(1, kPassResid);
                    } else {
                        for (int i = 0; i < 2 * unasked && ok; ++i)
                            ok = chunk_stage(i & 1, kPassResid, nch - 1 - i, false);
                        if (ok) ok = mbar_wait_suspend(&gsh[0].dec_bar, ndec & 1);
                        if (ok) {
                            ++ndec;
                            const int lim = nch - 2 * unasked;  // chunks [0, lim) stream only when listed
                            const volatile uint32_t *dm = gsh[0].dec_mask;
                            int L = 0;
                            for (int w = 0; w * 32 < lim; ++w) {
                                uint32_t m = dm[w];
                                if (lim - w * 32 < 32) m &= (1u << (lim - w * 32)) - 1u;
                                L += __popc(m);
                            }
                            // the next unit is claimed near this one's end (not before the
                            // accept test: a rejected pair's long pass would hold it back)
                            int idx = 0;
                            for (int c = lim - 1; c >= 0 && ok; --c) {
                                if (!((dm[c >> 5] >> (c & 31)) & 1u)) continue;
                                ok = chunk_stage(idx & 1, kPassResid, c, idx >= L - 2);
                                ++idx;
                                if (L - idx <= 3) pf_step();
                            }
                            for (int r = L; r < 2 && ok; ++r) ok = end_stage(r, kPassResid);
                            pf_step();
                        }
                    }
                }
                if (!ok) break;
            }
        } else {
            for (;;) {
                while (pf_state < 2) pf_step();
                pf_state = 0;
                const int u = pf_u;
                if (u >= nunits) {
                    const int s = static_cast<int>(n % kRS);
                    if (!mbar_wait_suspend(&gq.empty_bar[s], ((n / kRS) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    gq.hdr[s] = Hdr{-1, kPassStop | (1 << 4), 0, 0, 0, 0, 0, 0};
                    mbar_arrive_expect_tx(&gq.full_bar[s], 0);
                    break;
                }
                const int b = pf_b, k = pf_k, xt = pf_xt;
                const float tau = pf_tau;
                const int taub = __float_as_int(tau);
                const bool sampled = (tau > 0.f) && (tau < INFINITY);
                const bool pair = sampled && k < K;
                const bool p2 = pair && (do_verify || (do_cache && P.F[k] > 0));
                const uint32_t mask = (k >= 32) ? 0xFFFFFFFFu : ((1u << k) - 1u);
                const bool skip = (P.mode & kModeEarlyExit) && k > 0 && (pf_rej & mask) != 0;
                const unsigned char *trow = static_cast<const unsigned char *>(P.tgt) +
                                            (static_cast<int64_t>(b) * P.tgt_seq_stride + static_cast<int64_t>(k) * P.ld) * S;
                const unsigned char *drow =
                    pair ? static_cast<const unsigned char *>(P.drf) +
                               (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * P.ld) * S
                         : nullptr;
                const int cb = pair ? DOFF : kSB;
                const int nch = static_cast<int>((row_bytes + cb - 1) / cb);
                const int total = skip ? 1 : nch * (p2 ? 2 : 1);
                // A second pass longer than its unasked stages streams those first; the
                // rest follows the consumers' chunk list, which they publish once the
                // accept test and the top-F bound are known (before those stages are used).
                const bool gated = p2 && !skip && nch > unasked;
                int lowest = 0;  // gated: the smallest listed chunk (streamed last), -1 for none
                for (int i = 0; i < total; ++i) {
                    bool empty_end = false, listed_last = false;
                    if (gated && i >= nch + unasked) {
                        if (i == nch + unasked) {
                            if (!mbar_wait_suspend(&gq.dec_bar, ndec & 1)) {
                                ok = false;
                                break;
                            }
                            ++ndec;
                            lowest = -1;
                            for (int c = 0; c < nch - unasked && lowest < 0; ++c)
                                if ((reinterpret_cast<volatile uint32_t *>(gq.dec_mask)[c >> 5] >> (c & 31)) & 1u)
                                    lowest = c;
                        }
                        const int chunk = nch - 1 - (i - nch);
                        if (lowest < 0) {
                            empty_end = true;  // nothing listed: a header-only stage ends the pass
                            i = total - 1;
                        } else if (!((reinterpret_cast<volatile uint32_t *>(gq.dec_mask)[chunk >> 5] >> (chunk & 31)) & 1u)) {
                            if (total - i <= 3) pf_step();
                            continue;
                        } else {
                            listed_last = chunk == lowest;
                        }
                    }
                    const int s = static_cast<int>(n % kRS);
                    if (!mbar_wait_suspend(&gq.empty_bar[s], ((n / kRS) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    if (skip) {
                        gq.hdr[s] = Hdr{u, kPassSkip | (1 << 4), 0, 0, b, k, taub, xt};
                        mbar_arrive_expect_tx(&gq.full_bar[s], 0);
                    } else if (empty_end) {
                        gq.hdr[s] = Hdr{u, kPassResid | (1 << 4) | (1 << 5), -1, 0, b, k, taub, xt};
                        mbar_arrive_expect_tx(&gq.full_bar[s], 0);
                    } else {
                        const bool second = i >= nch;
                        // the second pass runs from the row's end back to its start: the
                        // chunks read last in the first pass are the likeliest still in L2
                        const int chunk = second ? nch - 1 - (i - nch) : i;
                        const int64_t off = static_cast<int64_t>(chunk) * cb;
                        const uint32_t bytes = static_cast<uint32_t>(row_bytes - off < cb ? row_bytes - off : cb);
                        const bool last = second ? (gated && i >= nch + unasked ? listed_last : chunk == 0)
                                                 : chunk == nch - 1;
                        const int code = (second ? kPassResid : kPassStats) | ((last ? 1 : 0) << 4) |
                                         ((pair ? 1 : 0) << 5);
                        gq.hdr[s] = Hdr{u, code, chunk, static_cast<int>(bytes / 16), b, k, taub, xt};
                        unsigned char *dst = ring + s * kSB;
                        mbar_arrive_expect_tx(&gq.full_bar[s], bytes * (pair ? 2u : 1u));
                        // evict_first throughout: most second passes are cut to a few chunks,
                        // so holding first-pass rows in L2 for them costs more than it saves
                        bulk_copy_hint(dst, trow + off, bytes, &gq.full_bar[s], pol);
                        if (pair) bulk_copy_hint(dst + DOFF, drow + off, bytes, &gq.full_bar[s], pol);
                    }
                    ++n;
                    if (total - i <= 3) pf_step();
                }
                if (!ok) break;
            }
        }
        if (!ok) {
            atomicOr(&s_abort, 1);
            if (P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
        }
        return;
    }

    // =========================== tail warps =================================
    if (warp >= kTailWarp0) {
        const int team = warp - kTailWarp0;
        GroupShared &gs = gsh[team];
        float *const arrays = reinterpret_cast<float *>(dyn_smem + kNG * kRS * kSB) + team * kNBuf * 2 * Gp;
        const int R = (G + 31) / 32;  // groups per lane, contiguous
        const int g0 = min(G, lane * R), g1 = min(G, g0 + R);

        for (uint32_t j = 0;; ++j) {
            const int buf = static_cast<int>(j % kNBuf);
            if (!mbar_wait_suspend(&gs.tail_full[buf], (j / kNBuf) & 1)) {
                if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
                break;
            }
            const TailDesc d = gs.desc[buf];
            if (d.kind == kKindStop) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&gs.tail_empty[buf]);
                break;
            }
            float *gmax = arrays + buf * 2 * Gp;
            float *gsum = gmax + Gp;
            const int b = d.b, k = d.k;
            const int Fk = do_cache ? P.F[k] : 0;
            const float c = d.c;
            const unsigned char *trow = static_cast<const unsigned char *>(P.tgt) +
                                        (static_cast<int64_t>(b) * P.tgt_seq_stride + static_cast<int64_t>(k) * P.ld) * S;
            const unsigned char *drow = static_cast<const unsigned char *>(P.drf) +
                                        (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * P.ld) * S;
            const int xt = d.xt;
            const int xmask = (d.kind == kKindGreedy && k < K) ? xt : -1;
            const float nLT = -d.LT;
            const DraftShape shape = d.shape;
            UnitRecord rec{};
            rec.p_tok = d.p_tok;
            rec.q_tok = d.q_tok;
            rec.accept = d.accept;
            rec.tk = -1;
            rec.flags = d.flags;
            rec.state = d.state;

            auto resid_e = [&](float zp, float zq, int e) -> float {
                return resid_of(zp, zq, c, nLT, draft_bias(shape, zq, e) - d.LD);
            };

            // ---- cache top-F_k (gmax holds the scores' group maxima) --------
            auto top_f = [&](bool resid) -> uint64_t {
                // Threshold: the F-th largest of each lane's two largest group
                // maxima (64 distinct groups), so at least F groups reach it.
                // Lane l scans groups 4l..4l+3 of every 128-group strip with one
                // 16-byte load (conflict-free); the padding reads as -inf.
                const int nstrip = Gp / 128;
                const float4 *gm4 = reinterpret_cast<const float4 *>(gmax) + lane;
                uint32_t m1 = 0, m2 = 0;
                for (int i = 0; i < nstrip; ++i) {
                    const float4 v = gm4[32 * i];
                    const uint32_t o[4] = {ordered_bits_nz(v.x), ordered_bits_nz(v.y), ordered_bits_nz(v.z),
                                           ordered_bits_nz(v.w)};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        m2 = max(m2, min(m1, o[j]));
                        m1 = max(m1, o[j]);
                    }
                }
                uint32_t th = 0;
                if (Fk <= 64) {
                    uint32_t v = m1, nxt = m2;
                    for (int it = 0; it < Fk; ++it) {
                        th = __reduce_max_sync(kFull, v);
                        const uint32_t who = __ballot_sync(kFull, v == th);
                        if (lane == __ffs(who) - 1) {
                            v = nxt;
                            nxt = 0;
                        }
                    }
                } else {
                    // largest th with at least F groups whose maximum reaches it
                    uint32_t lo = 0, hi = 0xFFFFFFFFu;
                    while (lo < hi) {
                        const uint32_t mid = lo + ((hi - lo) >> 1) + 1;
                        int cnt = 0;
                        for (int i = 0; i < nstrip; ++i) {
                            const float4 v = gm4[32 * i];
                            cnt += (ordered_bits_nz(v.x) >= mid) + (ordered_bits_nz(v.y) >= mid) +
                                   (ordered_bits_nz(v.z) >= mid) + (ordered_bits_nz(v.w) >= mid);
                        }
                        cnt = __reduce_add_sync(kFull, cnt);
                        if (cnt >= Fk)
                            lo = mid;
                        else
                            hi = mid - 1;
                    }
                    th = lo;
                }
                // a pair whose second pass covered only the groups that can hold its
                // top-F (the rest read as 0) brings a score at least F tokens reach:
                // the threshold is at least that, so those zeros never become candidates
                if (d.tlo > 0.f) th = max(th, ordered_bits_nz(d.tlo));
                // candidate groups (maximum reaches th): per-lane bit masks (bit 4i + j:
                // group 128 i + 4 lane + j), then a warp prefix places each lane's groups
                uint32_t cm[kMaskWords];
#pragma unroll
                for (int w = 0; w < kMaskWords; ++w) cm[w] = 0;
                for (int i = 0; i < nstrip; ++i) {
                    const float4 v = gm4[32 * i];
                    const uint32_t bits = (ordered_bits_nz(v.x) >= th ? 1u : 0u) | (ordered_bits_nz(v.y) >= th ? 2u : 0u) |
                                          (ordered_bits_nz(v.z) >= th ? 4u : 0u) | (ordered_bits_nz(v.w) >= th ? 8u : 0u);
#pragma unroll
                    for (int w = 0; w < kMaskWords; ++w)
                        if ((i >> 3) == w) cm[w] |= bits << (4 * (i & 7));
                }
                int mine = 0;
#pragma unroll
                for (int w = 0; w < kMaskWords; ++w) mine += __popc(cm[w]);
                int incl = mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += y;
                }
                const int ncg = __shfl_sync(kFull, incl, 31);
                if (ncg <= kCandGroupsCap) {
                    int pos = incl - mine;
#pragma unroll
                    for (int w = 0; w < kMaskWords; ++w) {
                        uint32_t m = cm[w];
                        while (m) {
                            const int bt = 32 * w + __ffs(m) - 1;
                            m &= m - 1;
                            gs.cgroups[pos++] = 128 * (bt >> 2) + 4 * lane + (bt & 3);
                        }
                    }
                }
                if (lane == 0) gs.cnt[1] = 0;
                __syncwarp();
                const bool all_groups = ncg > kCandGroupsCap;
                const int ngroups = all_groups ? G : ncg;
                uint64_t theta = static_cast<uint64_t>(th) << 32;
                const int sub = lane / LPG, li = lane % LPG;
                int count = 0;
                for (int round = 0; round < 64; ++round) {
                    // each lane holds kBatch vectors of one or more groups per batch
                    for (int q0 = 0; q0 < ngroups; q0 += kBatch / VPL * GPI) {
                        uint4 wt[kBatch], wd[kBatch];
                        int e0[kBatch];
#pragma unroll
                        for (int x = 0; x < kBatch; ++x) {
                            const int q = q0 + (x / VPL) * GPI + sub;
                            e0[x] = V;
                            if (q < ngroups) {
                                const int g = all_groups ? q : gs.cgroups[q];
                                e0[x] = g * kGTok + ((x % VPL) * LPG + li) * VEC;
                            }
                            if (e0[x] < V) {
                                wt[x] = __ldg(reinterpret_cast<const uint4 *>(trow + static_cast<int64_t>(e0[x]) * S));
                                if (resid)
                                    wd[x] = __ldg(reinterpret_cast<const uint4 *>(drow + static_cast<int64_t>(e0[x]) * S));
                            }
                        }
#pragma unroll
                        for (int x = 0; x < kBatch; ++x) {
                            if (e0[x] >= V) continue;
                            float zt[VEC], zd[VEC];
                            decode_vec<D>(wt[x], zt);
                            if (resid) decode_vec<D>(wd[x], zd);
#pragma unroll
                            for (int i = 0; i < VEC; ++i) {
                                const int e = e0[x] + i;
                                if (e >= V) break;  // the row's partial last vector
                                uint64_t key;
                                if (resid)
                                    key = make_key(resid_e(zt[i], zd[i], e), e);
                                else
                                    key = (e == xmask) ? excluded_key(e) : make_key(zt[i], e);
                                if (key >= theta) {
                                    const int idx = atomicAdd(&gs.cnt[1], 1);
                                    if (idx < kCandCap) gs.cand[idx] = key;
                                }
                            }
                        }
                    }
                    __syncwarp();
                    count = gs.cnt[1];
                    if (count <= kCandCap) break;
                    // overflow: raise theta to the F-th largest of the stored keys
                    for (int kk = 2; kk <= kCandCap; kk <<= 1) {
                        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                            for (int i = lane; i < kCandCap; i += 32) {
                                const int ixj = i ^ jj;
                                if (ixj > i) {
                                    const uint64_t a = gs.cand[i], cc2 = gs.cand[ixj];
                                    const bool desc = (i & kk) == 0;
                                    if (desc ? (a < cc2) : (a > cc2)) {
                                        gs.cand[i] = cc2;
                                        gs.cand[ixj] = a;
                                    }
                                }
                            }
                            __syncwarp();
                        }
                    }
                    theta = gs.cand[Fk - 1];
                    __syncwarp();
                    if (lane == 0) gs.cnt[1] = 0;
                    __syncwarp();
                }
                if (count > kCandCap) count = kCandCap;
                // rank by counting; ranks below F go straight to the cache row
                uint64_t best = 0;
                for (int i = lane; i < count; i += 32) {
                    const uint64_t key = gs.cand[i];
                    best = key > best ? key : best;
                    int rr = 0;
                    for (int jx = 0; jx < count; ++jx) rr += gs.cand[jx] > key ? 1 : 0;
                    if (rr < Fk) P.cache_tok[static_cast<int64_t>(b) * P.budget + P.off[k] + rr] = key_id(key);
                }
                __syncwarp();
                return warp_max_u64(best);
            };

            // ---- inverse-CDF bonus at u_K over ascending token id -----------
            // Group weights: residual masses (gsum), or, with pmode, p-masses
            // gsum * 2^(gmax c - Mc).
            auto crossing = [&](bool pmode, float Mc) {
                auto gweight = [&](int g) -> float {
                    if (!pmode) return gsum[g];
                    const float gm = gmax[g];
                    return (gm == -INFINITY) ? 0.f : gsum[g] * ex2(fmaf(gm, c, -Mc));
                };
                float run = 0.f;
                int lastpos = -1;
                for (int g = g0; g < g1; ++g) {
                    const float wg = gweight(g);
                    run += wg;
                    if (wg > 0.f) lastpos = g;
                }
                const double incl = warp_incl_scan(static_cast<double>(run), lane);
                const double tot = __shfl_sync(kFull, incl, 31);
                const double T = static_cast<double>(P.uniforms[static_cast<int64_t>(b) * (K + 1) + K]) * tot;
                const double before = incl - static_cast<double>(run);
                const uint32_t hit = __ballot_sync(kFull, run > 0.f && before + static_cast<double>(run) > T);
                int gstar;
                double cut;
                if (hit) {
                    // the crossing lane's groups, scanned by the whole warp
                    const int ls = __ffs(hit) - 1;
                    const double base = __shfl_sync(kFull, before, ls);
                    const int a0 = min(G, ls * R), a1 = min(G, a0 + R);
                    const int per = (a1 - a0 + 31) / 32;
                    const int h0 = min(a1, a0 + lane * per), h1 = min(a1, h0 + per);
                    float r2 = 0.f;
                    for (int g = h0; g < h1; ++g) r2 += gweight(g);
                    const double i2 = warp_incl_scan(static_cast<double>(r2), lane);
                    const double b2 = base + i2 - static_cast<double>(r2);
                    const uint32_t hit2 = __ballot_sync(kFull, r2 > 0.f && b2 + static_cast<double>(r2) > T);
                    const int l2 = hit2 ? __ffs(hit2) - 1 : 31 - __clz(__ballot_sync(kFull, r2 > 0.f) | 1u);
                    int gs2 = -1;
                    double cut2 = 1e300;
                    if (lane == l2) {
                        double acc = b2;
                        for (int g = h0; g < h1; ++g) {
                            const float wg = gweight(g);
                            if (hit2 && acc + static_cast<double>(wg) > T) {
                                gs2 = g;
                                cut2 = T - acc;
                                break;
                            }
                            acc += static_cast<double>(wg);
                        }
                        if (gs2 < 0) {  // rounding: last group of the lane with mass
                            for (int g = h1 - 1; g >= h0; --g)
                                if (gweight(g) > 0.f) {
                                    gs2 = g;
                                    break;
                                }
                            cut2 = 1e300;
                        }
                    }
                    gstar = __shfl_sync(kFull, gs2, l2);
                    cut = __shfl_sync(kFull, cut2, l2);
                    if (gstar < 0) {
                        gstar = a0;
                        cut = 1e300;
                    }
                } else {
                    // past the total only through rounding: last group with mass
                    const int lp = static_cast<int>(__reduce_max_sync(kFull, static_cast<unsigned>(lastpos + 1)));
                    gstar = lp > 0 ? lp - 1 : 0;
                    cut = 1e300;
                }
                // element level: TPL consecutive tokens per lane, ascending
                const int e0 = gstar * kGTok + TPL * lane;
                float w[TPL];
                double lsum = 0.0;
#pragma unroll
                for (int x = 0; x < TPL; ++x) {
                    const int e = e0 + x;
                    w[x] = 0.f;
                    if (e < V) {
                        const float zt = load_logit<D>(trow, e);
                        w[x] = pmode ? ex2(fmaf(zt, c, -Mc)) : resid_e(zt, load_logit<D>(drow, e), e);
                    }
                    lsum += static_cast<double>(w[x]);
                }
                double cum = warp_incl_scan(lsum, lane) - lsum;
                int first_over = -1, last_pos = -1;
#pragma unroll
                for (int x = 0; x < TPL; ++x) {
                    cum += static_cast<double>(w[x]);
                    if (first_over < 0 && cum > cut && e0 + x < V) first_over = x;
                    if (w[x] > 0.f && e0 + x < V) last_pos = x;
                }
                const uint32_t over = __ballot_sync(kFull, first_over >= 0);
                const uint32_t pos = __ballot_sync(kFull, last_pos >= 0);
                int pick;
                if (over) {
                    const int l = __ffs(over) - 1;
                    pick = gstar * kGTok + TPL * l + __shfl_sync(kFull, first_over, l);
                } else if (pos) {
                    const int l = 31 - __clz(pos);
                    pick = gstar * kGTok + TPL * l + __shfl_sync(kFull, last_pos, l);
                } else {
                    pick = gstar * kGTok;
                }
                rec.tk = pick;
            };

            if (d.kind == kKindPair) {
                if (Fk > 0) top_f(true);
                // the bonus at k is drawn only where k rejected (the second pass left
                // every residual mass only there), and not after an earlier rejection
                if (do_verify && !d.accept && !d.notfirst) {
                    float zs = 0.f;
                    for (int g = g0; g < g1; ++g) zs += gsum[g];
                    const float Z = warp_sum(zs);
                    if (Z > 0.f) {
                        crossing(false, 0.f);
                    } else {
                        // no residual mass: draw from p at this row (group p-masses again)
                        for (int g = g0; g < g1; ++g) {
                            float m = -INFINITY;
                            for (int i = 0; i < kGTok; ++i) {
                                const int e = g * kGTok + i;
                                if (e < V) m = fmaxf(m, load_logit<D>(trow, e));
                            }
                            float s2 = 0.f;
                            if (m != -INFINITY) {
                                for (int i = 0; i < kGTok; ++i) {
                                    const int e = g * kGTok + i;
                                    if (e < V) s2 += ex2(fmaf(load_logit<D>(trow, e), c, -m * c));
                                }
                            }
                            gmax[g] = canon_zero(m);
                            gsum[g] = s2;
                        }
                        __syncwarp();
                        crossing(true, d.LT);
                    }
                }
            } else if (d.kind == kKindGreedy) {
                // argmax: the best group (lowest index on ties), then the lowest id in it
                uint64_t gk = 0;
                for (int g = g0; g < g1; ++g) {
                    const uint64_t key = (static_cast<uint64_t>(ordered_bits_nz(gmax[g])) << 32) |
                                         static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(g));
                    gk = key > gk ? key : gk;
                }
                const uint64_t best = warp_max_u64(gk);
                const float M = value_of_ordered(static_cast<uint32_t>(best >> 32));
                const int gbest = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFu));
                if (M != M) {
                    rec.flags |= SSD_DEV_NONFINITE;
                } else {
                    // the argmax is the largest cache candidate (same exclusion, same
                    // (value, lowest id) order); without a cache, re-read the best group
                    const uint64_t top = (Fk > 0) ? top_f(false) : 0;
                    int id;
                    if (Fk > 0 && key_value(top) == M) {
                        id = key_id(top);
                    } else {
                        const int e0 = gbest * kGTok + TPL * lane;
                        int mfirst = -1;
#pragma unroll
                        for (int x = TPL - 1; x >= 0; --x) {
                            const int e = e0 + x;
                            if (e < V && e != xmask && load_logit<D>(trow, e) == M) mfirst = x;
                        }
                        const uint32_t who = __ballot_sync(kFull, mfirst >= 0);
                        id = gbest * kGTok;
                        if (who) {
                            const int l = __ffs(who) - 1;
                            id = gbest * kGTok + TPL * l + __shfl_sync(kFull, mfirst, l);
                        }
                    }
                    rec.tk = id;
                    if (k < K) {
                        rec.accept = make_key(d.ztx, xt) > make_key(M, id) ? 1 : 0;
                        rec.p_tok = rec.accept ? 1.f : 0.f;
                        rec.q_tok = 1.f;
                    }
                }
            } else if (d.kind == kKindSampled) {
                if (Fk > 0) top_f(false);
                if (do_verify) crossing(true, d.M);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&gs.tail_empty[buf]);

            // ---- publish the record; the last unit of b runs the epilogue ----
            if (lane == 0) {
                UnitRecord *Rr = P.rec + static_cast<int64_t>(b) * (K + 1) + k;
                *Rr = rec;
                if (rec.flags == 0 && rec.state == 1 && k < K && !rec.accept && (P.mode & kModeEarlyExit))
                    atomicOr(P.seq_reject + b, 1u << k);
            }
            // the record and this warp's cache writes are visible before the unit is counted
            __threadfence();
            uint32_t done = 0;
            if (lane == 0) done = atomicAdd(P.seq_count + b, 1u);
            done = __shfl_sync(kFull, done, 0);
            if (done != static_cast<uint32_t>(K)) continue;
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
                            const int jj = j0 + lane;
                            const bool m = jj < P.off[a + 1] && __ldcg(row + jj) == tstar;
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
        // this tail warp is done; the last one of the grid resets the unit scheduler
        if (lane == 0) {
            __threadfence();
            const uint32_t done = atomicAdd(P.exit_counter, 1u);
            if (done == gridDim.x * kNG - 1) {
                *P.unit_counter = 0;
                *P.unit_ends = 0;
                *P.exit_counter = 0;
            }
        }
        return;
    }

    // =========================== consumers ==================================
    const int grp = warp / kGW;
    GroupShared &gs = gsh[grp];
    const int t = tid - grp * kGT;
    const int gw = warp - grp * kGW;
    const int bar_id = 1 + grp;
    auto gbar = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(kGT) : "memory"); };
    unsigned char *const ring = dyn_smem + grp * kRS * kSB;
    float *const abase = reinterpret_cast<float *>(dyn_smem + kNG * kRS * kSB);
    float *const arrays = abase + grp * kNBuf * 2 * Gp;
    // Wide form: both groups take every unit (alternate chunks from their rings) and
    // write one set of group arrays; unit j goes to tail warp j % 2, buffer (j / 2) % 2.
    // The steps they share meet at s_ubar (a bounded wait), group 0 alone finds the
    // top-F bound and the chunk list, and group 0's thread 0 hands the unit off.
    constexpr bool wide = kWide;
    static_assert(kNG == 2 && kNBuf == 2, "wide unit hand-off");
    const bool lead = t == 0 && (!wide || grp == 0);
    uint32_t nub = 0;  // wide: s_ubar phases passed
    int u_team = grp, u_buf = 0;  // tail warp and buffer of the current unit
    // fused sigma: candidate keys after the group arrays (present only when P.sig_on)
    uint64_t *const sig_keys =
        reinterpret_cast<uint64_t *>(dyn_smem + kNG * kRS * kSB + static_cast<size_t>(kNG) * kNBuf * 2 * Gp * 4) +
        grp * kStreamSigKeys;

    // per-thread stage geometry (fixed for the whole launch)
    const int p1_row = t / (kGT / 2), p1_tr = t % (kGT / 2);
    const int p1_vbase = p1_tr * VPT1, p1_rot = (p1_tr >> 1) & 3;
    const int s_gl = t / TPGS, s_part = t % TPGS;
    const int s_vbase = s_gl * GV + s_part * VPTS, s_rot = (t >> 1) & 3;
    const int r_gl = t / TPG2, r_part = t % TPG2;
    const int r_vbase = r_gl * GV + r_part * VPT2, r_rot = (t >> 2) & 1;

    uint32_t n = 0;    // stages consumed
    uint32_t nho = 0;  // hand-offs to the tail warp
    int cur = -1;
    int b = 0, k = 0, flags = 0, xt = -1, xmask = -1;
    bool sampled = false, pair = false, active = false, want_p2 = false, sig = false;
    bool bnd = false;      // a pair that builds a cache: pass 1 keeps both rows' group maxima
    bool notfirst = false;  // thread 0: a rejection after an earlier one of the sequence (verification alone)
    float cthr = -INFINITY;  // pass 2: residuals of the groups whose upper bound reaches this only
    const int nch_pair = static_cast<int>((row_bytes + DOFF - 1) / DOFF);  // slots of a pair pass
    float c = 0.f, LT = 0.f, LD = 0.f;
    DraftShape shape{0, 0.f, 0, 0.f};
    Stat st{-INFINITY, 0.f};
    // the padding [G, Gp) of every buffer reads as an empty group (never written later)
    for (int i = G + t; i < Gp; i += kGT)
        for (int bf = 0; bf < kNBuf; ++bf) {
            arrays[bf * 2 * Gp + i] = -INFINITY;
            arrays[bf * 2 * Gp + Gp + i] = 0.f;
        }
    float *gmax = arrays, *gsum = arrays + Gp;
    // thread 0: the accept test's gathers and results
    float ztx = 0.f, zdx = 0.f, u_k = 0.f, p_tok = NAN, q_tok = NAN;
    int accept = 0;

    // the unit's shared steps: the group's barrier, and in the wide form both groups'
    // (bounded: a group that gave up on its ring cannot hold the other one forever)
    auto usync = [&]() {
        gbar();
        if (!wide) return;
        if (t == 0) {
            __threadfence_block();
            mbar_arrive(&s_ubar);
        }
        if (!mbar_wait_suspend(&s_ubar, nub & 1)) {
            atomicOr(&s_abort, 1);
            if (t == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
        }
        ++nub;
    };
    // hands the unit to the tail warp (the barrier orders every thread's array writes first)
    auto handoff = [&](int hk, int state, float M, float Ssum) {
        usync();
        if (lead) {
            TailDesc &D0 = gsh[u_team].desc[u_buf];
            D0.kind = hk;
            D0.b = b;
            D0.k = k;
            D0.flags = flags;
            D0.state = state;
            D0.accept = accept;
            D0.xt = xt;
            D0.notfirst = notfirst ? 1 : 0;
            D0.c = c;
            D0.M = M;
            D0.S = Ssum;
            D0.LT = LT;
            D0.LD = LD;
            D0.p_tok = p_tok;
            D0.q_tok = q_tok;
            D0.ztx = ztx;
            D0.shape = shape;
            D0.tlo = (hk == kKindPair && cthr > 0.f && cthr < INFINITY) ? cthr : -INFINITY;
            mbar_arrive(&gsh[u_team].tail_full[u_buf]);
        }
        ++nho;
    };

    for (;;) {
        const int s = static_cast<int>(n % kRS);
        if (!mbar_wait_suspend(&gs.full_bar[s], (n / kRS) & 1)) {
            atomicOr(&s_abort, 1);
            if (t == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
            break;
        }
        const Hdr h = gs.hdr[s];
        const int pass = h.code & 15;
        if (pass == kPassStop) break;
        if (h.unit != cur) {
            // a new unit: wait for its group-array buffer, then per-unit constants
            u_team = wide ? static_cast<int>(nho & 1) : grp;
            u_buf = static_cast<int>(wide ? (nho >> 1) & 1 : nho % kNBuf);
            const uint32_t upar = wide ? (nho >> 2) & 1 : (nho / kNBuf) & 1;
            if (!mbar_wait_suspend(&gsh[u_team].tail_empty[u_buf], upar ^ 1)) {
                atomicOr(&s_abort, 1);
                if (t == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
                break;
            }
            cur = h.unit;
            k = h.k;
            b = h.b;
            gmax = abase + (u_team * kNBuf + u_buf) * 2 * Gp;
            gsum = gmax + Gp;
            const float tau = __int_as_float(h.tau);  // loaded by the producer with the claim
            const bool tau_ok = (tau >= 0.f) && (tau < INFINITY);
            const bool greedy = tau_ok && tau == 0.f;
            sampled = tau_ok && tau > 0.f;
            pair = sampled && k < K;
            flags = tau_ok ? 0 : SSD_DEV_BAD_TEMPERATURE;
            xt = -1;
            if (k < K) {
                xt = h.xt;
                if (xt < 0 || xt >= V) flags |= SSD_DEV_BAD_TOKEN;
            }
            xmask = (greedy && k < K) ? xt : -1;
            active = flags == 0;
            want_p2 = pair && (do_verify || (do_cache && P.F[k] > 0));
            bnd = pair && do_cache && P.F[k] > 0;
            cthr = -INFINITY;
            notfirst = false;
            c = sampled ? kLog2e / tau : 0.f;
            shape = DraftShape{0, 0.f, 0, 0.f};
            sig = kSig && pair && P.sig_F[k] > 0;
            if (pair && P.reshape) {
                const ssd_reshape_desc dd = P.reshape[static_cast<int64_t>(b) * K + k];
                shape.on = dd.F > 0;
                shape.thr = dd.thr_val;
                shape.thr_id = dd.thr_id;
                shape.l2C = dd.C > 0.f ? (dd.C == 1.f ? 0.f : lg2(dd.C)) : -INFINITY;
            }
            st = Stat{-INFINITY, 0.f};
            LT = 0.f;
            LD = 0.f;
            p_tok = NAN;
            q_tok = NAN;
            accept = 0;
            ztx = 0.f;
            if (active && k < K) {
                const unsigned char *trow = static_cast<const unsigned char *>(P.tgt) +
                                            (static_cast<int64_t>(b) * P.tgt_seq_stride + static_cast<int64_t>(k) * P.ld) * S;
                ztx = load_logit<D>(trow, xt);
                if (pair) {
                    const unsigned char *drow = static_cast<const unsigned char *>(P.drf) +
                                                (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * P.ld) * S;
                    zdx = load_logit<D>(drow, xt);
                    u_k = P.uniforms ? P.uniforms[static_cast<int64_t>(b) * (K + 1) + k] : 0.f;
                }
            }
        }
        if (pass == kPassSkip) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&gs.empty_bar[s]);
            ++n;
            handoff(kKindPass, 2, 0.f, 0.f);
            continue;
        }
        const bool stage_pair = (h.code >> 5) & 1;
        // the slot's stages: chunk index and vector count of each (a header-only slot has none)
        // (one stage per slot: exactly the slot's header, no loop bookkeeping)
        const int full_v = stage_pair ? FULL_PAIR : FULL_ONE;
#pragma unroll 1
        for (int sj = 0; sj < kSubs; ++sj) {
        const int hchunk = kSubs == 1 ? h.chunk : h.chunk * kSubs + sj;
        const int hnvec = kSubs == 1 ? h.nvec : min(full_v, h.nvec - sj * full_v);
        if (kSubs > 1 && hnvec <= 0) break;
        const unsigned char *stg = ring + s * kSB + (kSubs == 1 ? 0 : sj * (stage_pair ? HALF : kSubB));
        // the stage holding a row's partial last vector (row stride longer than V)
        const bool part = vtail != 0 && hchunk * (stage_pair ? FULL_PAIR : FULL_ONE) + hnvec == nvec_row;
        const int pv = part ? hnvec - 1 : -1;
        // ---- stage processing (a header-only stage just ends a pass) -----------
        if (active && hnvec > 0) {
            if (pass == kPassStats && stage_pair) {
                // online statistics: threads [0, 128) target, the rest draft
                uint4 w[VPT1];
                load_vecs<D, VPT1>(stg + p1_row * DOFF, p1_vbase, hnvec, p1_rot, hnvec == FULL_PAIR && !part, w);
                if (part) mask_partial<D, VPT1>(w, p1_vbase, p1_rot, pv, vtail);
                const float rm = vecs_max<D, VPT1>(w);
                if (sig || bnd) {
                    // raw 64-token group maxima: the draft's to gmax (the fused sigma's
                    // candidates, the bound on q), the target's to gsum (the bound on p)
                    const float gm = tpg_max<TPG1>(rm);
                    const int g = hchunk * GPR + p1_tr / TPG1;
                    if (p1_tr % TPG1 == 0 && g < G) (p1_row ? gmax : gsum)[g] = canon_zero(gm);
                }
                // a reshaped draft row takes the plain path where none of the thread's
                // tokens reaches the top-F threshold (all but a few threads of the row)
                if (p1_row == 0 || !shape.on || !(rm >= shape.thr)) {
                    stat_fold(st, rm * c, [&](float mn) { return vecs_expsum<D, VPT1>(w, c, mn); });
                } else {
                    st = reshaped_fold<D, VPT1>(st, stg + DOFF, p1_vbase, hnvec, p1_rot, hnvec == FULL_PAIR && !part,
                                                c, shape, hchunk * (FULL_PAIR * VEC) + p1_vbase * VEC, pv, vtail);
                }
            } else if (pass == kPassStats) {
                // one row: sampled row K (maxima, masses, statistics) or greedy (maxima,
                // drafted token excluded)
                uint4 w[VPTS];
                load_vecs<D, VPTS>(stg, s_vbase, hnvec, s_rot, hnvec == FULL_ONE && !part, w);
                if (part) mask_partial<D, VPTS>(w, s_vbase, s_rot, pv, vtail);
                const int e0 = hchunk * (FULL_ONE * VEC) + s_vbase * VEC;
                if (static_cast<unsigned>(xmask - e0) < static_cast<unsigned>(VPTS * VEC)) {
#pragma unroll
                    for (int kk = 0; kk < VPTS; ++kk) {
                        const int ev = e0 + ((kk + s_rot) & (VPTS - 1)) * VEC;
                        if (static_cast<unsigned>(xmask - ev) < static_cast<unsigned>(VEC))
                            mask_vec<D>(w[kk], ev, 0, V, xmask);
                    }
                }
                const float gm = tpg_max_nan<TPGS>(vecs_max<D, VPTS>(w));
                const int g = hchunk * GPS + s_gl;
                if (sampled) {
                    const float gmc = gm * c;
                    const float vs = vecs_expsum<D, VPTS>(w, c, gmc);
                    const float gsum_all = tpg_sum<TPGS>(vs);  // every lane shuffles
                    const float gsv = (gm == -INFINITY) ? 0.f : gsum_all;
                    const bool lead = s_part == 0 && gm != -INFINITY;
                    st = stat_merge_nan(st, Stat{lead ? gmc : -INFINITY, lead ? gsv : 0.f});
                    if (s_part == 0 && g < G) {
                        gmax[g] = canon_zero(gm);
                        gsum[g] = gsv;
                    }
                } else if (s_part == 0 && g < G) {
                    gmax[g] = canon_zero(gm);
                }
            } else {
                // pass 2 (pair): residual masses and maxima per group
                const bool full = hnvec == FULL_PAIR && !part;
                float2 acc = make_float2(0.f, 0.f);
                float mx = 0.f;
                const int g = hchunk * GPR + r_gl;
                // at an accepted position only the groups whose bound reaches cthr
                const bool cand =
                    cthr == -INFINITY ||
                    (cthr < INFINITY && g < G && ex2(fmaf(gsum[g], c, -LT)) * (1.f + 0x1p-20f) >= cthr);
                uint4 wt[VPT2], wd[VPT2];
                if (cand) {
                    load_vecs<D, VPT2>(stg, r_vbase, hnvec, r_rot, full, wt);
                    load_vecs<D, VPT2>(stg + DOFF, r_vbase, hnvec, r_rot, full, wd);
                    if (part) {
                        mask_partial<D, VPT2>(wt, r_vbase, r_rot, pv, vtail);
                        mask_partial<D, VPT2>(wd, r_vbase, r_rot, pv, vtail);
                    }
                }
                // reshaped draft: only tokens at or above the top-F threshold carry a bias
                if (!cand) {
                } else if (!shape.on || !(vecs_max<D, VPT2>(wd) >= shape.thr)) {
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
                            const float2 dd = __ffma2_rn(make_float2(ex2(x0.y), ex2(x1.y)),
                                                         make_float2(-1.f, -1.f),
                                                         make_float2(ex2(x0.x), ex2(x1.x)));
                            const float w0 = fmaxf(dd.x, 0.f), w1 = fmaxf(dd.y, 0.f);
                            acc = __fadd2_rn(acc, make_float2(w0, w1));
                            mx = fmaxf(mx, fmaxf(w0, w1));
                        }
                    }
                } else {
                    const float2 r2 = reshaped_resid<D, VPT2>(stg, DOFF, r_vbase, hnvec, r_rot, full, c, LT, LD, shape,
                                                              hchunk * (FULL_PAIR * VEC) + r_vbase * VEC, pv, vtail);
                    acc.x = r2.x;
                    mx = r2.y;
                }
                const float gsv = tpg_sum<TPG2>(acc.x + acc.y);
                const float gmx = tpg_max<TPG2>(mx);
                if (r_part == 0 && g < G) {
                    gmax[g] = gmx;
                    gsum[g] = gsv;
                }
            }
        }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&gs.empty_bar[s]);
        ++n;
        if (!((h.code >> 4) & 1)) continue;

        // ---- end of a pass ------------------------------------------------------
        // A second pass longer than its unasked stages (a ring's worth per ring)
        // continues only with the chunks thread 0 lists here (dec_mask, then dec_bar).
        const bool gated = pass == kPassStats && want_p2 && nch_pair > (wide ? 2 : 1) * kRS;
        auto list_chunks = [&](uint32_t all) {
            if (gated && lead) {
                if (all != 0u)
#pragma unroll
                    for (int w = 0; w < kDecWords; ++w) gs.dec_mask[w] = all;
                mbar_arrive(&gs.dec_bar);
            }
        };
        if (!active) {
            // an inactive pair still receives (the unasked part of) its second pass;
            // hand off after it
            if (pass == kPassStats && pair) {
                if (gated && lead)
#pragma unroll
                    for (int w = 0; w < kDecWords; ++w) gs.dec_mask[w] = 0u;
                list_chunks(0u);
            }
            if (pass == kPassResid || !want_p2) handoff(kKindPass, 1, 0.f, 0.f);
            continue;
        }
        if (pass == kPassStats && pair) {
            // normalisers: warps 0-3 of a group hold the target statistics, 4-7 the
            // draft's (wide: group 0's, then group 1's, in every thread)
            const Stat ws = warp_stat(st);
            usync();
            if (lane == 0) gs.red[gw] = ws;
            usync();
            Stat gT = gsh[wide ? 0 : grp].red[0], gD = gsh[wide ? 0 : grp].red[kGW / 2];
#pragma unroll
            for (int w = 1; w < kGW / 2; ++w) {
                gT = stat_merge_nan(gT, gsh[wide ? 0 : grp].red[w]);
                gD = stat_merge_nan(gD, gsh[wide ? 0 : grp].red[kGW / 2 + w]);
            }
            if (wide)
#pragma unroll
                for (int w = 0; w < kGW / 2; ++w) {
                    gT = stat_merge_nan(gT, gsh[1].red[w]);
                    gD = stat_merge_nan(gD, gsh[1].red[kGW / 2 + w]);
                }
            if (!stat_ok(gT) || !stat_ok(gD)) {
                flags |= SSD_DEV_NONFINITE;
                active = false;
                if (gated && lead)
#pragma unroll
                    for (int w = 0; w < kDecWords; ++w) gs.dec_mask[w] = 0u;
                list_chunks(0u);
                if (!want_p2) handoff(kKindPass, 1, 0.f, 0.f);
                continue;
            }
            LT = gT.m + lg2(gT.S);
            // (wide: group 0 alone from here to the chunk list, with its own barriers;
            // group 1 takes L_D, the draft shape and the top-F bound from it below)
            if (!wide || grp == 0) {
            float qm = gD.m, qS = gD.S;
            if (sig) {
                const unsigned char *drow = static_cast<const unsigned char *>(P.drf) +
                                            (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * P.ld) * S;
                const SigResult sr = sigma_fuse<D>(drow, gmax, G, V, P.sig_F[k], P.sig_C, c, gD, sig_keys, &gs.scnt,
                                                   wide ? s_wscr : reinterpret_cast<float *>(gs.red), t, bar_id);
                shape = sr.shape;
                qm = sr.qm;
                qS = sr.qS;
            }
            LD = qm + lg2(qS);
            // the same operations for both, so identical rows give identical p and q
            // (every thread: the accept bit decides the second pass's extent)
            p_tok = ex2(fmaf(ztx, c, -gT.m)) / gT.S;
            q_tok = ex2(fmaf(zdx, c, draft_bias(shape, zdx, xt) - qm)) / qS;
            accept = (u_k * q_tok < p_tok) ? 1 : 0;
            // A rejection publishes its bit at once (thread 0; the round trip overlaps the
            // bound search below).  In verification alone the sequence's units not yet
            // started then skip their rows; in any mode a rejection after an earlier one
            // of the sequence draws no bonus (only the first rejection's is used), so its
            // residual ranks the cache top-F alone, as at an accepted position.
            const bool rej = do_verify && !accept;
            uint32_t rej_old = 0;
            if (t == 0 && rej && k < 32) rej_old = atomicOr(P.seq_reject + b, 1u << k);
            if (!rej || bnd) {
                // the residual is not sampled here: it ranks the cache top-F alone (or
                // nothing).  For t* the target maximum of group g, r(t*) >= p(max z_p) -
                // q(max z_q), and no token of g exceeds p(max z_p) (a reshaped draft only
                // lowers q); both widened by 2^-20 relative against ex2's rounding.  The
                // threads' largest lower bounds (groups t, t + kGT, ...) give, bit by bit
                // over their upper 16 ordered bits, a value that at least F tokens reach.
                cthr = INFINITY;
                if (bnd) {
                    const int F = P.F[k];
                    float lbm = -INFINITY;
                    for (int gg = t; gg < G; gg += kGT) {
                        const float ub = ex2(fmaf(gsum[gg], c, -LT));
                        const float qb = ex2(fmaf(gmax[gg], c, -LD));
                        lbm = fmaxf(lbm, fmaf(-qb, 1.f + 0x1p-20f, ub));
                    }
                    const uint32_t ob = ordered_bits_nz(lbm);
                    uint32_t T = 0;
                    for (int bit = 31; bit >= 16; --bit) {
                        const uint32_t cand = T | (1u << bit);
                        if (group_count(bar_id, kGT, ob >= cand) >= F) T = cand;
                    }
                    const float tv = value_of_ordered(T);
                    cthr = tv > 0.f ? tv : -INFINITY;  // no positive bound: every group
                }
            }
            if (rej && bnd) {
                // the whole group needs the answer: the first rejection streams the whole
                // second pass (its bonus), a later one only its candidate groups
                if (t == 0) gs.rnf = (rej_old & ((1u << k) - 1u)) != 0u ? 1 : 0;
                gbar();
                notfirst = gs.rnf != 0;
                if (!notfirst) cthr = -INFINITY;
            } else if (rej) {
                if (t == 0) notfirst = (rej_old & ((1u << k) - 1u)) != 0u;
                cthr = -INFINITY;
            }
            if (gated) {
                if (cthr == INFINITY) {
                    // no residual is used (no cache top-F here, no bonus): no chunk, and
                    // no group array is read after this pass
                    if (t == 0)
#pragma unroll
                        for (int w = 0; w < kDecWords; ++w) gs.dec_mask[w] = 0u;
                    list_chunks(0u);
                } else if (cthr == -INFINITY) {
                    // every chunk: the first rejection's bonus, or a cache top-F without a
                    // positive bound; none for a later rejection that builds no cache
                    const bool none = notfirst && !bnd;
                    if (t == 0 && none)
#pragma unroll
                        for (int w = 0; w < kDecWords; ++w) gs.dec_mask[w] = 0u;
                    list_chunks(none ? 0u : 0xFFFFFFFFu);
                } else {
                    // The groups whose bound reaches cthr are the candidates; every other
                    // group's largest residual reads as 0.  Only the candidates' largest
                    // residuals matter here (the tail ranks the cache top-F from them; no
                    // residual is sampled at this position), so the group loads those 64
                    // tokens of both rows directly -- a warp per group, the same per-token
                    // arithmetic as the second pass -- and lists no chunk.  Past
                    // kConsCandCap candidates the chunks holding them are streamed instead.
                    if (t == 0) {
#pragma unroll
                        for (int w = 0; w < kDecWords; ++w) gs.dec_mask[w] = 0u;
                        gs.ccnt = 0;
                    }
                    gbar();
                    auto is_cand = [&](int gg) {
                        return cthr < INFINITY && ex2(fmaf(gsum[gg], c, -LT)) * (1.f + 0x1p-20f) >= cthr;
                    };
                    for (int gg = t; gg < G; gg += kGT) {
                        if (is_cand(gg)) {
                            const int ci = atomicAdd(&gs.ccnt, 1);
                            if (ci < kConsCandCap) gs.ccg[ci] = static_cast<uint16_t>(gg);
                        } else {
                            gmax[gg] = 0.f;
                        }
                    }
                    gbar();
                    const int ncg = gs.ccnt;
                    if (ncg <= kConsCandCap) {
                        list_chunks(0u);
                        const unsigned char *trow = static_cast<const unsigned char *>(P.tgt) +
                                                    (static_cast<int64_t>(b) * P.tgt_seq_stride + static_cast<int64_t>(k) * P.ld) * S;
                        const unsigned char *drow = static_cast<const unsigned char *>(P.drf) +
                                                    (static_cast<int64_t>(b) * P.drf_seq_stride + static_cast<int64_t>(k) * P.ld) * S;
                        const float nLT = -LT;
                        // two groups per warp at a time (both groups' loads in flight together)
                        for (int ci = gw; ci < ncg; ci += 2 * kGW) {
                            const int ci2 = ci + kGW;
                            const int ga = gs.ccg[ci], gb2 = ci2 < ncg ? gs.ccg[ci2] : ga;
                            float zp[4], zq[4];
                            int ee[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                ee[j] = (j < 2 ? ga : gb2) * kGTok + 2 * lane + (j & 1);
                                const bool in = ee[j] < V;
                                zp[j] = in ? load_logit<D>(trow, ee[j]) : -INFINITY;
                                zq[j] = in ? load_logit<D>(drow, ee[j]) : -INFINITY;
                            }
                            float ra = 0.f, rb = 0.f;
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float r = ee[j] < V ? resid_of(zp[j], zq[j], c, nLT, draft_bias(shape, zq[j], ee[j]) - LD)
                                                          : 0.f;
                                if (j < 2) ra = fmaxf(ra, r);
                                else rb = fmaxf(rb, r);
                            }
                            // non-negative values order like their bits (+0 for a zero)
                            const uint32_t ma = __reduce_max_sync(kFull, __float_as_uint(ra > 0.f ? ra : 0.f));
                            const uint32_t mb = __reduce_max_sync(kFull, __float_as_uint(rb > 0.f ? rb : 0.f));
                            if (lane == 0) {
                                gmax[ga] = __uint_as_float(ma);
                                if (ci2 < ncg) gmax[gb2] = __uint_as_float(mb);
                            }
                        }
                    } else {
                        for (int gg = t; gg < G; gg += kGT)
                            if (is_cand(gg)) {
                                const int ch = gg / (GPR * kSubs);  // the slot holding group gg
                                atomicOr(&gs.dec_mask[ch >> 5], 1u << (ch & 31));
                            }
                        gbar();
                        list_chunks(0u);
                    }
                }
            }
            }
            if (wide) {
                if (lead) {
                    s_pub.cthr = cthr;
                    s_pub.LD = LD;
                    s_pub.shape = shape;
                }
                usync();
                cthr = s_pub.cthr;
                LD = s_pub.LD;
                shape = s_pub.shape;
            }
            if (lead) {
                if (kSig && P.desc_out) {
                    ssd_reshape_desc dd;
                    dd.F = sig ? P.sig_F[k] : 0;
                    dd.C = P.sig_C;
                    dd.thr_val = sig ? shape.thr : INFINITY;
                    dd.thr_id = sig ? shape.thr_id : -1;
                    P.desc_out[static_cast<int64_t>(b) * K + k] = dd;
                }
            }
            if (!want_p2) handoff(kKindPass, 1, 0.f, 0.f);
            continue;
        }
        if (pass == kPassStats && sampled) {
            // sampled single row: target statistics for the tail's p-masses
            const Stat ws = warp_stat(st);
            usync();
            if (lane == 0) gs.red[gw] = ws;
            usync();
            Stat gT = gsh[wide ? 0 : grp].red[0];
#pragma unroll
            for (int w = 1; w < kGW; ++w) gT = stat_merge_nan(gT, gsh[wide ? 0 : grp].red[w]);
            if (wide)
#pragma unroll
                for (int w = 0; w < kGW; ++w) gT = stat_merge_nan(gT, gsh[1].red[w]);
            if (!stat_ok(gT)) {
                flags |= SSD_DEV_NONFINITE;
                handoff(kKindPass, 1, 0.f, 0.f);
                continue;
            }
            handoff(kKindSampled, 1, gT.m, gT.S);
            continue;
        }
        if (pass == kPassStats) {
            handoff(kKindGreedy, 1, 0.f, 0.f);
            continue;
        }
        handoff(kKindPair, 1, 0.f, 0.f);
    }

    // this group is done: tell its tail warp (wide: at the next unit index of that warp)
    {
        const uint32_t j = wide ? nho + ((nho ^ static_cast<uint32_t>(grp)) & 1u) : nho;
        const int sb = static_cast<int>(wide ? (j >> 1) & 1 : j % kNBuf);
        const uint32_t spar = wide ? (j >> 2) & 1 : (j / kNBuf) & 1;
        if (!mbar_wait_suspend(&gs.tail_empty[sb], spar ^ 1)) {
            if (t == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
        }
        gbar();
        if (t == 0) {
            gs.desc[sb].kind = kKindStop;
            mbar_arrive(&gs.tail_full[sb]);
        }
    }
}

#ifndef SSD_STREAM_WIDE_TU
// the one-group forms (this translation unit)
template <class D>
int stream_setup_d(size_t optin, size_t *max_dyn) {
    bool dummy = true;
    size_t lim[4];
    int st = setup_kernel(ssd_stream_kernel<D, true, false, false>, optin, &lim[0], &dummy);
    if (st == SSD_OK) st = setup_kernel(ssd_stream_kernel<D, false, true, false>, optin, &lim[1], &dummy);
    if (st == SSD_OK) st = setup_kernel(ssd_stream_kernel<D, false, false, false>, optin, &lim[2], &dummy);
    if (st == SSD_OK) st = stream_wide_setup(D::kBytes == 4 ? SSD_F32 : SSD_BF16, optin, &lim[3]);
    if (st != SSD_OK) return st;
    *max_dyn = std::min(std::min(lim[0], lim[1]), std::min(lim[2], lim[3]));  // one limit for every form
    return SSD_OK;
}

int stream_setup(int dtype, size_t optin, size_t *max_dyn) {
    return dtype == SSD_F32 ? stream_setup_d<F32Tag>(optin, max_dyn) : stream_setup_d<BF16Tag>(optin, max_dyn);
}

template <class D>
cudaError_t stream_launch_d(const cudaLaunchConfig_t &cfg, const UnitParams &P) {
    if (P.wide) return stream_wide_launch(D::kBytes == 4 ? SSD_F32 : SSD_BF16, cfg, P);
    if (P.sig_on) return cudaLaunchKernelEx(&cfg, ssd_stream_kernel<D, true, false, false>, P);
    if (P.V % D::kVec != 0) return cudaLaunchKernelEx(&cfg, ssd_stream_kernel<D, false, true, false>, P);
    return cudaLaunchKernelEx(&cfg, ssd_stream_kernel<D, false, false, false>, P);
}

int stream_launch(int dtype, const UnitParams &P, int grid, size_t dyn, void *stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = static_cast<cudaStream_t>(stream);
    // may start while the previous kernel on the stream drains (see griddepcontrol.wait)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = dtype == SSD_F32 ? stream_launch_d<F32Tag>(cfg, P) : stream_launch_d<BF16Tag>(cfg, P);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SSD_ERR_CUDA;
    }
    return SSD_OK;
}
#else
// the wide forms (rows of whole 16-byte vectors; sigma found in the pass or not)
template <class D>
int stream_wide_setup_d(size_t optin, size_t *max_dyn) {
    bool dummy = true;
    size_t lim[2];
    int st = setup_kernel(ssd_stream_kernel<D, true, false, true>, optin, &lim[0], &dummy);
    if (st == SSD_OK) st = setup_kernel(ssd_stream_kernel<D, false, false, true>, optin, &lim[1], &dummy);
    if (st != SSD_OK) return st;
    *max_dyn = std::min(lim[0], lim[1]);
    return SSD_OK;
}

int stream_wide_setup(int dtype, size_t optin, size_t *max_dyn) {
    return dtype == SSD_F32 ? stream_wide_setup_d<F32Tag>(optin, max_dyn) : stream_wide_setup_d<BF16Tag>(optin, max_dyn);
}

cudaError_t stream_wide_launch(int dtype, const cudaLaunchConfig_t &cfg, const UnitParams &P) {
    if (dtype == SSD_F32)
        return P.sig_on ? cudaLaunchKernelEx(&cfg, ssd_stream_kernel<F32Tag, true, false, true>, P)
                        : cudaLaunchKernelEx(&cfg, ssd_stream_kernel<F32Tag, false, false, true>, P);
    return P.sig_on ? cudaLaunchKernelEx(&cfg, ssd_stream_kernel<BF16Tag, true, false, true>, P)
                    : cudaLaunchKernelEx(&cfg, ssd_stream_kernel<BF16Tag, false, false, true>, P);
}
#endif

}  // namespace ssd
