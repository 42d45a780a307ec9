// ssd_slice.cu -- slice form of the fused verify / cache-build / lookup kernel
// (sm_103a): every logit row is split into S slices of whole 16 KB blocks, and
// (unit, slice) items are handed out dynamically to every consumer group of a
// persistent grid (one CTA per SM), so that a batch with few units still keeps
// every SM streaming and a unit's rows are read within a short window.
//
// Roles per CTA (as in the streaming kernel): per work lane g = 0, 1 a producer
// warp (one lane) that claims items and streams their slices with cp.async.bulk
// into ring g, a consumer group of 8 warps that folds each stage into online
// statistics and per-64-token-group arrays of the slice, and a tail warp that
// combines slices in global memory:
//   * first pass of a slice: pair units (sampled sequence, k < K) keep both
//     rows' statistics and, when a cache is built, both rows' group maxima;
//     single rows keep group maxima (greedy: drafted token excluded) and, when
//     sampled, group masses and statistics;
//   * the tail warp writes the slice's partial results (statistics, group
//     arrays, its local top-F_k keys) to the workspace and counts the slice;
//     the tail that counts a unit's last slice finishes it: a pair reduces the
//     slices' statistics to L_T, L_D, takes the accept test ([SD] step 3) and
//     queues its second pass -- every chunk at a rejected position (the bonus
//     is drawn from the whole residual), at an accepted one only the chunks
//     holding a group whose residual bound p(max z_p) reaches the F-th largest
//     lower bound p(max z_p) - q(max z_q) (the cache top-F_k alone);
//   * second pass of a pair slice (from the queue, taken before new first-pass
//     items, so the rows are still in L2): residual sums and maxima per group,
//     then its tail's local top-F_k keys and residual mass; the last one merges
//     the slices' keys into the cache segment and draws the bonus by inverse
//     CDF over ascending token id (slice prefix, group prefix, token);
//   * a single row's last slice merges the keys (greedy: the argmax is the
//     best key, x~ excluded) and, for the sampled row K, draws the bonus from p_K.
// The last unit of a sequence runs the epilogue (scan -> a, bonus t_a, outputs,
// cache lookup) as in the streaming kernel.  No role waits on another CTA.
//
// Operation sources: [SD] "Speculative decoding" (brentwoodlivery.com), "The
// Algorithm (Step-by-Step)" and "Temperature and Sampling"; [WHY] "Why does
// speculative decoding exist?", "How it works"; [SSD] "Speculative Speculative
// Decoding" notes (papernotes.org), "关键设计" items 1-2 and "整体框架".
#include <algorithm>

#include "ssd_device.cuh"
#include "ssd_launch.cuh"
#include "ssd_slice.cuh"
#include "ssd_stream.cuh"
#include "ssd_stream_ops.cuh"
#include "ssd_unit.cuh"
#include "ssd_vec.cuh"

namespace ssd {
namespace {

constexpr int kGW = kStreamGroupWarps;  // warps per consumer group
constexpr int kGT = kGW * 32;           // threads per consumer group
constexpr int kNG = kStreamGroups;      // consumer groups (= rings = tail warps)
constexpr int kRS = kStreamRingStages;  // stages per ring
constexpr int kSB = kStreamStageBytes;  // bytes per stage (one 16 KB block)
constexpr int kGTok = kGroupTokens;
constexpr int kNBuf = kSliceBuffers;
constexpr int kGs = kSliceMaxGroups;  // entries of one group array
constexpr int kProducerWarp0 = kNG * kGW;
constexpr int kTailWarp0 = kProducerWarp0 + kNG;
constexpr int kCandGroupsCap = 512;
constexpr int kSchedCap = 2048;  // batches ordered by unit kind (larger batches take other kernels)
constexpr int kMaskWords = kGs / (32 * 32);  // tail: candidate-group mask words per lane
static_assert(kSB == kSliceBlockBytes && kGT == kThreads, "slice geometry");
static_assert(kTailWarp0 + kNG == kStreamThreads / 32, "warp roles");
static_assert(kMaskWords >= 1, "candidate masks");
static_assert(kSliceCand == 64 && kSliceMaxSlices * kSliceCand <= kSliceScratch, "residual-bound candidates");

// scheduler counters in the workspace
enum : int { kCtrP1 = 0, kCtrQAlloc = 1, kCtrQClaim = 2, kCtrPairsDone = 3, kCtrExit = 4 };
enum : int { kPassP1 = 1, kPassP2 = 2, kPassSkip = 3, kPassStop = 4 };
enum : int { kTStop = 0, kTPair1 = 1, kTGreedy = 2, kTSampled = 3, kTPair2 = 4, kTSkip = 5 };

// Stage header: code = pass | last << 4 | pair << 5.  Every stage of an item
// also carries the item's inputs, which the producer loads when it claims the
// item, a few stages ahead (the consumers take no global round trip to start it).
struct __align__(16) SHdr {
    int item;   // per-ring item number (a new value starts a new item)
    int code;
    int chunk;  // stage index within the row: pair chunk (8 KB per row) or block (16 KB)
    int nvec;   // 16-byte vectors per row in this stage
    int b, k, s, xt;     // xt: drafted token (k < K), else -1
    float tau;           // temperature of sequence b
    float LT, LD, cthr;  // second pass of a pair: the unit's normalisers and residual bound
    int accept, pad0, pad1, pad2;
};
static_assert(sizeof(SHdr) == 64, "stage header");

// A finished item's hand-off from a consumer group to its tail warp.
struct STail {
    int kind, b, k, s;
    int flags, xmask, accept, pad;
    float c;
    float m0, S0, m1, S1;  // slice statistics (pair: target, draft; sampled row: m0, S0)
    float LT, LD, cthr;    // second pass of a pair
    DraftShape shape;
};

struct SGroup {
    uint64_t full_bar[kRS];
    uint64_t empty_bar[kRS];
    uint64_t tail_full[kNBuf];
    uint64_t tail_empty[kNBuf];
    SHdr hdr[kRS];
    STail desc[kNBuf];
    Stat red[kGW];
    uint64_t cand[kCandCap];  // tail: candidate keys
    int cgroups[kCandGroupsCap];
    int cnt[2];
};

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint32_t ld_volatile(const uint32_t *p) {
    return *reinterpret_cast<const volatile uint32_t *>(p);
}
__device__ __forceinline__ unsigned long long ld_volatile64(const unsigned long long *p) {
    return *reinterpret_cast<const volatile unsigned long long *>(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace

template <class D>
__global__ void __launch_bounds__(kStreamThreads, 1) ssd_slice_kernel(const __grid_constant__ UnitParams P) {
    constexpr int VEC = D::kVec, EB = D::kBytes;
    constexpr int GV = kGTok / VEC;        // vectors per group
    constexpr int HALF = kSB / 2;          // bytes per row in a pair stage
    constexpr int FULL_PAIR = HALF / 16;   // vectors per row in a full pair stage
    constexpr int FULL_ONE = kSB / 16;     // vectors in a full single-row stage
    constexpr int GPR = FULL_PAIR / GV;    // groups per row in a pair stage
    constexpr int GPS = FULL_ONE / GV;     // groups in a single-row stage (one block)
    constexpr int TPGS = kGT / GPS;        // single rows: threads per group
    constexpr int TPG2 = kGT / GPR;        // pass 2: threads per group
    constexpr int VPT1 = FULL_PAIR / (kGT / 2), VPTS = GV / TPGS, VPT2 = GV / TPG2;
    constexpr int TPG1 = GV / VPT1;        // pass 1 of a pair: threads per group of one row
    static_assert(VPT1 == 4 && VPTS == 4 && VPT2 == 2, "stage geometry");
    constexpr int TPL = kGTok / 32;         // tail: tokens per lane of one group
    static_assert(TPL >= 1, "tail geometry");

    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ SGroup gsh[kNG];
    __shared__ int s_abort;
    __shared__ int s_nS;
    __shared__ int s_cnt[kSchedCap / 32];
    __shared__ uint16_t sched[kSchedCap];  // sampled sequences, then the others

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = P.B, K = P.K, V = P.V, S = P.S, nblk = P.nblk;
    const int G = (V + kGTok - 1) / kGTok;
    const int GA = (G + 3) & ~3;  // per-unit group arrays in the workspace, 16-byte aligned
    const bool do_verify = (P.mode & kModeVerify) != 0;
    const bool do_cache = (P.mode & kModeCache) != 0;
    const int nunits = B * (K + 1);
    const int nvec_row = V / VEC;  // rows are whole 16-byte vectors (checked on the host)
    const int64_t row_bytes = static_cast<int64_t>(nvec_row) * 16;
    const int npc = (nvec_row + FULL_PAIR - 1) / FULL_PAIR;  // pair chunks per row

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
        }
        s_abort = 0;
        s_nS = 0;
        fence_mbar_init();
    }
    // global memory is read only once the previous grid on the stream has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    // Unit order, the same in every CTA: pair units (sampled sequence, k < K)
    // first, then the sampled rows K, then the other sequences' rows (a stable
    // compaction in ascending b).
    {
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
    const int nS = s_nS;
    const int total_pairs = nS * K;
    auto row_ptr = [&](const void *base, int64_t seq_stride, int b, int k) {
        return static_cast<const unsigned char *>(base) +
               (static_cast<int64_t>(b) * seq_stride + static_cast<int64_t>(k) * P.ld) * EB;
    };

    // =========================== producers ==================================
    if (warp >= kProducerWarp0 && warp < kTailWarp0) {
        if (lane != 0) return;
        const int rg = warp - kProducerWarp0;
        SGroup &gq = gsh[rg];
        unsigned char *ring = dyn_smem + rg * kRS * kSB;
        const uint64_t pol_first = policy_evict_first();
        const uint64_t pol_keep = policy_evict_normal();
        const uint32_t n_p1 = static_cast<uint32_t>(nunits) * static_cast<uint32_t>(S);
        const uint32_t n_queue = n_p1;  // queue entries: one per (unit, slice)
        const int nG = B - nS;
        auto unit_bk = [&](int u, int &b, int &k) {
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
        };
        uint32_t n = 0;
        int item = 0;
        bool ok = true, p1_out = false;
        const uint64_t t_start = globaltimer();
        // The next item is claimed (one attempt: a queued second pass, else a
        // first-pass item) and its inputs loaded while the current item's last
        // stages are issued; only when nothing can be claimed does the producer poll.
        int nx_pass = 0;  // 0: nothing claimed yet
        int nx_b = 0, nx_k = 0, nx_s = 0, nx_xt = -1, nx_acc = 0;
        float nx_tau = 0.f, nx_LT = 0.f, nx_LD = 0.f, nx_cthr = 0.f;
        uint32_t nx_mask = 0, nx_rej = 0;
        // A queued item is taken with a ticket (one atomic add on the claim counter)
        // when the queue looks non-empty, so that every waiting producer takes a
        // different item at once.  A ticket past the items queued so far waits for its
        // item, which comes unless every pair unit has already queued its second pass
        // and the ticket is past the last one; then a first-pass item is tried.
        auto try_claim = [&]() -> bool {
            int b = 0, k = 0, s = 0;
            bool got = false;
            uint32_t qc = 0;
            unsigned long long e = 0;
            if (ld_volatile(P.slice_ctr + kCtrQClaim) < ld_volatile(P.slice_ctr + kCtrQAlloc)) {
                qc = atomicAdd(P.slice_ctr + kCtrQClaim, 1u);
                // producers that see the queue non-empty at once take consecutive tickets,
                // possibly past its capacity (every queued index is below n_queue)
                for (; qc < n_queue;) {
                    e = ld_volatile64(P.queue + qc);
                    if (e != 0ull) {
                        got = true;
                        break;
                    }
                    __threadfence();
                    if (ld_volatile(P.slice_ctr + kCtrPairsDone) >= static_cast<uint32_t>(total_pairs) &&
                        ld_volatile(P.slice_ctr + kCtrQAlloc) <= qc)
                        break;  // no item will come for this ticket
                    if (globaltimer() - t_start > kWaitLimitNs) {
                        ok = false;
                        return false;
                    }
                    __nanosleep(64);
                }
            }
            if (got) {
                P.queue[qc] = 0ull;  // empty again for the next launch
                nx_mask = static_cast<uint32_t>(e >> 32);
                const uint32_t us = static_cast<uint32_t>(e & 0xFFFFFFFFull) - 1u;
                const int u = static_cast<int>(us / static_cast<uint32_t>(S));
                s = static_cast<int>(us % static_cast<uint32_t>(S));
                b = u / (K + 1);
                k = u % (K + 1);
                nx_pass = kPassP2;
            } else {
                if (p1_out) return false;
                const uint32_t i = atomicAdd(P.slice_ctr + kCtrP1, 1u);
                if (i >= n_p1) {
                    p1_out = true;
                    return false;
                }
                unit_bk(static_cast<int>(i / static_cast<uint32_t>(S)), b, k);
                s = static_cast<int>(i % static_cast<uint32_t>(S));
                nx_pass = kPassP1;
            }
            // the item's inputs (used when its first stage is issued)
            nx_b = b;
            nx_k = k;
            nx_s = s;
            nx_tau = P.temperature[b];
            nx_xt = k < K ? P.tokens[static_cast<int64_t>(b) * K + k] : -1;
            nx_rej = (nx_pass == kPassP1 && (P.mode & kModeEarlyExit)) ? __ldcg(P.seq_reject + b) : 0u;
            if (nx_pass == kPassP2) {
                const SliceUnitState *us = P.ustate + (b * (K + 1) + k);
                nx_LT = __ldcg(&us->LT);
                nx_LD = __ldcg(&us->LD);
                nx_cthr = __ldcg(&us->cthr);
                nx_acc = __ldcg(&us->accept);
            }
            return true;
        };
        for (;;) {
            // ---- the next item: the prefetched claim, else poll until one appears ----
            while (nx_pass == 0 && ok) {
                if (try_claim()) break;
                if (!ok) break;
                // nothing to take now: done once every pair unit has queued its second pass
                __threadfence();
                if (ld_volatile(P.slice_ctr + kCtrPairsDone) >= static_cast<uint32_t>(total_pairs)) {
                    __threadfence();
                    if (ld_volatile(P.slice_ctr + kCtrQClaim) >= ld_volatile(P.slice_ctr + kCtrQAlloc)) break;
                    continue;
                }
                if (globaltimer() - t_start > kWaitLimitNs) {
                    ok = false;
                    break;
                }
                __nanosleep(128);
            }
            if (!ok) break;
            const int st_ = static_cast<int>(n % kRS);
            if (nx_pass == 0) {
                if (!mbar_wait_suspend(&gq.empty_bar[st_], ((n / kRS) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                SHdr hs{};
                hs.item = -1;
                hs.code = kPassStop | (1 << 4);
                gq.hdr[st_] = hs;
                mbar_arrive_expect_tx(&gq.full_bar[st_], 0);
                ++n;
                break;
            }
            const int pass = nx_pass;
            const uint32_t cmask = nx_mask, rej = nx_rej;
            const int b = nx_b, k = nx_k, s = nx_s, xt = nx_xt, acc = nx_acc;
            const float tau = nx_tau, LTn = nx_LT, LDn = nx_LD, cthrn = nx_cthr;
            nx_pass = 0;
            ++item;
            // a stage header of this item
            auto put_hdr = [&](int sl, int code, int chunk, int nvec) {
                SHdr &hh = gq.hdr[sl];
                *reinterpret_cast<int4 *>(&hh) = make_int4(item, code, chunk, nvec);
                *(reinterpret_cast<int4 *>(&hh) + 1) = make_int4(b, k, s, xt);
                *(reinterpret_cast<float4 *>(&hh) + 2) = make_float4(tau, LTn, LDn, cthrn);
                *(reinterpret_cast<int4 *>(&hh) + 3) = make_int4(acc, 0, 0, 0);
            };
            const bool sampled = (tau > 0.f) && (tau < INFINITY);
            const bool pair = pass == kPassP2 || (sampled && k < K);
            const uint32_t below = (k >= 32) ? 0xFFFFFFFFu : ((1u << k) - 1u);
            const bool skip = pass == kPassP1 && (P.mode & kModeEarlyExit) && k > 0 && (rej & below) != 0;
            const int bl0 = slice_block0(s, S, nblk), bl1 = slice_block0(s + 1, S, nblk);
            const unsigned char *trow = row_ptr(P.tgt, P.tgt_seq_stride, b, k);
            const unsigned char *drow = pair ? row_ptr(P.drf, P.drf_seq_stride, b, k) : nullptr;
            int c0, c1;
            if (pair) {
                c0 = 2 * bl0;
                c1 = min(2 * bl1, npc);
            } else {
                c0 = bl0;
                c1 = bl1;
            }
            const int cb = pair ? HALF : kSB;
            const uint64_t pol = (pass == kPassP1 && pair) ? pol_keep : pol_first;
            if (skip) {
                if (!mbar_wait_suspend(&gq.empty_bar[st_], ((n / kRS) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                put_hdr(st_, kPassSkip | (1 << 4), 0, 0);
                mbar_arrive_expect_tx(&gq.full_bar[st_], 0);
                ++n;
                continue;
            }
            int last_c = c1 - 1;
            if (pass == kPassP2) last_c = c0 + 31 - __clz(cmask);
            int left = 0;  // stages of this item still to issue
            for (int c = c0; c < c1; ++c) left += (pass != kPassP2 || ((cmask >> (c - c0)) & 1u)) ? 1 : 0;
            for (int c = c0; c < c1 && ok; ++c) {
                if (pass == kPassP2 && !((cmask >> (c - c0)) & 1u)) continue;
                const int sl = static_cast<int>(n % kRS);
                if (!mbar_wait_suspend(&gq.empty_bar[sl], ((n / kRS) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                const int64_t off = static_cast<int64_t>(c) * cb;
                const uint32_t bytes = static_cast<uint32_t>(row_bytes - off < cb ? row_bytes - off : cb);
                put_hdr(sl, pass | ((c == last_c ? 1 : 0) << 4) | ((pair ? 1 : 0) << 5), c,
                        static_cast<int>(bytes / 16));
                unsigned char *dst = ring + sl * kSB;
                mbar_arrive_expect_tx(&gq.full_bar[sl], bytes * (pair ? 2u : 1u));
                bulk_copy_hint(dst, trow + off, bytes, &gq.full_bar[sl], pol);
                if (pair) bulk_copy_hint(dst + HALF, drow + off, bytes, &gq.full_bar[sl], pol);
                ++n;
                if (--left == 2 && nx_pass == 0) try_claim();
            }
            if (!ok) break;
            if (nx_pass == 0) try_claim();
        }
        if (!ok) {
            atomicOr(&s_abort, 1);
            if (P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
            // the ring's consumers still need a stop
            const int sl = static_cast<int>(n % kRS);
            if (mbar_wait_suspend(&gq.empty_bar[sl], ((n / kRS) & 1) ^ 1)) {
                gq.hdr[sl] = SHdr{-1, kPassStop | (1 << 4), 0, 0, 0, 0, 0, 0};
                mbar_arrive_expect_tx(&gq.full_bar[sl], 0);
            }
        }
        return;
    }

    // =========================== tail warps =================================
    if (warp >= kTailWarp0) {
        const int team = warp - kTailWarp0;
        SGroup &gs = gsh[team];
        float *const arrays = reinterpret_cast<float *>(dyn_smem + kNG * kRS * kSB) + team * kNBuf * 2 * kGs;
        // finishing scratch: two arrays of one slice's groups loaded from the workspace
        float *const scr = reinterpret_cast<float *>(dyn_smem + kNG * kRS * kSB) + kNG * kNBuf * 2 * kGs +
                           team * kSliceScratch;
        float *const sgmax = scr, *const sgsum = scr + kGs;
        auto unit_of = [&](int b, int k) { return b * (K + 1) + k; };
        auto slice_groups = [&](int s, int &g0, int &gn) {
            const int bl0 = slice_block0(s, S, nblk), bl1 = slice_block0(s + 1, S, nblk);
            g0 = bl0 * GPS;
            gn = min(bl1 * GPS, G) - g0;
        };
        auto key_area = [&](int b, int s, int k) {
            return P.skeys + (static_cast<int64_t>(b) * S + s) * P.key_stride + P.koff[k];
        };

        // ---- local top-F of a slice (group maxima gm[0, gn), first group g0) -----------
        // mode 0: raw logits (xmask excluded), 1: residual (p - q)^+ at (LT, LD, shape).
        // Writes the F best keys in descending order to out[0, F) (0 past the count).
        auto slice_topf = [&](const float *gm, int g0, int gn, int F, int mode, int xmask,
                              const unsigned char *trow, const unsigned char *drow, float c, float nLT,
                              float LD, DraftShape shape, float tlo, unsigned long long *out) -> uint64_t {
            if (F <= 0) return 0;
            const int nstrip = (gn + 127) / 128;
            // F-th largest of the lanes' two largest group maxima (F <= 64), else bisection
            uint32_t m1 = 0, m2 = 0;
            for (int i = 0; i < nstrip; ++i) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int g = 128 * i + 4 * lane + j;
                    const uint32_t o = g < gn ? ordered_bits_nz(gm[g]) : 0u;
                    m2 = max(m2, min(m1, o));
                    m1 = max(m1, o);
                }
            }
            uint32_t th = 0;
            if (F <= 64) {
                uint32_t v = m1, nxt = m2;
                for (int it = 0; it < F; ++it) {
                    th = __reduce_max_sync(kFull, v);
                    const uint32_t who = __ballot_sync(kFull, v == th);
                    if (lane == __ffs(who) - 1) {
                        v = nxt;
                        nxt = 0;
                    }
                }
            } else {
                uint32_t lo = 0, hi = 0xFFFFFFFFu;
                while (lo < hi) {
                    const uint32_t mid = lo + ((hi - lo) >> 1) + 1;
                    int cnt = 0;
                    for (int g = lane; g < gn; g += 32) cnt += ordered_bits_nz(gm[g]) >= mid;
                    cnt = __reduce_add_sync(kFull, cnt);
                    if (cnt >= F)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                th = lo;
            }
            if (tlo > 0.f) th = max(th, ordered_bits_nz(tlo));
            // candidate groups (maximum reaches th)
            uint32_t cm[kMaskWords];
#pragma unroll
            for (int w = 0; w < kMaskWords; ++w) cm[w] = 0;
            for (int i = 0; i < nstrip; ++i) {
                uint32_t bits = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int g = 128 * i + 4 * lane + j;
                    if (g < gn && ordered_bits_nz(gm[g]) >= th) bits |= 1u << j;
                }
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
            const int ngroups = all_groups ? gn : ncg;
            uint64_t theta = static_cast<uint64_t>(th) << 32;
            // The candidate groups' vectors are fetched into the scratch with cp.async,
            // as many groups at a time as it holds, so that a batch costs one round trip.
            const int nrow = mode == 1 ? 2 : 1;
            const int gcap = (kSliceScratch * 4) / (GV * 16 * nrow);  // groups per batch
            unsigned char *const stage = reinterpret_cast<unsigned char *>(scr);
            int count = 0;
            for (int round = 0; round < 64; ++round) {
                for (int q0 = 0; q0 < ngroups; q0 += gcap) {
                    const int nb = min(gcap, ngroups - q0);
                    for (int v = lane; v < nb * GV * nrow; v += 32) {
                        const int q = v / (GV * nrow), r = (v / GV) % nrow, j = v % GV;
                        const int g = g0 + (all_groups ? q0 + q : gs.cgroups[q0 + q]);
                        const int e = g * kGTok + j * VEC;
                        if (e < V) {
                            const unsigned char *src = (r ? drow : trow) + static_cast<int64_t>(e) * EB;
                            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(stage + 16 * v)),
                                         "l"(src)
                                         : "memory");
                        }
                    }
                    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
                    __syncwarp();
                    for (int v = lane; v < nb * GV; v += 32) {
                        const int q = v / GV, j = v % GV;
                        const int g = g0 + (all_groups ? q0 + q : gs.cgroups[q0 + q]);
                        const int e0 = g * kGTok + j * VEC;
                        if (e0 >= V) continue;
                        float zt[VEC], zd[VEC];
                        decode_vec<D>(*reinterpret_cast<const uint4 *>(stage + 16 * ((q * nrow) * GV + j)), zt);
                        if (mode == 1)
                            decode_vec<D>(*reinterpret_cast<const uint4 *>(stage + 16 * ((q * nrow + 1) * GV + j)), zd);
#pragma unroll
                        for (int i = 0; i < VEC; ++i) {
                            const int e = e0 + i;
                            uint64_t key;
                            if (mode == 1)
                                key = make_key(resid_of(zt[i], zd[i], c, nLT, draft_bias(shape, zd[i], e) - LD), e);
                            else
                                key = (e == xmask) ? excluded_key(e) : make_key(zt[i], e);
                            if (key >= theta) {
                                const int idx = atomicAdd(&gs.cnt[1], 1);
                                if (idx < kCandCap) gs.cand[idx] = key;
                            }
                        }
                    }
                    __syncwarp();
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
                theta = gs.cand[F - 1];
                __syncwarp();
                if (lane == 0) gs.cnt[1] = 0;
                __syncwarp();
            }
            if (count > kCandCap) count = kCandCap;
            // rank by counting; ranks below F go to the key area
            uint64_t best = 0;
            for (int i = lane; i < count; i += 32) {
                const uint64_t key = gs.cand[i];
                best = key > best ? key : best;
                int rr = 0;
                for (int jx = 0; jx < count; ++jx) rr += gs.cand[jx] > key ? 1 : 0;
                if (rr < F) out[rr] = key;
            }
            for (int r = count + lane; r < F; r += 32) out[r] = 0ull;
            __syncwarp();
            return warp_max_u64(best);
        };

        // ---- the F best of the keys of the slices in smask (each list: F_list keys,
        // descending) -> cache segment ranks [0, Fout); returns the best key ----
        auto merge_keys = [&](int b, int k, uint32_t smask, int F_list, int Fout) -> uint64_t {
            const int nl = __popc(smask);
            const int n = nl * F_list;
            int32_t *seg = P.cache_tok + static_cast<int64_t>(b) * P.budget + P.off[k];
            uint64_t best = 0;
            if (n <= kCandCap) {
                // key x of the n: list x / F_list (the (x / F_list)-th slice in smask), entry
                // x % F_list; loaded eight per lane at a time, all in flight together
                for (int x0 = 0; x0 < n; x0 += 32 * 8) {
                    unsigned long long kv[8];
#pragma unroll
                    for (int y = 0; y < 8; ++y) {
                        const int x = x0 + 32 * y + lane;
                        kv[y] = 0ull;
                        if (x < n) {
                            int li = x / F_list, s = 0;
                            uint32_t m = smask;
                            for (; li > 0; --li) m &= m - 1;  // drop the lists before it
                            s = __ffs(m) - 1;
                            kv[y] = __ldcg(key_area(b, s, k) + x % F_list);
                        }
                    }
#pragma unroll
                    for (int y = 0; y < 8; ++y) {
                        const int x = x0 + 32 * y + lane;
                        if (x < n) gs.cand[x] = kv[y];
                    }
                }
                __syncwarp();
                for (int i = lane; i < n; i += 32) {
                    const uint64_t key = gs.cand[i];
                    if (key == 0) continue;
                    best = key > best ? key : best;
                    if (Fout > 0) {
                        int rr = 0;
                        for (int jx = 0; jx < n; ++jx) rr += gs.cand[jx] > key ? 1 : 0;
                        if (rr < Fout) seg[rr] = key_id(key);
                    }
                }
                __syncwarp();
                return warp_max_u64(best);
            }
            // many keys: merge the sorted lists head by head (one list per lane)
            int sl = -1;
            {
                int idx = 0;
                for (int s = 0; s < S; ++s)
                    if ((smask >> s) & 1u) {
                        if (idx == lane) sl = s;
                        ++idx;
                    }
            }
            int pos = 0;
            uint64_t head = (sl >= 0 && F_list > 0) ? __ldcg(key_area(b, sl, k)) : 0ull;
            const int want = max(Fout, 1);
            for (int r = 0; r < want; ++r) {
                const uint64_t top = warp_max_u64(head);
                if (top == 0) break;
                if (r == 0) best = top;
                if (r < Fout && lane == 0) seg[r] = key_id(top);
                if (head == top && sl >= 0) {
                    ++pos;
                    head = pos < F_list ? __ldcg(key_area(b, sl, k) + pos) : 0ull;
                }
            }
            return best;
        };

        // ---- inverse CDF at T over group weights w(g) of one slice (g in [0, gn)),
        // the slice's first token e_first; returns the token ----
        auto slice_crossing = [&](int gn, int g0, double T0, auto gweight, auto tokw) -> int {
            const int R = (gn + 31) / 32;
            const int a0 = min(gn, lane * R), a1 = min(gn, a0 + R);
            float run = 0.f;
            int lastpos = -1;
            for (int g = a0; g < a1; ++g) {
                const float wg = gweight(g);
                run += wg;
                if (wg > 0.f) lastpos = g;
            }
            const double incl = warp_incl_scan(static_cast<double>(run), lane);
            const double before = incl - static_cast<double>(run);
            const uint32_t hit = __ballot_sync(kFull, run > 0.f && before + static_cast<double>(run) > T0);
            int gstar;
            double cut;
            if (hit) {
                const int ls = __ffs(hit) - 1;
                const double base = __shfl_sync(kFull, before, ls);
                const int h0 = min(gn, ls * R), h1 = min(gn, h0 + R);
                const int per = (h1 - h0 + 31) / 32;
                const int q0 = min(h1, h0 + lane * per), q1 = min(h1, q0 + per);
                float r2 = 0.f;
                for (int g = q0; g < q1; ++g) r2 += gweight(g);
                const double i2 = warp_incl_scan(static_cast<double>(r2), lane);
                const double b2 = base + i2 - static_cast<double>(r2);
                const uint32_t hit2 = __ballot_sync(kFull, r2 > 0.f && b2 + static_cast<double>(r2) > T0);
                const int l2 = hit2 ? __ffs(hit2) - 1 : 31 - __clz(__ballot_sync(kFull, r2 > 0.f) | 1u);
                int gs2 = -1;
                double cut2 = 1e300;
                if (lane == l2) {
                    double acc = b2;
                    for (int g = q0; g < q1; ++g) {
                        const float wg = gweight(g);
                        if (hit2 && acc + static_cast<double>(wg) > T0) {
                            gs2 = g;
                            cut2 = T0 - acc;
                            break;
                        }
                        acc += static_cast<double>(wg);
                    }
                    if (gs2 < 0) {
                        for (int g = q1 - 1; g >= q0; --g)
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
                    gstar = h0;
                    cut = 1e300;
                }
            } else {
                const int lp = static_cast<int>(__reduce_max_sync(kFull, static_cast<unsigned>(lastpos + 1)));
                gstar = lp > 0 ? lp - 1 : 0;
                cut = 1e300;
            }
            // element level: TPL consecutive tokens per lane, ascending
            const int e0 = (g0 + gstar) * kGTok + TPL * lane;
            float w[TPL];
            double lsum = 0.0;
#pragma unroll
            for (int x = 0; x < TPL; ++x) {
                const int e = e0 + x;
                w[x] = e < V ? tokw(e) : 0.f;
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
            const int gbase = (g0 + gstar) * kGTok;
            if (over) {
                const int l = __ffs(over) - 1;
                return gbase + TPL * l + __shfl_sync(kFull, first_over, l);
            }
            if (pos) {
                const int l = 31 - __clz(pos);
                return gbase + TPL * l + __shfl_sync(kFull, last_pos, l);
            }
            return gbase;
        };

        // ---- a slice-level prefix over weights ws (lane s holds slice s's weight):
        // the slice where the running sum first exceeds T, and the weight before it ----
        auto slice_prefix = [&](float wsl, double T, double &before_out) -> int {
            const double incl = warp_incl_scan(static_cast<double>(wsl), lane);
            const double before = incl - static_cast<double>(wsl);
            const uint32_t hit = __ballot_sync(kFull, lane < S && wsl > 0.f && incl > T);
            int sc;
            if (hit) {
                sc = __ffs(hit) - 1;
            } else {
                const uint32_t any = __ballot_sync(kFull, lane < S && wsl > 0.f);
                sc = any ? 31 - __clz(any) : 0;
            }
            before_out = __shfl_sync(kFull, before, sc);
            return sc;
        };

        // ---- a finished unit: record, counters, and the sequence's epilogue ----
        auto complete_unit = [&](int b, int k, UnitRecord rec, bool rejected_verify) {
            const int u = unit_of(b, k);
            if (lane == 0) {
                P.rec[u] = rec;
                SliceUnitState *us = P.ustate + u;
                us->p1_done = 0;
                us->p2_done = 0;
                us->p2_expect = 0;
                us->flags = 0;
                us->slice_mask = 0;
                if (rejected_verify && (P.mode & kModeEarlyExit)) atomicOr(P.seq_reject + b, 1u << k);
            }
            __threadfence();
            uint32_t done = 0;
            if (lane == 0) done = atomicAdd(P.seq_count + b, 1u);
            done = __shfl_sync(kFull, done, 0);
            if (done != static_cast<uint32_t>(K)) return;
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
                if ((fl & ~static_cast<int>(kSliceSkipped)) && P.dev_status)
                    atomicOr(P.dev_status, fl & ~static_cast<int>(kSliceSkipped));
                P.seq_count[b] = 0;
                P.seq_reject[b] = 0;
            }
        };

        // ---- a pair's last first-pass slice: normalisers, accept test, second pass ----
        auto finish_pair1 = [&](int b, int k) {
            const int u = unit_of(b, k);
            SliceUnitState *us = P.ustate + u;
            // every input of the unit requested at once (the logits at x~ one step later)
            int flags = static_cast<int>(__ldcg(&us->flags));
            const float tau = P.temperature[b];
            const int xt = P.tokens[static_cast<int64_t>(b) * K + k];
            const float u_k = P.uniforms ? P.uniforms[static_cast<int64_t>(b) * (K + 1) + k] : 0.f;
            ssd_reshape_desc rdesc{0.f, 0, 0, 1.f};
            if (P.reshape) rdesc = P.reshape[static_cast<int64_t>(b) * K + k];
            float4 st4 = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
            if (lane < S) st4 = __ldcg(P.sstat + static_cast<int64_t>(u) * S + lane);
            const unsigned char *trow = row_ptr(P.tgt, P.tgt_seq_stride, b, k);
            const unsigned char *drow = row_ptr(P.drf, P.drf_seq_stride, b, k);
            const bool xt_ok = xt >= 0 && xt < V;
            const float ztx = xt_ok ? load_logit<D>(trow, xt) : 0.f;
            const float zdx = xt_ok ? load_logit<D>(drow, xt) : 0.f;
            const float c = kLog2e / tau;
            // slice statistics merged in slice order (the same in every CTA)
            Stat gT{-INFINITY, 0.f}, gD{-INFINITY, 0.f};
            for (int s = 0; s < S; ++s) {
                const Stat a{__shfl_sync(kFull, st4.x, s), __shfl_sync(kFull, st4.y, s)};
                const Stat d{__shfl_sync(kFull, st4.z, s), __shfl_sync(kFull, st4.w, s)};
                gT = stat_merge_nan(gT, a);
                gD = stat_merge_nan(gD, d);
            }
            const bool skipped = (flags & static_cast<int>(kSliceSkipped)) != 0;
            if (!skipped && flags == 0 && (!stat_ok(gT) || !stat_ok(gD))) flags |= SSD_DEV_NONFINITE;
            UnitRecord rec{};
            rec.tk = -1;
            rec.flags = flags & ~static_cast<int>(kSliceSkipped);
            rec.state = skipped ? 2 : 1;
            rec.p_tok = NAN;
            rec.q_tok = NAN;
            uint32_t smask = 0, row_chunks[3] = {0, 0, 0};
            int accept = 0;
            float cthr = -INFINITY, LT = 0.f, LD = 0.f;
            bool need_bonus = false;
            if (!skipped && flags == 0) {
                DraftShape shape{0, 0.f, 0, 0.f};
                if (P.reshape) {
                    shape.on = rdesc.F > 0;
                    shape.thr = rdesc.thr_val;
                    shape.thr_id = rdesc.thr_id;
                    shape.l2C = rdesc.C > 0.f ? (rdesc.C == 1.f ? 0.f : lg2(rdesc.C)) : -INFINITY;
                }
                LT = gT.m + lg2(gT.S);
                LD = gD.m + lg2(gD.S);
                const float p_tok = ex2(fmaf(ztx, c, -gT.m)) / gT.S;
                const float q_tok = ex2(fmaf(zdx, c, draft_bias(shape, zdx, xt) - gD.m)) / gD.S;
                accept = (u_k * q_tok < p_tok) ? 1 : 0;
                rec.p_tok = p_tok;
                rec.q_tok = q_tok;
                rec.accept = accept;
                need_bonus = do_verify && !accept;
                // verification alone: publish the rejection now (units of the sequence not yet
                // started skip their rows); after an earlier rejection no residual is needed
                if (need_bonus && (P.mode & kModeEarlyExit) && k < 32) {
                    uint32_t old = 0;
                    if (lane == 0) old = atomicOr(P.seq_reject + b, 1u << k);
                    old = __shfl_sync(kFull, old, 0);
                    if (old & ((1u << k) - 1u)) need_bonus = false;
                }
                const bool need_cache = do_cache && P.F[k] > 0;
                if (need_bonus) {
                    row_chunks[0] = row_chunks[1] = row_chunks[2] = 0xFFFFFFFFu;
                } else if (need_cache) {
                    // Bounds on a group's largest residual: below p(max z_p) - q(max z_q) (the
                    // token holding the target maximum), above p(max z_p); both widened by 2^-20
                    // relative (ex2 rounding).  The F-th largest lower bound among the groups the
                    // slices reported is a value at least F tokens reach; a chunk can hold a
                    // top-F token only if its largest target maximum's bound reaches it.
                    const int F = P.F[k];
                    const int nc = S * kSliceCand;
                    const float2 *pc = reinterpret_cast<const float2 *>(P.pcand + static_cast<int64_t>(u) * S * kSliceCand * 2);
                    float *const lbs = scr;
                    for (int i0 = 0; i0 < nc; i0 += 32 * 4) {
                        float2 v[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int i = i0 + 32 * x + lane;
                            v[x] = i < nc ? __ldcg(pc + i) : make_float2(-INFINITY, 0.f);
                        }
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int i = i0 + 32 * x + lane;
                            if (i >= nc) continue;
                            const float ub = ex2(fmaf(v[x].x, c, -LT));
                            const float qb = ex2(fmaf(v[x].y, c, -LD));
                            lbs[i] = (v[x].x == -INFINITY) ? -INFINITY : fmaf(-qb, 1.f + 0x1p-20f, ub);
                        }
                    }
                    __syncwarp();
                    // the F-th largest candidate: F rounds of a warp maximum over the lanes'
                    // best remaining candidates (the winner takes its next one)
                    uint32_t lo = 0;
                    if (F <= nc) {
                        uint32_t bv = 0;
                        int bi = -1;
                        auto lane_best = [&]() {
                            bv = 0;
                            bi = -1;
                            for (int i = lane; i < nc; i += 32) {
                                const uint32_t o = ordered_bits(lbs[i]);
                                if (o > bv) {
                                    bv = o;
                                    bi = i;
                                }
                            }
                        };
                        lane_best();
                        for (int it = 0; it < F; ++it) {
                            lo = __reduce_max_sync(kFull, bv);
                            const uint32_t who = __ballot_sync(kFull, bv == lo && bi >= 0);
                            if (who && lane == __ffs(who) - 1) {
                                lbs[bi] = -INFINITY;
                                lane_best();
                            }
                        }
                    }
                    __syncwarp();
                    const float tv = value_of_ordered(lo);
                    cthr = tv > 0.f ? tv : -INFINITY;  // no positive bound: every chunk
                    const float *cm = P.cmax + static_cast<int64_t>(u) * npc;
                    for (int w = 0; w < 3; ++w) {
                        const int pcn = 32 * w + lane;
                        bool cand = false;
                        if (pcn < npc)
                            cand = cthr == -INFINITY || ex2(fmaf(__ldcg(cm + pcn), c, -LT)) * (1.f + 0x1p-20f) >= cthr;
                        row_chunks[w] = __ballot_sync(kFull, cand);
                    }
                }
                // per slice: its chunks' bits
                for (int s = 0; s < S; ++s) {
                    const int c0 = 2 * slice_block0(s, S, nblk);
                    const int c1 = min(2 * slice_block0(s + 1, S, nblk), npc);
                    uint32_t m = 0;
                    for (int pc = c0; pc < c1; ++pc)
                        if ((row_chunks[pc >> 5] >> (pc & 31)) & 1u) m |= 1u << (pc - c0);
                    if (m) smask |= 1u << s;
                }
            }
            const int nq = __popc(smask);
            if (lane == 0) {
                us->LT = LT;
                us->LD = LD;
                us->c = c;
                us->cthr = cthr;
                us->p_tok = rec.p_tok;
                us->q_tok = rec.q_tok;
                us->accept = accept;
                us->slice_mask = smask;
                us->p2_expect = static_cast<uint32_t>(nq);
            }
            __threadfence();
            __syncwarp();
            // queue the second pass, one item per slice with chunks to stream (the slots
            // taken with one atomic add)
            uint32_t qbase = 0;
            if (lane == 0 && nq > 0) qbase = atomicAdd(P.slice_ctr + kCtrQAlloc, static_cast<uint32_t>(nq));
            qbase = __shfl_sync(kFull, qbase, 0);
            if (lane < S && ((smask >> lane) & 1u)) {
                const int s = lane;
                const int c0 = 2 * slice_block0(s, S, nblk);
                const int c1 = min(2 * slice_block0(s + 1, S, nblk), npc);
                uint32_t m = 0;
                for (int pc = c0; pc < c1; ++pc)
                    if ((row_chunks[pc >> 5] >> (pc & 31)) & 1u) m |= 1u << (pc - c0);
                const uint32_t idx = qbase + static_cast<uint32_t>(__popc(smask & ((1u << s) - 1u)));
                const unsigned long long e = (static_cast<unsigned long long>(m) << 32) |
                                             static_cast<unsigned long long>(static_cast<uint32_t>(u) * S + s + 1u);
                atomicExch(P.queue + idx, e);
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) atomicAdd(P.slice_ctr + kCtrPairsDone, 1u);
            if (nq == 0) complete_unit(b, k, rec, false);
        };

        // ---- a pair's last second-pass item: cache segment and bonus ----
        auto finish_pair2 = [&](int b, int k) {
            const int u = unit_of(b, k);
            SliceUnitState *us = P.ustate + u;
            // the slices' residual masses and the bonus uniform, requested with the state
            const float zs = lane < S ? __ldcg(&P.sstat[static_cast<int64_t>(u) * S + lane].x) : 0.f;
            const float uK = P.uniforms ? P.uniforms[static_cast<int64_t>(b) * (K + 1) + K] : 0.f;
            UnitRecord rec{};
            rec.accept = __ldcg(&us->accept);
            rec.p_tok = __ldcg(&us->p_tok);
            rec.q_tok = __ldcg(&us->q_tok);
            rec.flags = 0;
            rec.state = 1;
            rec.tk = -1;
            const uint32_t smask = __ldcg(&us->slice_mask);
            const float c = __ldcg(&us->c), LT = __ldcg(&us->LT), LD = __ldcg(&us->LD);
            if (do_cache && P.F[k] > 0) merge_keys(b, k, smask, P.F[k], P.F[k]);
            const bool need_bonus = do_verify && !rec.accept;
            if (need_bonus) {
                const unsigned char *trow = row_ptr(P.tgt, P.tgt_seq_stride, b, k);
                const unsigned char *drow = row_ptr(P.drf, P.drf_seq_stride, b, k);
                DraftShape shape{0, 0.f, 0, 0.f};
                if (P.reshape) {
                    const ssd_reshape_desc dd = P.reshape[static_cast<int64_t>(b) * K + k];
                    shape.on = dd.F > 0;
                    shape.thr = dd.thr_val;
                    shape.thr_id = dd.thr_id;
                    shape.l2C = dd.C > 0.f ? (dd.C == 1.f ? 0.f : lg2(dd.C)) : -INFINITY;
                }
                float Z = zs;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(kFull, Z, o);
                if (Z > 0.f) {
                    // totals summed in slice order in fp64 (the same as the prefix)
                    const double tot = __shfl_sync(kFull, warp_incl_scan(static_cast<double>(zs), lane), 31);
                    const double T = static_cast<double>(uK) * tot;
                    double base = 0.0;
                    const int sc = slice_prefix(zs, T, base);
                    int g0, gn;
                    slice_groups(sc, g0, gn);
                    const float *src = P.garr + static_cast<int64_t>(u) * 2 * GA + GA + g0;  // residual sums
                    for (int g = lane; g < gn; g += 32) sgsum[g] = __ldcg(src + g);
                    __syncwarp();
                    rec.tk = slice_crossing(
                        gn, g0, T - base, [&](int g) { return sgsum[g]; },
                        [&](int e) {
                            return resid_of(load_logit<D>(trow, e), load_logit<D>(drow, e), c, -LT,
                                            draft_bias(shape, load_logit<D>(drow, e), e) - LD);
                        });
                } else {
                    // no residual mass (p == q at this row): draw from p, group masses summed
                    // over the whole row from global memory
                    auto pmass = [&](int g) {
                        float m = -INFINITY;
                        for (int i = 0; i < kGTok; ++i) {
                            const int e = g * kGTok + i;
                            if (e < V) m = fmaxf(m, load_logit<D>(trow, e));
                        }
                        if (m == -INFINITY) return 0.f;
                        float s2 = 0.f;
                        for (int i = 0; i < kGTok; ++i) {
                            const int e = g * kGTok + i;
                            if (e < V) s2 += ex2(fmaf(load_logit<D>(trow, e), c, -m * c));
                        }
                        return s2 * ex2(fmaf(m, c, -LT));
                    };
                    // the row's group masses through the scratch array, kGs groups at a time
                    double Tp = -1.0, run_before = 0.0;
                    double ptot = 0.0;
                    for (int g = lane; g < G; g += 32) ptot += static_cast<double>(pmass(g));
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) ptot += __shfl_xor_sync(kFull, ptot, o);
                    Tp = static_cast<double>(uK) * ptot;
                    int done_tk = -1;
                    for (int gb = 0; gb < G && done_tk < 0; gb += kGs) {
                        const int gn = min(kGs, G - gb);
                        for (int g = lane; g < gn; g += 32) sgsum[g] = pmass(gb + g);
                        __syncwarp();
                        float part = 0.f;
                        for (int g = lane; g < gn; g += 32) part += sgsum[g];
                        double dpart = static_cast<double>(part);
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) dpart += __shfl_xor_sync(kFull, dpart, o);
                        if (run_before + dpart > Tp || gb + gn >= G) {
                            done_tk = slice_crossing(
                                gn, gb, Tp - run_before, [&](int g) { return sgsum[g]; },
                                [&](int e) { return ex2(fmaf(load_logit<D>(trow, e), c, -LT)); });
                        }
                        run_before += dpart;
                        __syncwarp();
                    }
                    rec.tk = done_tk;
                }
            }
            complete_unit(b, k, rec, need_bonus);
        };

        // ---- a single row's last slice: cache segment, greedy argmax, or the bonus from p_K ----
        auto finish_single = [&](int b, int k, bool greedy) {
            const int u = unit_of(b, k);
            SliceUnitState *us = P.ustate + u;
            const int flags = static_cast<int>(__ldcg(&us->flags));
            UnitRecord rec{};
            rec.tk = -1;
            rec.flags = flags & ~static_cast<int>(kSliceSkipped);
            rec.state = (flags & static_cast<int>(kSliceSkipped)) ? 2 : 1;
            rec.p_tok = NAN;
            rec.q_tok = NAN;
            bool rejected = false;
            if (flags == 0) {
                const uint32_t all = (S >= 32) ? 0xFFFFFFFFu : ((1u << S) - 1u);
                const int Fk = do_cache ? P.F[k] : 0;
                if (greedy) {
                    const uint64_t top = merge_keys(b, k, all, max(Fk, 1), Fk);
                    const float M = key_value(top);
                    if (top == 0 || M != M) {
                        rec.flags |= SSD_DEV_NONFINITE;
                    } else {
                        rec.tk = key_id(top);
                        if (k < K) {
                            const int xt = P.tokens[static_cast<int64_t>(b) * K + k];
                            const float ztx = load_logit<D>(row_ptr(P.tgt, P.tgt_seq_stride, b, k), xt);
                            rec.accept = make_key(ztx, xt) > top ? 1 : 0;
                            rec.p_tok = rec.accept ? 1.f : 0.f;
                            rec.q_tok = 1.f;
                            rejected = !rec.accept;
                        }
                    }
                } else {
                    if (Fk > 0) merge_keys(b, k, all, Fk, Fk);
                    if (do_verify) {
                        const float tau = P.temperature[b];
                        const float c = kLog2e / tau;
                        float4 st4 = make_float4(-INFINITY, 0.f, 0.f, 0.f);
                        if (lane < S) st4 = __ldcg(P.sstat + static_cast<int64_t>(u) * S + lane);
                        Stat g{-INFINITY, 0.f};
                        for (int s = 0; s < S; ++s)
                            g = stat_merge_nan(g, Stat{__shfl_sync(kFull, st4.x, s), __shfl_sync(kFull, st4.y, s)});
                        if (!stat_ok(g)) {
                            rec.flags |= SSD_DEV_NONFINITE;
                        } else {
                            // slice p-masses relative to the row maximum, then the crossing slice's groups
                            const float wsl = (lane < S && st4.x != -INFINITY) ? st4.y * ex2(st4.x - g.m) : 0.f;
                            const double tot = __shfl_sync(kFull, warp_incl_scan(static_cast<double>(wsl), lane), 31);
                            const float uK = P.uniforms[static_cast<int64_t>(b) * (K + 1) + K];
                            const double T = static_cast<double>(uK) * tot;
                            double base = 0.0;
                            const int sc = slice_prefix(wsl, T, base);
                            int g0, gn;
                            slice_groups(sc, g0, gn);
                            const float *src = P.garr + static_cast<int64_t>(u) * 2 * GA + g0;
                            for (int gg = lane; gg < gn; gg += 32) {
                                sgmax[gg] = __ldcg(src + gg);
                                sgsum[gg] = __ldcg(src + GA + gg);
                            }
                            __syncwarp();
                            const unsigned char *trow = row_ptr(P.tgt, P.tgt_seq_stride, b, k);
                            const float Mc = g.m;
                            rec.tk = slice_crossing(
                                gn, g0, T - base,
                                [&](int gg) {
                                    const float gm = sgmax[gg];
                                    return (gm == -INFINITY) ? 0.f : sgsum[gg] * ex2(fmaf(gm, c, -Mc));
                                },
                                [&](int e) { return ex2(fmaf(load_logit<D>(trow, e), c, -Mc)); });
                        }
                    }
                }
            }
            complete_unit(b, k, rec, rejected && do_verify);
        };

        for (uint32_t j = 0;; ++j) {
            const int buf = static_cast<int>(j % kNBuf);
            if (!mbar_wait_suspend(&gs.tail_full[buf], (j / kNBuf) & 1)) {
                if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
                break;
            }
            const STail d = gs.desc[buf];
            if (d.kind == kTStop) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&gs.tail_empty[buf]);
                break;
            }
            float *gmax = arrays + buf * 2 * kGs;
            float *gsum = gmax + kGs;
            const int b = d.b, k = d.k, s = d.s;
            const int u = unit_of(b, k);
            int g0, gn;
            slice_groups(s, g0, gn);
            const int Fk = do_cache ? P.F[k] : 0;
            SliceUnitState *us = P.ustate + u;
            const unsigned char *trow = row_ptr(P.tgt, P.tgt_seq_stride, b, k);
            const unsigned char *drow = row_ptr(P.drf, P.drf_seq_stride, b, k);
            auto release = [&]() {
                __syncwarp();
                if (lane == 0) mbar_arrive(&gs.tail_empty[buf]);
            };
            auto copy_arrays = [&](bool both) {
                float *dst = P.garr + static_cast<int64_t>(u) * 2 * GA + g0;
                for (int g = lane; g < gn; g += 32) {
                    if (both) dst[g] = gmax[g];
                    dst[GA + g] = gsum[g];
                }
            };
            if (d.kind == kTPair1) {
                if (lane == 0)
                    P.sstat[static_cast<int64_t>(u) * S + s] = make_float4(d.m0, d.S0, d.m1, d.S1);
                if (d.flags == 0 && Fk > 0) {
                    // For the residual bound of the unit: each lane's two groups with the
                    // largest target maximum (target max, draft max), and every chunk's
                    // largest target maximum.  gsum holds the target maxima, gmax the draft's.
                    const int R = (gn + 31) / 32;
                    const int a0 = min(gn, lane * R), a1 = min(gn, a0 + R);
                    float t1 = -INFINITY, t2 = -INFINITY, d1 = 0.f, d2 = 0.f;
                    for (int g = a0; g < a1; ++g) {
                        const float tv = gsum[g];
                        if (tv > t1) {
                            t2 = t1;
                            d2 = d1;
                            t1 = tv;
                            d1 = gmax[g];
                        } else if (tv > t2) {
                            t2 = tv;
                            d2 = gmax[g];
                        }
                    }
                    float4 *pc = reinterpret_cast<float4 *>(P.pcand + (static_cast<int64_t>(u) * S + s) * kSliceCand * 2);
                    pc[lane] = make_float4(t1, d1, t2, d2);
                    const int c0 = 2 * slice_block0(s, S, nblk);
                    const int nch = min(2 * slice_block0(s + 1, S, nblk), npc) - c0;
                    if (lane < nch) {
                        float m = -INFINITY;
                        const int e1 = min(gn, (lane + 1) * GPR);
                        for (int g = lane * GPR; g < e1; ++g) m = fmaxf(m, gsum[g]);
                        P.cmax[static_cast<int64_t>(u) * npc + c0 + lane] = m;
                    }
                }
                release();
                if (lane == 0 && d.flags) atomicOr(&us->flags, static_cast<uint32_t>(d.flags));
                __threadfence();
                uint32_t cnt = 0;
                if (lane == 0) cnt = atomicAdd(&us->p1_done, 1u);
                cnt = __shfl_sync(kFull, cnt, 0);
                if (cnt == static_cast<uint32_t>(S - 1)) {
                    __threadfence();
                    finish_pair1(b, k);
                }
            } else if (d.kind == kTGreedy || d.kind == kTSampled) {
                const bool greedy = d.kind == kTGreedy;
                const int Fl = greedy ? max(Fk, 1) : Fk;
                if (d.flags == 0 && Fl > 0)
                    slice_topf(gmax, g0, gn, Fl, 0, d.xmask, trow, nullptr, 0.f, 0.f, 0.f, DraftShape{0, 0.f, 0, 0.f},
                               -INFINITY, key_area(b, s, k));
                if (!greedy && d.flags == 0 && do_verify) {
                    if (lane == 0) P.sstat[static_cast<int64_t>(u) * S + s] = make_float4(d.m0, d.S0, 0.f, 0.f);
                    copy_arrays(true);
                }
                release();
                if (lane == 0 && d.flags) atomicOr(&us->flags, static_cast<uint32_t>(d.flags));
                __threadfence();
                uint32_t cnt = 0;
                if (lane == 0) cnt = atomicAdd(&us->p1_done, 1u);
                cnt = __shfl_sync(kFull, cnt, 0);
                if (cnt == static_cast<uint32_t>(S - 1)) {
                    __threadfence();
                    finish_single(b, k, greedy);
                }
            } else if (d.kind == kTPair2) {
                if (Fk > 0)
                    slice_topf(gmax, g0, gn, Fk, 1, -1, trow, drow, d.c, -d.LT, d.LD, d.shape, d.cthr,
                               key_area(b, s, k));
                if (do_verify && !d.accept) {
                    float zs = 0.f;
                    for (int g = lane; g < gn; g += 32) zs += gsum[g];
                    // slice total in a fixed lane order, so that every run gives the same bits
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(kFull, zs, o);
                    if (lane == 0) P.sstat[static_cast<int64_t>(u) * S + s].x = zs;
                    copy_arrays(false);
                }
                release();
                __threadfence();
                uint32_t cnt = 0;
                if (lane == 0) cnt = atomicAdd(&us->p2_done, 1u);
                cnt = __shfl_sync(kFull, cnt, 0);
                if (cnt + 1 == __ldcg(&us->p2_expect)) {
                    __threadfence();
                    finish_pair2(b, k);
                }
            } else {  // skipped slice (an earlier position of the sequence already rejected)
                release();
                if (lane == 0) atomicOr(&us->flags, kSliceSkipped);
                __threadfence();
                uint32_t cnt = 0;
                if (lane == 0) cnt = atomicAdd(&us->p1_done, 1u);
                cnt = __shfl_sync(kFull, cnt, 0);
                if (cnt == static_cast<uint32_t>(S - 1)) {
                    __threadfence();
                    const float tau = P.temperature[b];
                    const bool smp = tau > 0.f && tau < INFINITY;
                    if (smp && k < K)
                        finish_pair1(b, k);
                    else
                        finish_single(b, k, !smp);
                }
            }
        }
        // this tail warp is done; the last one of the grid resets the scheduler counters
        if (lane == 0) {
            __threadfence();
            const uint32_t done = atomicAdd(P.slice_ctr + kCtrExit, 1u);
            if (done == gridDim.x * kNG - 1) {
                P.slice_ctr[kCtrP1] = 0;
                P.slice_ctr[kCtrQAlloc] = 0;
                P.slice_ctr[kCtrQClaim] = 0;
                P.slice_ctr[kCtrPairsDone] = 0;
                P.slice_ctr[kCtrExit] = 0;
            }
        }
        return;
    }

    // =========================== consumers ==================================
    const int grp = warp / kGW;
    SGroup &gs = gsh[grp];
    const int t = tid - grp * kGT;
    const int gw = warp - grp * kGW;
    const int bar_id = 1 + grp;
    auto gbar = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(kGT) : "memory"); };
    unsigned char *const ring = dyn_smem + grp * kRS * kSB;
    float *const arrays = reinterpret_cast<float *>(dyn_smem + kNG * kRS * kSB) + grp * kNBuf * 2 * kGs;

    const int p1_row = t / (kGT / 2), p1_tr = t % (kGT / 2);
    const int p1_vbase = p1_tr * VPT1, p1_rot = (p1_tr >> 1) & 3;
    const int s_gl = t / TPGS, s_part = t % TPGS;
    const int s_vbase = s_gl * GV + s_part * VPTS, s_rot = (t >> 1) & 3;
    const int r_gl = t / TPG2, r_part = t % TPG2;
    const int r_vbase = r_gl * GV + r_part * VPT2, r_rot = (t >> 2) & 1;

    uint32_t n = 0, nho = 0;
    int cur = -1;
    int b = 0, k = 0, sl = 0, flags = 0, xmask = -1, accept = 0, g0 = 0, pass_cur = 0;
    bool sampled = false, pair = false, active = false, bnd = false;
    float c = 0.f, LT = 0.f, LD = 0.f, cthr = -INFINITY;
    DraftShape shape{0, 0.f, 0, 0.f};
    Stat st{-INFINITY, 0.f};
    float *gmax = arrays, *gsum = arrays + kGs;

    auto handoff = [&](int kind, Stat a, Stat d2) {
        gbar();
        if (t == 0) {
            STail &D0 = gs.desc[nho % kNBuf];
            D0.kind = kind;
            D0.b = b;
            D0.k = k;
            D0.s = sl;
            D0.flags = flags;
            D0.xmask = xmask;
            D0.accept = accept;
            D0.c = c;
            D0.m0 = a.m;
            D0.S0 = a.S;
            D0.m1 = d2.m;
            D0.S1 = d2.S;
            D0.LT = LT;
            D0.LD = LD;
            D0.cthr = cthr;
            D0.shape = shape;
            mbar_arrive(&gs.tail_full[nho % kNBuf]);
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
        // the stage's own fields every time; the item's inputs only when it starts (the
        // slot stays this group's until its warps arrive on empty_bar below)
        const int4 hq = *reinterpret_cast<const int4 *>(&gs.hdr[s]);  // item, code, chunk, nvec
        struct {
            int item, code, chunk, nvec;
        } h{hq.x, hq.y, hq.z, hq.w};
        const int pass = h.code & 15;
        if (pass == kPassStop) break;
        if (h.item != cur) {
            const SHdr &hu = gs.hdr[s];
            // a new item: wait for its group-array buffer, then its constants
            if (!mbar_wait_suspend(&gs.tail_empty[nho % kNBuf], ((nho / kNBuf) & 1) ^ 1)) {
                atomicOr(&s_abort, 1);
                if (t == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
                break;
            }
            cur = h.item;
            pass_cur = pass;
            b = hu.b;
            k = hu.k;
            sl = hu.s;
            gmax = arrays + (nho % kNBuf) * 2 * kGs;
            gsum = gmax + kGs;
            g0 = slice_block0(sl, S, nblk) * GPS;
            const float tau = hu.tau;
            const bool tau_ok = (tau >= 0.f) && (tau < INFINITY);
            const bool greedy = tau_ok && tau == 0.f;
            sampled = tau_ok && tau > 0.f;
            pair = sampled && k < K;
            flags = tau_ok ? 0 : SSD_DEV_BAD_TEMPERATURE;
            const int xt = hu.xt;
            if (k < K && (xt < 0 || xt >= V)) flags |= SSD_DEV_BAD_TOKEN;
            xmask = (greedy && k < K) ? xt : -1;
            active = flags == 0;
            bnd = pair && do_cache && P.F[k] > 0;
            c = sampled ? kLog2e / tau : 0.f;
            shape = DraftShape{0, 0.f, 0, 0.f};
            if (pair && P.reshape) {
                const ssd_reshape_desc dd = P.reshape[static_cast<int64_t>(b) * K + k];
                shape.on = dd.F > 0;
                shape.thr = dd.thr_val;
                shape.thr_id = dd.thr_id;
                shape.l2C = dd.C > 0.f ? (dd.C == 1.f ? 0.f : lg2(dd.C)) : -INFINITY;
            }
            st = Stat{-INFINITY, 0.f};
            accept = 0;
            LT = 0.f;
            LD = 0.f;
            cthr = -INFINITY;
            if (pass == kPassP2) {
                LT = hu.LT;
                LD = hu.LD;
                cthr = hu.cthr;
                accept = hu.accept;
                // groups of chunks that are not streamed read as empty (no residual)
                int gs0, gsn;
                {
                    const int bl0 = slice_block0(sl, S, nblk), bl1 = slice_block0(sl + 1, S, nblk);
                    gs0 = bl0 * GPS;
                    gsn = min(bl1 * GPS, G) - gs0;
                }
                for (int i = t; i < gsn; i += kGT) {
                    gmax[i] = 0.f;
                    gsum[i] = 0.f;
                }
                gbar();
            }
        }
        if (pass == kPassSkip) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&gs.empty_bar[s]);
            ++n;
            handoff(kTSkip, st, st);
            continue;
        }
        const unsigned char *stg = ring + s * kSB;
        const bool stage_pair = (h.code >> 5) & 1;
        if (active) {
            if (pass == kPassP1 && stage_pair) {
                uint4 w[VPT1];
                load_vecs<D, VPT1>(stg + p1_row * HALF, p1_vbase, h.nvec, p1_rot, h.nvec == FULL_PAIR, w);
                const float rm = vecs_max<D, VPT1>(w);
                if (bnd) {
                    // raw group maxima: the draft's to gmax (the bound on q), the target's to gsum (on p)
                    const float gm = tpg_max<TPG1>(rm);
                    const int g = h.chunk * GPR + p1_tr / TPG1;
                    if (p1_tr % TPG1 == 0 && g < G) (p1_row ? gmax : gsum)[g - g0] = canon_zero(gm);
                }
                if (p1_row == 0 || !shape.on || !(rm >= shape.thr)) {
                    stat_fold(st, rm * c, [&](float mn) { return vecs_expsum<D, VPT1>(w, c, mn); });
                } else {
                    st = reshaped_fold<D, VPT1>(st, stg + HALF, p1_vbase, h.nvec, p1_rot, h.nvec == FULL_PAIR, c, shape,
                                                h.chunk * (FULL_PAIR * VEC) + p1_vbase * VEC, -1, 0);
                }
            } else if (pass == kPassP1) {
                uint4 w[VPTS];
                load_vecs<D, VPTS>(stg, s_vbase, h.nvec, s_rot, h.nvec == FULL_ONE, w);
                const int e0 = h.chunk * (FULL_ONE * VEC) + s_vbase * VEC;
                if (static_cast<unsigned>(xmask - e0) < static_cast<unsigned>(VPTS * VEC)) {
#pragma unroll
                    for (int kk = 0; kk < VPTS; ++kk) {
                        const int ev = e0 + ((kk + s_rot) & (VPTS - 1)) * VEC;
                        if (static_cast<unsigned>(xmask - ev) < static_cast<unsigned>(VEC))
                            mask_vec<D>(w[kk], ev, 0, V, xmask);
                    }
                }
                const float gm = tpg_max_nan<TPGS>(vecs_max<D, VPTS>(w));
                const int g = h.chunk * GPS + s_gl;
                if (sampled) {
                    const float gmc = gm * c;
                    const float vs = vecs_expsum<D, VPTS>(w, c, gmc);
                    const float gsum_all = tpg_sum<TPGS>(vs);
                    const float gsv = (gm == -INFINITY) ? 0.f : gsum_all;
                    const bool lead = s_part == 0 && gm != -INFINITY;
                    st = stat_merge_nan(st, Stat{lead ? gmc : -INFINITY, lead ? gsv : 0.f});
                    if (s_part == 0 && g < G) {
                        gmax[g - g0] = canon_zero(gm);
                        gsum[g - g0] = gsv;
                    }
                } else if (s_part == 0 && g < G) {
                    gmax[g - g0] = canon_zero(gm);
                }
            } else {
                // second pass of a pair: residual masses and maxima of every group of the stage
                const bool full = h.nvec == FULL_PAIR;
                float2 acc = make_float2(0.f, 0.f);
                float mx = 0.f;
                const int g = h.chunk * GPR + r_gl;
                uint4 wt[VPT2], wd[VPT2];
                load_vecs<D, VPT2>(stg, r_vbase, h.nvec, r_rot, full, wt);
                load_vecs<D, VPT2>(stg + HALF, r_vbase, h.nvec, r_rot, full, wd);
                if (!shape.on || !(vecs_max<D, VPT2>(wd) >= shape.thr)) {
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
                            const float2 dd = __ffma2_rn(make_float2(ex2(x0.y), ex2(x1.y)), make_float2(-1.f, -1.f),
                                                         make_float2(ex2(x0.x), ex2(x1.x)));
                            const float w0 = fmaxf(dd.x, 0.f), w1 = fmaxf(dd.y, 0.f);
                            acc = __fadd2_rn(acc, make_float2(w0, w1));
                            mx = fmaxf(mx, fmaxf(w0, w1));
                        }
                    }
                } else {
                    const float2 r2 = reshaped_resid<D, VPT2>(stg, HALF, r_vbase, h.nvec, r_rot, full, c, LT, LD, shape,
                                                              h.chunk * (FULL_PAIR * VEC) + r_vbase * VEC, -1, 0);
                    acc.x = r2.x;
                    mx = r2.y;
                }
                const float gsv = tpg_sum<TPG2>(acc.x + acc.y);
                const float gmx = tpg_max<TPG2>(mx);
                if (r_part == 0 && g < G) {
                    gmax[g - g0] = gmx;
                    gsum[g - g0] = gsv;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&gs.empty_bar[s]);
        ++n;
        if (!((h.code >> 4) & 1)) continue;

        // ---- end of the item ----------------------------------------------------
        const Stat none{-INFINITY, 0.f};
        if (pass_cur == kPassP2) {
            handoff(kTPair2, none, none);
            continue;
        }
        if (!active) {
            handoff(pair ? kTPair1 : (sampled ? kTSampled : kTGreedy), none, none);
            continue;
        }
        if (pair) {
            // warps 0-3 hold the target statistics, 4-7 the draft's
            const Stat ws = warp_stat(st);
            gbar();
            if (lane == 0) gs.red[gw] = ws;
            gbar();
            Stat gT = gs.red[0], gD = gs.red[kGW / 2];
#pragma unroll
            for (int w = 1; w < kGW / 2; ++w) {
                gT = stat_merge_nan(gT, gs.red[w]);
                gD = stat_merge_nan(gD, gs.red[kGW / 2 + w]);
            }
            handoff(kTPair1, gT, gD);
            continue;
        }
        if (sampled) {
            const Stat ws = warp_stat(st);
            gbar();
            if (lane == 0) gs.red[gw] = ws;
            gbar();
            Stat gT = gs.red[0];
#pragma unroll
            for (int w = 1; w < kGW; ++w) gT = stat_merge_nan(gT, gs.red[w]);
            handoff(kTSampled, gT, none);
            continue;
        }
        handoff(kTGreedy, none, none);
    }

    // this group is done: tell its tail warp
    if (!mbar_wait_suspend(&gs.tail_empty[nho % kNBuf], ((nho / kNBuf) & 1) ^ 1)) {
        if (t == 0 && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
    }
    const Stat none{-INFINITY, 0.f};
    handoff(kTStop, none, none);
}

template <class D>
int slice_setup_d(size_t optin, size_t *max_dyn) {
    bool dummy = true;
    return setup_kernel(ssd_slice_kernel<D>, optin, max_dyn, &dummy);
}

int slice_setup(int dtype, size_t optin, size_t *max_dyn) {
    return dtype == SSD_F32 ? slice_setup_d<F32Tag>(optin, max_dyn) : slice_setup_d<BF16Tag>(optin, max_dyn);
}

int slice_launch(int dtype, const UnitParams &P, int grid, size_t dyn, void *stream) {
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
    const cudaError_t e = dtype == SSD_F32 ? cudaLaunchKernelEx(&cfg, ssd_slice_kernel<F32Tag>, P)
                                           : cudaLaunchKernelEx(&cfg, ssd_slice_kernel<BF16Tag>, P);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SSD_ERR_CUDA;
    }
    return SSD_OK;
}

}  // namespace ssd
