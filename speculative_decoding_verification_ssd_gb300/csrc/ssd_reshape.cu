// ssd_reshape.cu -- sigma_{F,C} reshaping of draft rows (sm_103a).
//
// [SSD] "Speculative Speculative Decoding" notes (papernotes.org), "关键设计"
// item 2 (SAGUARO sampling): given draft logits z, fan-out F and C in [0, 1],
// sigma_{F,C}(z)_t is proportional to C exp(z_t) for the F largest logits and
// to exp(z_t) otherwise.  Temperature is applied first (z -> z / tau); the set
// is taken on the raw logits (ties to the lowest id), so it is the same for
// every tau > 0.
//
// One thread-block cluster per row.  Each CTA stages its vocabulary slice in
// shared memory (one bulk copy), selects its local top-(F+1) by (value, id),
// and the cluster ranks the local lists against each other to find the F-th
// largest key (the descriptor threshold) and the (F+1)-th (the largest
// non-member, which fixes the shift of the reshaped softmax).  When q' is
// requested, two more passes over the staged slice give the normaliser and
// write q'_t = c_t 2^(x_t - m') / S'.
//
// Draft-cache mode runs the same selection on the K+1 draft rows of every
// sequence with F = F_k at position k and also writes segment k of the
// speculation cache: the F_k tokens of largest raw draft logit (ties to the
// lowest id), best first, with the drafted token x~_k left out for k < K
// (a bonus drawn after rejecting x~_k is never x~_k).  These are the cache
// keys the notes' item 2 describes as chosen from the draft logits; the
// per-position descriptors are the sigma_{F_k,C} reshape of the same rows.
#include <cooperative_groups.h>

#include <climits>

#include "ssd_device.cuh"
#include "ssd_launch.cuh"
#include "ssd_reshape.cuh"
#include "ssd_vec.cuh"

namespace cg = cooperative_groups;

namespace ssd {
namespace {
constexpr float kLog2e = 1.4426950408889634f;

struct RXchg {
    int nlist;
    int xpos;          // global rank of the excluded token (INT_MAX when not in the lists)
    float ssum;
    uint64_t slot[3];  // written by peers into rank 0: keys of global rank 0, F-1, F
};
}  // namespace

template <class D>
__global__ void __launch_bounds__(kThreads)
    ssd_reshape_kernel(const __grid_constant__ ReshapeParams P) {
    constexpr int VEC = D::kVec, S = D::kBytes;
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ __align__(16) uint64_t cand[kCandCap];
    __shared__ int cpos[kCandCap];
    __shared__ RXchg xc;
    __shared__ __align__(8) uint64_t bar;
    __shared__ float red_f[kWarps];
    __shared__ int s_cnt;
    __shared__ int s_timeout;

    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x;
    const int CL = P.CL;
    const int rank = static_cast<int>(cluster.block_rank());
    const int row = blockIdx.x / CL;
    const int V = P.V;
    const int lo = min(V, rank * P.slice), hi = min(V, lo + P.slice);
    const int seq = P.seq_rows > 0 ? row / P.seq_rows : row;
    const int pos_k = P.seq_rows > 0 ? row - seq * P.seq_rows : 0;
    const int F = P.seq_rows > 0 ? P.Fk[pos_k] : P.F;
    const int xt = (P.seq_rows > 0 && P.tokens && pos_k < P.K)
                       ? __ldg(P.tokens + static_cast<int64_t>(seq) * P.K + pos_k) : -1;
    const unsigned char *grow =
        static_cast<const unsigned char *>(P.drf) + static_cast<int64_t>(row) * V * S;

    // ---- staging (same placement rule as the verify kernel) ---------------
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(grow) + static_cast<uintptr_t>(lo) * S;
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(grow) + static_cast<uintptr_t>(hi) * S;
    const uintptr_t base = a0 & ~static_cast<uintptr_t>(15);
    const int lead = static_cast<int>((a0 - base) / S);
    const int n = hi - lo;
    const int ebase = lo - lead;
    const int nv = n > 0 ? (lead + n + VEC - 1) / VEC : 0;
    unsigned char *buf = dyn_smem;
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        s_timeout = 0;
        xc.xpos = INT_MAX;
        xc.slot[0] = xc.slot[1] = xc.slot[2] = 0;
    }
    __syncthreads();
    {
        const uintptr_t c0 = (a0 + 15) & ~static_cast<uintptr_t>(15);
        const uintptr_t c1 = a1 & ~static_cast<uintptr_t>(15);
        uintptr_t h1 = a1, t0 = a1;
        uint32_t bulk = 0;
        if (n > 0 && c1 > c0) {
            h1 = c0;
            t0 = c1;
            bulk = static_cast<uint32_t>(c1 - c0);
        }
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar, bulk);
            if (bulk) bulk_copy_g2s(buf + (c0 - base), reinterpret_cast<const void *>(c0), bulk, &bar);
        }
        const int nh = n > 0 ? static_cast<int>((h1 - a0) / S) : 0;
        const int nt = n > 0 ? static_cast<int>((a1 - t0) / S) : 0;
        for (int i = tid; i < nh + nt; i += kThreads) {
            const uintptr_t ga = i < nh ? a0 + static_cast<uintptr_t>(i) * S
                                        : t0 + static_cast<uintptr_t>(i - nh) * S;
            if (S == 4)
                *reinterpret_cast<uint32_t *>(buf + (ga - base)) =
                    __ldg(reinterpret_cast<const uint32_t *>(ga));
            else
                *reinterpret_cast<uint16_t *>(buf + (ga - base)) =
                    __ldg(reinterpret_cast<const unsigned short *>(ga));
        }
    }
    __syncthreads();
    if (!mbar_wait_bounded(&bar, 0)) atomicOr(&s_timeout, 1);
    __syncthreads();

    auto vec = [&](int v, float (&z)[VEC]) {
        decode_vec<D>(*reinterpret_cast<const uint4 *>(buf + 16 * v), z);
    };

    // ---- local top-(F+1) by raw (value, id) --------------------------------
    // Vectors wholly inside [lo, hi) go through packed maxima and lane masks; the
    // two boundary vectors of the slice element by element.
    auto inside = [&](int v) { return ebase + v * VEC >= lo && ebase + v * VEC + VEC <= hi; };
    float tmax = -INFINITY;
    {
        RawMax<D> rm;
        for (int v = tid; v < nv; v += kThreads) {
            if (inside(v)) {
                rm.add(*reinterpret_cast<const uint4 *>(buf + 16 * v));
            } else {
                float z[VEC];
                vec(v, z);
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const int e = ebase + v * VEC + i;
                    if (e >= lo && e < hi) tmax = fmax_nan(tmax, z[i]);
                }
            }
        }
        tmax = fmax_nan(tmax, rm.get());
    }
    // id V ranks below every token of value tmax: a lower bound on the thread's best key
    const uint64_t tb = (tmax == -INFINITY) ? 0 : make_key(tmax, V);
    const int Fsel = F + 1;
    const int nlist = block_topf_fast(
        Fsel, tb,
        [&](uint64_t theta, auto emit) {
            const uint32_t tv = static_cast<uint32_t>(theta >> 32);
            // every token whose key reaches theta is at or above this storage value
            const float tstore = tv ? round_down_storage<D>(value_of_ordered(tv)) : -INFINITY;
            for (int v = tid; v < nv; v += kThreads) {
                const uint4 w = *reinterpret_cast<const uint4 *>(buf + 16 * v);
                const bool in = inside(v);
                uint32_t m = in ? ge_lanes<D>(w, tstore) : ((1u << VEC) - 1u);
                if (!m) continue;
                float z[VEC];
                decode_vec<D>(w, z);
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const int e = ebase + v * VEC + i;
                    if (((m >> i) & 1u) && e >= lo && e < hi && ordered_bits(z[i]) >= tv) {
                        const uint64_t key = make_key(z[i], e);
                        if (key >= theta) emit(key);
                    }
                }
            }
        },
        cand, &s_cnt);
    if (tid == 0) xc.nlist = nlist;
    cluster.sync();

    // Global rank of each own entry; ranks 0, F-1 and F are posted to rank 0.
    for (int i = tid; i < nlist; i += kThreads) {
        const uint64_t key = cand[i];
        int pos = i;
        for (int j = 0; j < CL; ++j) {
            if (j == rank) continue;
            const RXchg *px = cluster.map_shared_rank(&xc, j);
            const uint64_t *pl = cluster.map_shared_rank(cand, j);
            int l = 0, h = px->nlist;
            while (l < h) {
                const int mid = (l + h) >> 1;
                if (pl[mid] > key)
                    l = mid + 1;
                else
                    h = mid;
            }
            pos += l;
        }
        RXchg *r0 = cluster.map_shared_rank(&xc, 0);
        cpos[i] = pos;
        if (pos == 0) r0->slot[0] = key;
        if (F > 0 && pos == F - 1) r0->slot[1] = key;
        if (pos == F) r0->slot[2] = key;
        if (static_cast<int>(key_id(key)) == xt) r0->xpos = pos;
    }
    cluster.sync();
    const RXchg *r0 = cluster.map_shared_rank(&xc, 0);
    const uint64_t top1 = r0->slot[0], thr = r0->slot[1], next = r0->slot[2];
    const bool timed_out = s_timeout != 0;

    ssd_reshape_desc d;
    d.F = F;
    d.C = P.C;
    if (F > 0) {
        d.thr_val = key_value(thr);
        d.thr_id = key_id(thr);
    } else {
        d.thr_val = INFINITY;
        d.thr_id = -1;
    }
    if (rank == 0 && tid == 0) {
        if (P.desc && P.seq_rows == 0)
            P.desc[row] = d;
        else if (P.desc && pos_k < P.K)
            P.desc[static_cast<int64_t>(seq) * P.K + pos_k] = d;
        if (timed_out && P.dev_status) atomicOr(P.dev_status, SSD_DEV_TIMEOUT);
    }
    if (P.cache_tok) {
        // ranks 0..F of the row, the excluded token dropped: slot = rank minus one
        // past the excluded token's rank; slots left over (F_k = V with a token
        // excluded) hold -1
        int32_t *seg = P.cache_tok + static_cast<int64_t>(seq) * P.budget + P.off[pos_k];
        const int xpos = r0->xpos;
        for (int i = tid; i < nlist; i += kThreads) {
            const int pos = cpos[i];
            if (pos == xpos) continue;
            const int slot = pos - (xpos < pos ? 1 : 0);
            if (slot < F) seg[slot] = static_cast<int32_t>(key_id(cand[i]));
        }
        if (rank == 0) {
            const int avail = V - ((xt >= 0 && xt < V) ? 1 : 0);
            for (int j = avail + tid; j < F; j += kThreads) seg[j] = -1;
        }
    }

    if (P.q_out) {
        const float tau = P.tau[row];
        const float c = kLog2e / tau;
        const float l2C = P.C > 0.f ? (P.C == 1.f ? 0.f : lg2(P.C)) : -INFINITY;
        // shift m' = max over weighted tokens of x_t + log2 c_t
        float mprime;
        const float xtop = key_value(top1) * c;
        if (F == 0)
            mprime = xtop;
        else {
            const float xnext = next ? key_value(next) * c : -INFINITY;
            mprime = fmaxf(xtop + l2C, xnext);
        }
        auto wx = [&](float z, int e) -> float {  // log2 of the unnormalised weight
            const bool mem = F > 0 && (z > d.thr_val || (z == d.thr_val && e <= d.thr_id));
            return z * c + (mem ? l2C : 0.f) - mprime;
        };
        float acc = 0.f;
        for (int v = tid; v < nv; v += kThreads) {
            float z[VEC];
            vec(v, z);
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                const int e = ebase + v * VEC + i;
                if (e >= lo && e < hi) acc += ex2(wx(z[i], e));
            }
        }
        acc = block_sum(acc, red_f);
        if (tid == 0) xc.ssum = acc;
        cluster.sync();
        float Ssum = 0.f;
        for (int j = 0; j < CL; ++j) Ssum += cluster.map_shared_rank(&xc, j)->ssum;
        const float inv = 1.f / Ssum;
        float *out = P.q_out + static_cast<int64_t>(row) * V;
        for (int v = tid; v < nv; v += kThreads) {
            float z[VEC];
            vec(v, z);
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                const int e = ebase + v * VEC + i;
                if (e >= lo && e < hi) out[e] = ex2(wx(z[i], e)) * inv;
            }
        }
    }
    cluster.sync();  // peers done reading this CTA's shared memory
}

int reshape_setup(int dtype, size_t optin, size_t *max_dyn, bool *allow16) {
    return dtype == SSD_F32 ? setup_kernel(ssd_reshape_kernel<F32Tag>, optin, max_dyn, allow16)
                            : setup_kernel(ssd_reshape_kernel<BF16Tag>, optin, max_dyn, allow16);
}

int reshape_launch(int dtype, const ReshapeParams &P, int grid, int CL, size_t dyn, void *stream) {
    return dtype == SSD_F32
               ? launch_clustered(ssd_reshape_kernel<F32Tag>, P, grid, CL, dyn, stream)
               : launch_clustered(ssd_reshape_kernel<BF16Tag>, P, grid, CL, dyn, stream);
}

__global__ void ssd_lookup_kernel(const __grid_constant__ LookupParams P) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= P.B) return;
    const int a = P.accept_len[b];
    const int t = P.bonus[b];
    int s = -1;
    if (a >= 0 && a <= P.K) {
        const int32_t *row = P.cache_tok + static_cast<int64_t>(b) * P.budget;
        for (int j = P.off[a]; j < P.off[a + 1]; ++j) {
            if (row[j] == t) {
                s = j;
                break;
            }
        }
    }
    P.hit[b] = s >= 0 ? 1 : 0;
    P.slot[b] = s;
}

int lookup_launch(const LookupParams &P, void *stream) {
    const int threads = 128;
    ssd_lookup_kernel<<<(P.B + threads - 1) / threads, threads, 0,
                        static_cast<cudaStream_t>(stream)>>>(P);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace ssd
