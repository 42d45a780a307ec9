// ssd_api.cu -- the C ABI of libssd (declared in include/ssd.h): host-side
// validation, launch geometry and kernel launches.  No entry point allocates
// or frees memory or synchronises the stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/ssd.h"
#include "ssd_device.cuh"
#include "ssd_launch.cuh"
#include "ssd_reshape.cuh"
#include "ssd_slice.cuh"
#include "ssd_stream.cuh"
#include "ssd_unit.cuh"

namespace {

constexpr int kMaxDevices = 64;

// Per-device facts and one-time kernel attribute set-up.
struct DeviceInfo {
    bool ready = false;
    int status = SSD_OK;
    int sm_count = 0;
    int max_cluster = 8;       // 16 when the non-portable size is available
    size_t max_dyn[8] = {0};   // max dynamic smem: unit, reshape, stream, slice (f32 / bf16 each)
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

int device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SSD_ERR_CUDA;
        if (prop.major < 10) return SSD_ERR_UNSUPPORTED;
        d.sm_count = prop.multiProcessorCount;
        const size_t optin = prop.sharedMemPerBlockOptin;
        bool allow16 = true;
        int st = SSD_OK;
        st = st ? st : ssd::unit_setup(SSD_F32, optin, &d.max_dyn[0], &allow16);
        st = st ? st : ssd::unit_setup(SSD_BF16, optin, &d.max_dyn[1], &allow16);
        st = st ? st : ssd::reshape_setup(SSD_F32, optin, &d.max_dyn[2], &allow16);
        st = st ? st : ssd::reshape_setup(SSD_BF16, optin, &d.max_dyn[3], &allow16);
        st = st ? st : ssd::stream_setup(SSD_F32, optin, &d.max_dyn[4]);
        st = st ? st : ssd::stream_setup(SSD_BF16, optin, &d.max_dyn[5]);
        st = st ? st : ssd::slice_setup(SSD_F32, optin, &d.max_dyn[6]);
        st = st ? st : ssd::slice_setup(SSD_BF16, optin, &d.max_dyn[7]);
        if (st != SSD_OK) return st;
        d.max_cluster = allow16 ? 16 : 8;
        d.ready = true;
    }
    *out = &d;
    return SSD_OK;
}

struct Geometry {
    int CL = 0;
    int slice = 0;
    int row_buf_bytes = 0;
    size_t dyn = 0;
};

int ceil_div(int a, int b) { return (a + b - 1) / b; }
int round_up(int a, int b) { return ceil_div(a, b) * b; }

// Chooses the cluster size CL and the per-CTA vocabulary slice.  Prefers the
// smallest cluster whose staged rows leave room for 3 (then 2, then 1) CTAs
// per SM, then widens the cluster while the grid would not fill the GPU.
int choose_geometry(int V, int elem, int rows_staged, int units, const DeviceInfo &dv,
                    size_t max_dyn, Geometry *g) {
    const int vec = 16 / elem;
    auto make = [&](int CL) {
        Geometry r;
        r.CL = CL;
        r.slice = round_up(ceil_div(V, CL), vec);
        r.row_buf_bytes = round_up(r.slice * elem + 64, 128);
        r.dyn = static_cast<size_t>(rows_staged) * r.row_buf_bytes;
        return r;
    };
    const size_t tiers[3] = {68 * 1024, 100 * 1024, max_dyn};
    Geometry pick;
    bool found = false;
    for (int t = 0; t < 3 && !found; ++t) {
        for (int CL = 1; CL <= dv.max_cluster; CL <<= 1) {
            Geometry cand = make(CL);
            if (cand.dyn <= tiers[t] && cand.dyn <= max_dyn) {
                pick = cand;
                found = true;
                break;
            }
        }
    }
    if (!found) return SSD_ERR_UNSUPPORTED;
    while (static_cast<long long>(units) * pick.CL < 2LL * dv.sm_count &&
           pick.CL < dv.max_cluster && pick.slice >= 2048) {
        pick = make(pick.CL * 2);
    }
    if (static_cast<long long>(units) * pick.CL > INT_MAX) return SSD_ERR_UNSUPPORTED;
    *g = pick;
    return SSD_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int gcd(int a, int b) { return b == 0 ? a : gcd(b, a % b); }

// A multiplier coprime to B near 0.618 B: the streaming kernel visits sequence
// (i * m) % B for the i-th unit of a position, which interleaves sequences of
// different kinds (greedy / sampled) across the persistent CTAs.
int coprime_stride(int B) {
    if (B <= 2) return 1;
    for (int m = static_cast<int>(0.618 * B); m > 1; --m)
        if (gcd(m, B) == 1) return m;
    return 1;
}

int check_fanout(const int32_t *F_host, int K, int V, int budget, int *off) {
    if (!F_host) return SSD_ERR_INVALID_ARG;
    off[0] = 0;
    for (int k = 0; k <= K; ++k) {
        const int f = F_host[k];
        if (f < 0 || f > SSD_MAX_F || f > V) return SSD_ERR_INVALID_ARG;
        off[k + 1] = off[k] + f;
    }
    if (budget < off[K + 1]) return SSD_ERR_INVALID_ARG;
    return SSD_OK;
}

// Kernel choice for aligned rows (ssd_set_dispatch).
std::atomic<int> g_dispatch{SSD_DISPATCH_AUTO};
// The kernel the calling thread's last verify / cache / round call launched.
thread_local const char *t_last_kernel = "none";

// Shared driver of ssd_verify / ssd_build_cache / ssd_round.
int run_units(int mode, const void *tgt, const void *drf, int dtype, int B, int K, int V,
              int drf_rows, const int32_t *tokens, const float *uniforms, const float *temperature,
              const ssd_reshape_desc *reshape, const int32_t *F_host, int budget,
              int32_t *accept_len, int32_t *bonus, float *p_tok, float *q_tok, int32_t *cache_tok,
              uint8_t *hit, int32_t *slot, void *workspace, size_t workspace_bytes,
              int32_t *dev_status, void *stream, const int32_t *sig_F = nullptr, float sig_C = 1.f,
              ssd_reshape_desc *desc_out = nullptr, int64_t ld = -1) {
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_DTYPE;
    if (B < 1 || K < 1 || K > SSD_MAX_K || V < 2) return SSD_ERR_INVALID_ARG;
    if (drf_rows != K && drf_rows != K + 1) return SSD_ERR_INVALID_ARG;
    if (ld < 0) ld = V;
    if (ld < V) return SSD_ERR_INVALID_ARG;
    if (sig_F && ld != V) return SSD_ERR_INVALID_ARG;  // descriptors are found on contiguous rows
    if (sig_F) {
        // sigma_{F_k,C} found in the pass: no descriptors in, descriptors out
        if (reshape || !desc_out) return SSD_ERR_INVALID_ARG;
        if (!(sig_C >= 0.f && sig_C <= 1.f)) return SSD_ERR_INVALID_ARG;
        for (int k = 0; k < K; ++k) {
            if (sig_F[k] < 0 || sig_F[k] > SSD_MAX_F || sig_F[k] > V) return SSD_ERR_INVALID_ARG;
            if (sig_C == 0.f && sig_F[k] >= V) return SSD_ERR_INVALID_ARG;
        }
    }
    if (!tgt || !temperature || !tokens) return SSD_ERR_INVALID_ARG;
    const bool verify = (mode & ssd::kModeVerify) != 0;
    const bool cache = (mode & ssd::kModeCache) != 0;
    if (!drf) return SSD_ERR_INVALID_ARG;
    if (verify && (!uniforms || !accept_len || !bonus)) return SSD_ERR_INVALID_ARG;
    if ((p_tok == nullptr) != (q_tok == nullptr)) return SSD_ERR_INVALID_ARG;
    if ((mode & ssd::kModeLookup) && (!hit || !slot)) return SSD_ERR_INVALID_ARG;
    if (V > (dtype == SSD_F32 ? SSD_MAX_V_F32 : SSD_MAX_V_BF16)) return SSD_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * (K + 1) > INT_MAX / 16) return SSD_ERR_UNSUPPORTED;
    ssd::UnitParams P = {};
    if (cache) {
        const int st = check_fanout(F_host, K, V, budget, P.off);
        if (st != SSD_OK) return st;
        if (P.off[K + 1] > 0 && !cache_tok) return SSD_ERR_INVALID_ARG;
        for (int k = 0; k <= K; ++k) P.F[k] = F_host[k];
    }
    if (!workspace || !aligned(workspace, 256)) return SSD_ERR_WORKSPACE;
    if (workspace_bytes < ssd::ws_total_bytes(B, K)) return SSD_ERR_WORKSPACE;

    DeviceInfo *dv = nullptr;
    int st = device_info(&dv);
    if (st != SSD_OK) return st;
    const int elem = dtype == SSD_F32 ? 4 : 2;
    const int units = B * (K + 1);
    // The persistent streaming kernel needs every row on a 16-byte boundary and
    // its per-group arrays within shared memory; other inputs take the cluster kernel.
    const size_t sdyn = ssd::stream_dyn_bytes(V, sig_F != nullptr);
    // rows on the 16-byte grid, each row readable as whole 16-byte vectors
    const bool stream_ok = aligned(tgt, 16) && aligned(drf, 16) && (ld * elem) % 16 == 0 &&
                           ld >= round_up(V, 16 / elem) &&
                           (V + ssd::kGroupTokens - 1) / ssd::kGroupTokens <= ssd::kStreamMaxGroups &&
                           sdyn <= dv->max_dyn[dtype == SSD_F32 ? 4 : 5];
    // With fewer units than SMs the persistent kernel leaves SMs idle and each unit
    // streams at one group's share of an SM; the cluster kernel splits every row
    // across a cluster instead (c2: 8 sequences, K = 5: 38.5 us against 58.7), and
    // so does the streaming kernel's wide form, which puts both consumer groups of
    // a CTA on each unit.  The wide form pays where units are few for the grid:
    // verification alone below 8 units per SM (c3, 576 units: 82.5 against 96.0 us;
    // c2: 38.4 against 37.8 on the cluster kernel; 1280 units: 89.8 against 87.5
    // for the one-group form) and cache builds below 2 units per SM (c4: 112.5
    // against 119.0); with more units the one-group form's two units per SM keep
    // the HBM stream busier.
    const int policy = g_dispatch.load(std::memory_order_relaxed);
    // The slice kernel (rows split into slices scheduled over every SM) needs rows of
    // whole vectors, its own workspace regions and a batch it can order by kind.
    const int key_stride = ssd::slice_key_stride(K, cache ? F_host : nullptr);
    const ssd::SliceWs SW = ssd::slice_ws_layout(B, K, V, elem, key_stride);
    const bool slice_ok = stream_ok && sig_F == nullptr && V % (16 / elem) == 0 && B <= 2048 &&
                          ssd::slice_pair_chunks(V, elem) <= 96 &&
                          workspace_bytes >= SW.total && ssd::slice_dyn_bytes() <= dv->max_dyn[dtype == SSD_F32 ? 6 : 7];
    const bool sliced = slice_ok && policy == SSD_DISPATCH_SLICE;
    const bool wide = !sliced && stream_ok && V % (16 / elem) == 0 &&
                      (policy == SSD_DISPATCH_WIDE ||
                       (policy == SSD_DISPATCH_AUTO &&
                        ((verify && !cache && units < 8 * dv->sm_count) ||
                         (units >= dv->sm_count && units < 2 * dv->sm_count))));
    const bool streaming = !sliced && stream_ok && policy != SSD_DISPATCH_CLUSTER &&
                           (wide || policy == SSD_DISPATCH_STREAM || sig_F != nullptr || units >= dv->sm_count);
    Geometry g;
    if (!streaming && !sliced) {
        st = choose_geometry(V, elem, 2, units, *dv, dv->max_dyn[dtype == SSD_F32 ? 0 : 1], &g);
        if (st != SSD_OK) return st;
    }

    P.tgt = tgt;
    P.drf = drf;
    P.ld = ld;
    P.tgt_seq_stride = static_cast<int64_t>(K + 1) * ld;
    P.drf_seq_stride = static_cast<int64_t>(drf_rows) * ld;
    P.B = B;
    P.K = K;
    P.V = V;
    P.CL = g.CL;
    P.slice = g.slice;
    P.row_buf_bytes = g.row_buf_bytes;
    P.mode = mode;
    if (verify && !cache) P.mode |= ssd::kModeEarlyExit;
    P.tokens = tokens;
    P.uniforms = uniforms;
    P.temperature = temperature;
    P.reshape = reshape;
    P.budget = budget;
    P.cache_tok = cache_tok;
    P.accept_len = accept_len;
    P.bonus = bonus;
    P.p_tok = p_tok;
    P.q_tok = q_tok;
    P.hit = hit;
    P.slot = slot;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    P.rec = reinterpret_cast<ssd::UnitRecord *>(ws);
    P.seq_count = reinterpret_cast<uint32_t *>(ws + ssd::ws_rec_bytes(B, K));
    P.seq_reject =
        reinterpret_cast<uint32_t *>(ws + ssd::ws_rec_bytes(B, K) + ssd::ws_count_bytes(B));
    P.dev_status = dev_status;
    uint32_t *sched = reinterpret_cast<uint32_t *>(ws + ssd::ws_rec_bytes(B, K) + 2 * ssd::ws_count_bytes(B));
    P.unit_counter = sched;
    P.exit_counter = sched + 1;
    P.unit_ends = reinterpret_cast<unsigned long long *>(sched + 2);
    P.perm_mul = coprime_stride(B);
    if (sliced) {
        P.S = ssd::slice_count(units, V, elem);
        P.nblk = ssd::slice_blocks(V, elem);
        P.key_stride = key_stride;
        int ko = 0;
        for (int k = 0; k <= K; ++k) {
            P.koff[k] = ko;
            const int f = cache ? F_host[k] : 0;
            ko += f > 1 ? f : 1;
        }
        P.slice_ctr = reinterpret_cast<uint32_t *>(ws + SW.counters);
        P.ustate = reinterpret_cast<ssd::SliceUnitState *>(ws + SW.ustate);
        P.sstat = reinterpret_cast<float4 *>(ws + SW.sstat);
        P.skeys = reinterpret_cast<unsigned long long *>(ws + SW.skeys);
        P.garr = reinterpret_cast<float *>(ws + SW.garr);
        P.queue = reinterpret_cast<unsigned long long *>(ws + SW.queue);
        P.pcand = reinterpret_cast<float *>(ws + SW.pcand);
        P.cmax = reinterpret_cast<float *>(ws + SW.cmax);
        t_last_kernel = "slice";
        return ssd::slice_launch(dtype, P, dv->sm_count, ssd::slice_dyn_bytes(), stream);
    }
    if (streaming) {
        if (sig_F) {
            P.sig_on = 1;
            for (int k = 0; k < K; ++k) P.sig_F[k] = sig_F[k];
            P.sig_C = sig_C;
            P.desc_out = desc_out;
        }
        const int grid = std::min(dv->sm_count, units);
        P.wide = wide ? 1 : 0;
        t_last_kernel = wide ? "stream-wide" : "stream";
        return ssd::stream_launch(dtype, P, grid, sdyn, stream);
    }
    if (sig_F) {
        // the cluster kernel takes descriptors: find them first (one more read of
        // the draft rows), into desc_out
        ssd::ReshapeParams R = {};
        Geometry rg;
        st = choose_geometry(V, elem, 1, B * drf_rows, *dv, dv->max_dyn[dtype == SSD_F32 ? 2 : 3], &rg);
        if (st != SSD_OK) return st;
        R.drf = drf;
        R.rows = B * drf_rows;
        R.V = V;
        R.CL = rg.CL;
        R.slice = rg.slice;
        R.row_buf_bytes = rg.row_buf_bytes;
        R.C = sig_C;
        R.desc = desc_out;
        R.dev_status = dev_status;
        R.seq_rows = drf_rows;
        R.K = K;
        for (int k = 0; k < K; ++k) R.Fk[k] = sig_F[k];
        st = ssd::reshape_launch(dtype, R, R.rows * rg.CL, rg.CL, rg.dyn, stream);
        if (st != SSD_OK) return st;
        P.reshape = desc_out;
    }
    const int grid = units * g.CL;
    t_last_kernel = sig_F ? "reshape+cluster" : "cluster";
    return ssd::unit_launch(dtype, P, grid, g.CL, g.dyn, stream);
}

}  // namespace

extern "C" {

const char *ssd_strerror(int status) {
    switch (status) {
        case SSD_OK: return "SSD_OK";
        case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: invalid argument";
        case SSD_ERR_DTYPE: return "SSD_ERR_DTYPE: unsupported logit dtype";
        case SSD_ERR_CUDA: return "SSD_ERR_CUDA: CUDA runtime error";
        case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: size or device not supported";
        default: return "unknown ssd status";
    }
}

const char *ssd_version(void) { return "libssd 0.2 (sm_103a)"; }

const char *ssd_last_kernel(void) { return t_last_kernel; }

int ssd_set_dispatch(int policy) {
    if (policy != SSD_DISPATCH_AUTO && policy != SSD_DISPATCH_STREAM && policy != SSD_DISPATCH_CLUSTER &&
        policy != SSD_DISPATCH_SLICE && policy != SSD_DISPATCH_WIDE)
        return -1;
    return g_dispatch.exchange(policy);
}

size_t ssd_workspace_size(int B, int K) {
    if (B < 1 || K < 1 || K > SSD_MAX_K) return 0;
    return ssd::ws_total_bytes(B, K);
}

size_t ssd_workspace_size_v(int B, int K, int V, int dtype, int budget) {
    if (B < 1 || K < 1 || K > SSD_MAX_K || V < 2 || budget < 0) return 0;
    if (dtype != SSD_F32 && dtype != SSD_BF16) return 0;
    const int elem = dtype == SSD_F32 ? 4 : 2;
    // every position keeps max(F_k, 1) keys per slice, and sum F_k <= budget
    const size_t sl = ssd::slice_ws_layout(B, K, V, elem, budget + K + 1).total;
    const size_t base = ssd::ws_total_bytes(B, K);
    return sl > base ? sl : base;
}

int ssd_verify(const void *tgt, const void *drf, int dtype, int B, int K, int V, int drf_rows,
               const int32_t *tokens, const float *uniforms, const float *temperature,
               const ssd_reshape_desc *reshape, int32_t *accept_len, int32_t *bonus,
               float *p_tok, float *q_tok, void *workspace, size_t workspace_bytes,
               int32_t *dev_status, void *stream) {
    return run_units(ssd::kModeVerify, tgt, drf, dtype, B, K, V, drf_rows, tokens, uniforms,
                     temperature, reshape, nullptr, 0, accept_len, bonus, p_tok, q_tok, nullptr,
                     nullptr, nullptr, workspace, workspace_bytes, dev_status, stream);
}

int ssd_build_cache(const void *tgt, const void *drf, int dtype, int B, int K, int V,
                    int drf_rows, const int32_t *tokens, const float *temperature,
                    const ssd_reshape_desc *reshape, const int32_t *F_host, int budget,
                    int32_t *cache_tok, void *workspace, size_t workspace_bytes,
                    int32_t *dev_status, void *stream) {
    return run_units(ssd::kModeCache, tgt, drf, dtype, B, K, V, drf_rows, tokens, nullptr,
                     temperature, reshape, F_host, budget, nullptr, nullptr, nullptr, nullptr,
                     cache_tok, nullptr, nullptr, workspace, workspace_bytes, dev_status, stream);
}

int ssd_round(const void *tgt, const void *drf, int dtype, int B, int K, int V, int drf_rows,
              const int32_t *tokens, const float *uniforms, const float *temperature,
              const ssd_reshape_desc *reshape, const int32_t *F_host, int budget,
              int32_t *accept_len, int32_t *bonus, float *p_tok, float *q_tok,
              int32_t *cache_tok, uint8_t *hit, int32_t *slot, void *workspace,
              size_t workspace_bytes, int32_t *dev_status, void *stream) {
    return run_units(ssd::kModeVerify | ssd::kModeCache | ssd::kModeLookup, tgt, drf, dtype, B, K,
                     V, drf_rows, tokens, uniforms, temperature, reshape, F_host, budget,
                     accept_len, bonus, p_tok, q_tok, cache_tok, hit, slot, workspace,
                     workspace_bytes, dev_status, stream);
}

int ssd_verify_ld(const void *tgt, const void *drf, int dtype, int B, int K, int V, int ld,
                  int drf_rows, const int32_t *tokens, const float *uniforms, const float *temperature,
                  const ssd_reshape_desc *reshape, int32_t *accept_len, int32_t *bonus, float *p_tok,
                  float *q_tok, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                  void *stream) {
    return run_units(ssd::kModeVerify, tgt, drf, dtype, B, K, V, drf_rows, tokens, uniforms,
                     temperature, reshape, nullptr, 0, accept_len, bonus, p_tok, q_tok, nullptr,
                     nullptr, nullptr, workspace, workspace_bytes, dev_status, stream, nullptr, 1.f,
                     nullptr, ld);
}

int ssd_round_ld(const void *tgt, const void *drf, int dtype, int B, int K, int V, int ld,
                 int drf_rows, const int32_t *tokens, const float *uniforms, const float *temperature,
                 const ssd_reshape_desc *reshape, const int32_t *F_host, int budget,
                 int32_t *accept_len, int32_t *bonus, float *p_tok, float *q_tok, int32_t *cache_tok,
                 uint8_t *hit, int32_t *slot, void *workspace, size_t workspace_bytes,
                 int32_t *dev_status, void *stream) {
    return run_units(ssd::kModeVerify | ssd::kModeCache | ssd::kModeLookup, tgt, drf, dtype, B, K,
                     V, drf_rows, tokens, uniforms, temperature, reshape, F_host, budget,
                     accept_len, bonus, p_tok, q_tok, cache_tok, hit, slot, workspace,
                     workspace_bytes, dev_status, stream, nullptr, 1.f, nullptr, ld);
}

int ssd_verify_sigma(const void *tgt, const void *drf, int dtype, int B, int K, int V, int drf_rows,
                     const int32_t *tokens, const float *uniforms, const float *temperature,
                     const int32_t *sigma_F_host, float sigma_C, ssd_reshape_desc *desc_out,
                     int32_t *accept_len, int32_t *bonus, float *p_tok, float *q_tok,
                     void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream) {
    if (!sigma_F_host) return SSD_ERR_INVALID_ARG;
    return run_units(ssd::kModeVerify, tgt, drf, dtype, B, K, V, drf_rows, tokens, uniforms,
                     temperature, nullptr, nullptr, 0, accept_len, bonus, p_tok, q_tok, nullptr,
                     nullptr, nullptr, workspace, workspace_bytes, dev_status, stream, sigma_F_host,
                     sigma_C, desc_out);
}

int ssd_round_sigma(const void *tgt, const void *drf, int dtype, int B, int K, int V, int drf_rows,
                    const int32_t *tokens, const float *uniforms, const float *temperature,
                    const int32_t *sigma_F_host, float sigma_C, ssd_reshape_desc *desc_out,
                    const int32_t *F_host, int budget, int32_t *accept_len, int32_t *bonus,
                    float *p_tok, float *q_tok, int32_t *cache_tok, uint8_t *hit, int32_t *slot,
                    void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream) {
    if (!sigma_F_host) return SSD_ERR_INVALID_ARG;
    return run_units(ssd::kModeVerify | ssd::kModeCache | ssd::kModeLookup, tgt, drf, dtype, B, K,
                     V, drf_rows, tokens, uniforms, temperature, nullptr, F_host, budget, accept_len,
                     bonus, p_tok, q_tok, cache_tok, hit, slot, workspace, workspace_bytes,
                     dev_status, stream, sigma_F_host, sigma_C, desc_out);
}

int ssd_cache_lookup(const int32_t *cache_tok, int B, int K, int budget, const int32_t *F_host,
                     const int32_t *accept_len, const int32_t *bonus, uint8_t *hit,
                     int32_t *slot, void *stream) {
    if (B < 1 || K < 1 || K > SSD_MAX_K) return SSD_ERR_INVALID_ARG;
    if (!accept_len || !bonus || !hit || !slot) return SSD_ERR_INVALID_ARG;
    ssd::LookupParams P = {};
    const int st = check_fanout(F_host, K, INT_MAX, budget, P.off);
    if (st != SSD_OK) return st;
    if (P.off[K + 1] > 0 && !cache_tok) return SSD_ERR_INVALID_ARG;
    P.cache_tok = cache_tok;
    P.B = B;
    P.K = K;
    P.budget = budget;
    P.accept_len = accept_len;
    P.bonus = bonus;
    P.hit = hit;
    P.slot = slot;
    return ssd::lookup_launch(P, stream);
}

int ssd_reshape_draft(const void *drf, int dtype, int rows, int V, const float *temperature_rows,
                      int F, float C, ssd_reshape_desc *desc, float *q_out, int32_t *dev_status,
                      void *stream) {
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_DTYPE;
    if (!drf || !desc || rows < 1 || V < 2) return SSD_ERR_INVALID_ARG;
    if (F < 0 || F > SSD_MAX_F || F > V) return SSD_ERR_INVALID_ARG;
    if (!(C >= 0.f && C <= 1.f)) return SSD_ERR_INVALID_ARG;
    if (C == 0.f && F >= V) return SSD_ERR_INVALID_ARG;
    if (q_out && !temperature_rows) return SSD_ERR_INVALID_ARG;
    if (V > (dtype == SSD_F32 ? SSD_MAX_V_F32 : SSD_MAX_V_BF16)) return SSD_ERR_UNSUPPORTED;
    DeviceInfo *dv = nullptr;
    int st = device_info(&dv);
    if (st != SSD_OK) return st;
    const int elem = dtype == SSD_F32 ? 4 : 2;
    Geometry g;
    st = choose_geometry(V, elem, 1, rows, *dv, dv->max_dyn[dtype == SSD_F32 ? 2 : 3], &g);
    if (st != SSD_OK) return st;
    ssd::ReshapeParams P = {};
    P.drf = drf;
    P.rows = rows;
    P.V = V;
    P.CL = g.CL;
    P.slice = g.slice;
    P.row_buf_bytes = g.row_buf_bytes;
    P.tau = temperature_rows;
    P.F = F;
    P.C = C;
    P.desc = desc;
    P.q_out = q_out;
    P.dev_status = dev_status;
    const int grid = rows * g.CL;
    return ssd::reshape_launch(dtype, P, grid, g.CL, g.dyn, stream);
}

int ssd_draft_cache(const void *drf, int dtype, int B, int K, int V, const int32_t *tokens,
                    const int32_t *F_host, int budget, float C, int32_t *cache_tok,
                    ssd_reshape_desc *desc, int32_t *dev_status, void *stream) {
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_DTYPE;
    if (!drf || B < 1 || K < 1 || K > SSD_MAX_K || V < 2) return SSD_ERR_INVALID_ARG;
    if (!cache_tok && !desc) return SSD_ERR_INVALID_ARG;
    if (static_cast<int64_t>(B) * (K + 1) > INT_MAX / 16) return SSD_ERR_UNSUPPORTED;
    ssd::ReshapeParams P = {};
    int st = check_fanout(F_host, K, V, budget, P.off);
    if (st != SSD_OK) return st;
    if (desc) {
        if (!(C >= 0.f && C <= 1.f)) return SSD_ERR_INVALID_ARG;
        for (int k = 0; k < K; ++k)
            if (C == 0.f && F_host[k] >= V) return SSD_ERR_INVALID_ARG;
    }
    if (V > (dtype == SSD_F32 ? SSD_MAX_V_F32 : SSD_MAX_V_BF16)) return SSD_ERR_UNSUPPORTED;
    DeviceInfo *dv = nullptr;
    st = device_info(&dv);
    if (st != SSD_OK) return st;
    const int elem = dtype == SSD_F32 ? 4 : 2;
    const int rows = B * (K + 1);
    Geometry g;
    st = choose_geometry(V, elem, 1, rows, *dv, dv->max_dyn[dtype == SSD_F32 ? 2 : 3], &g);
    if (st != SSD_OK) return st;
    P.drf = drf;
    P.rows = rows;
    P.V = V;
    P.CL = g.CL;
    P.slice = g.slice;
    P.row_buf_bytes = g.row_buf_bytes;
    P.C = C;
    P.desc = desc;
    P.dev_status = dev_status;
    P.seq_rows = K + 1;
    P.K = K;
    for (int k = 0; k <= K; ++k) P.Fk[k] = F_host[k];
    P.tokens = tokens;
    P.cache_tok = cache_tok;
    P.budget = budget;
    return ssd::reshape_launch(dtype, P, rows * g.CL, g.CL, g.dyn, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Workspace-free round.  Some callers cannot allocate device memory on their
// own: an inference-server plugin whose host framework owns every device
// buffer and forbids allocation while it enqueues work (cudaMalloc can block
// the device and can fail under memory pressure mid-serving), or a runtime
// that fixes its memory footprint at start-up.  For them ssd_round_noalloc
// keeps the per-round scratch (unit records, per-sequence counters) in the
// array below, which every GPU that loads the library holds until the
// process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB per device
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocSlot {
    bool ready = false;
    void *ptr = nullptr;
};
NoAllocSlot g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of this device's scratch array.  In host code the array's
// name stands for a host-side shadow, not a device address, so the address is
// looked up once per device, with that device current.
int noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocSlot &slot = g_noalloc[dev];
    if (!slot.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return SSD_ERR_CUDA;
        }
        slot.ptr = p;
        slot.ready = true;
    }
    *out = slot.ptr;
    return SSD_OK;
}

}  // namespace

extern "C" {

size_t ssd_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

int ssd_round_noalloc(const void *tgt, const void *drf, int dtype, int B, int K, int V,
                      int drf_rows, const int32_t *tokens, const float *uniforms,
                      const float *temperature, const ssd_reshape_desc *reshape,
                      const int32_t *F_host, int budget, int32_t *accept_len, int32_t *bonus,
                      float *p_tok, float *q_tok, int32_t *cache_tok, uint8_t *hit,
                      int32_t *slot, int32_t *dev_status, void *stream) {
    if (B < 1 || K < 1 || K > SSD_MAX_K) return SSD_ERR_INVALID_ARG;
    const size_t need = ssd::ws_total_bytes(B, K);
    if (need > kNoAllocScratchBytes) return SSD_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != SSD_OK) return st;
    // The array keeps the previous call's contents.  A round that completes leaves
    // its per-sequence and scheduler counters at zero (the last unit of a sequence
    // and the grid's last tail warp reset them), but one that gave up early (a
    // device timeout) or a different batch shape would not: clearing them here
    // makes every call start from zero.  This clear sits between back-to-back
    // calls, so these rounds do not overlap one another through programmatic
    // dependent launch.
    unsigned char *base = static_cast<unsigned char *>(scratch);
    const size_t rec = ssd::ws_rec_bytes(B, K);
    if (cudaMemsetAsync(base + rec, 0, need - rec, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SSD_ERR_CUDA;
    }
    return ssd_round(tgt, drf, dtype, B, K, V, drf_rows, tokens, uniforms, temperature, reshape,
                     F_host, budget, accept_len, bonus, p_tok, q_tok, cache_tok, hit, slot, scratch,
                     need, dev_status, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Rounds from host buffers: the staging layout in device memory (every part on
// a 256-byte boundary) and the copies around the round.
namespace {

struct HostStaging {
    size_t tgt, drf, tok, uni, tau, acc, bon, cache, hit, slot, total;
};

HostStaging host_staging_layout(int dtype, int B, int K, int V, int budget) {
    const auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t s = dtype == SSD_F32 ? 4 : 2;
    const size_t b = static_cast<size_t>(B);
    HostStaging L;
    size_t o = 0;
    L.tgt = o;
    o = up(o + b * (K + 1) * V * s);
    L.drf = o;
    o = up(o + b * K * V * s);
    L.tok = o;
    o = up(o + b * K * 4);
    L.uni = o;
    o = up(o + b * (K + 1) * 4);
    L.tau = o;
    o = up(o + b * 4);
    L.acc = o;
    o = up(o + b * 4);
    L.bon = o;
    o = up(o + b * 4);
    L.cache = o;
    o = up(o + b * static_cast<size_t>(budget) * 4);
    L.hit = o;
    o = up(o + b);
    L.slot = o;
    o = up(o + b * 4);
    L.total = o;
    return L;
}

bool host_staging_args_ok(int dtype, int B, int K, int V, int budget) {
    return B >= 1 && K >= 1 && K <= SSD_MAX_K && V >= 2 && budget >= 0 &&
           (dtype == SSD_F32 || dtype == SSD_BF16);
}

// Per device, for ssd_round_host: one stream for the host-to-device copies, so that
// a chunk's round overlaps the copies of the next chunk, and the events that order
// the copies and the rounds (created on first use, kept until the process exits).
// A call holds its device's lock while it enqueues: an event is re-recorded only by
// the next call, and a stream wait binds to the record made before it, so reuse
// across calls is safe.
constexpr int kHostChunks = 4;

struct HostRoundRes {
    std::mutex mu;
    cudaStream_t copy = nullptr;
    cudaEvent_t ev[kHostChunks + 1] = {};
    bool ready = false;
};

std::mutex g_copy_mu;
HostRoundRes g_host_res[kMaxDevices];

int host_round_res(HostRoundRes **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_copy_mu);
    HostRoundRes &r = g_host_res[dev];
    if (!r.ready) {
        if (!r.copy && cudaStreamCreateWithFlags(&r.copy, cudaStreamNonBlocking) != cudaSuccess) {
            r.copy = nullptr;
            cudaGetLastError();
            return SSD_ERR_CUDA;
        }
        for (int i = 0; i <= kHostChunks; ++i) {
            if (!r.ev[i] && cudaEventCreateWithFlags(&r.ev[i], cudaEventDisableTiming) != cudaSuccess) {
                r.ev[i] = nullptr;
                cudaGetLastError();
                return SSD_ERR_CUDA;
            }
        }
        r.ready = true;
    }
    *out = &r;
    return SSD_OK;
}

// The fan-out checks of the round, taken before any copy is enqueued.
bool host_fanout_ok(const int32_t *F_host, int K, int V, int budget) {
    int64_t sum = 0;
    for (int k = 0; k <= K; ++k) {
        if (F_host[k] < 0 || F_host[k] > V || F_host[k] > SSD_MAX_F) return false;
        sum += F_host[k];
    }
    return sum <= budget;
}

}  // namespace

extern "C" {

size_t ssd_host_staging_size(int dtype, int B, int K, int V, int budget) {
    if (!host_staging_args_ok(dtype, B, K, V, budget)) return 0;
    return host_staging_layout(dtype, B, K, V, budget).total;
}

int ssd_round_host(const void *tgt, const void *drf, int dtype, int B, int K, int V,
                   const int32_t *tokens, const float *uniforms, const float *temperature,
                   const int32_t *F_host, int budget, int32_t *accept_len, int32_t *bonus,
                   int32_t *cache_tok, uint8_t *hit, int32_t *slot, void *staging,
                   size_t staging_bytes, void *workspace, size_t workspace_bytes,
                   int32_t *dev_status, size_t *h2d_bytes, void *stream) {
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_DTYPE;
    if (!host_staging_args_ok(dtype, B, K, V, budget)) return SSD_ERR_INVALID_ARG;
    if (!tgt || !drf || !tokens || !uniforms || !temperature || !F_host || !accept_len || !bonus ||
        !cache_tok || !hit || !slot || !staging)
        return SSD_ERR_INVALID_ARG;
    if (!host_fanout_ok(F_host, K, V, budget)) return SSD_ERR_INVALID_ARG;
    const HostStaging L = host_staging_layout(dtype, B, K, V, budget);
    if (staging_bytes < L.total) return SSD_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    HostRoundRes *res = nullptr;
    const int rst = host_round_res(&res);
    if (rst != SSD_OK) return rst;
    std::lock_guard<std::mutex> enqueue_lock(res->mu);
    cudaStream_t cs = res->copy;  // the copies run here, each chunk's round on `stream`
    cudaEvent_t *ev = res->ev;
    // Consecutive sequences in up to 4 chunks of at least 64: the round on chunk c
    // runs while the next chunk is copied (sequences are independent).
    const int nchunk = std::max(1, std::min(kHostChunks, B / 64));
    unsigned char *base = static_cast<unsigned char *>(staging);
    size_t moved = 0;
    bool ok = true;
    const auto h2d = [&](size_t off, const void *src, size_t n) {
        if (!ok || n == 0) return;
        moved += n;
        ok = cudaMemcpyAsync(base + off, src, n, cudaMemcpyHostToDevice, cs) == cudaSuccess;
    };
    const auto d2h = [&](void *dst, size_t off, size_t n) {
        if (!ok || n == 0) return;
        ok = cudaMemcpyAsync(dst, base + off, n, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    };
    const size_t row = static_cast<size_t>(V) * (dtype == SSD_F32 ? 4 : 2);
    const size_t seq_t = static_cast<size_t>(K + 1) * row;
    const size_t seq_d = static_cast<size_t>(K) * row;
    // the copies start after the work already on `stream` (an earlier round reading staging)
    ok = cudaEventRecord(ev[0], st) == cudaSuccess && cudaStreamWaitEvent(cs, ev[0], 0) == cudaSuccess;
    h2d(L.tok, tokens, static_cast<size_t>(B) * K * 4);
    h2d(L.uni, uniforms, static_cast<size_t>(B) * (K + 1) * 4);
    h2d(L.tau, temperature, static_cast<size_t>(B) * 4);
    const auto sampled = [&](int i) { return temperature[i] > 0.f && temperature[i] < INFINITY; };
    for (int c = 0; c < nchunk; ++c) {
        const int c0 = static_cast<int>(static_cast<int64_t>(B) * c / nchunk);
        const int c1 = static_cast<int>(static_cast<int64_t>(B) * (c + 1) / nchunk);
        h2d(L.tgt + c0 * seq_t, static_cast<const unsigned char *>(tgt) + c0 * seq_t,
            static_cast<size_t>(c1 - c0) * seq_t);
        // Draft rows of the sampled sequences only (a run of consecutive ones in one
        // copy): a greedy or invalid sequence's draft logits are never read.
        for (int b = c0; b < c1;) {
            if (!sampled(b)) {
                ++b;
                continue;
            }
            int e = b + 1;
            while (e < c1 && sampled(e)) ++e;
            h2d(L.drf + static_cast<size_t>(b) * seq_d,
                static_cast<const unsigned char *>(drf) + static_cast<size_t>(b) * seq_d,
                static_cast<size_t>(e - b) * seq_d);
            b = e;
        }
        if (ok) ok = cudaEventRecord(ev[c + 1], cs) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        return SSD_ERR_CUDA;
    }
    for (int c = 0; c < nchunk; ++c) {
        const int c0 = static_cast<int>(static_cast<int64_t>(B) * c / nchunk);
        const int c1 = static_cast<int>(static_cast<int64_t>(B) * (c + 1) / nchunk);
        const int nb = c1 - c0;
        if (cudaStreamWaitEvent(st, ev[c + 1], 0) != cudaSuccess) {
            cudaGetLastError();
            return SSD_ERR_CUDA;
        }
        const int rc = ssd_round(
            base + L.tgt + c0 * seq_t, base + L.drf + c0 * seq_d, dtype, nb, K, V, K,
            reinterpret_cast<const int32_t *>(base + L.tok) + static_cast<size_t>(c0) * K,
            reinterpret_cast<const float *>(base + L.uni) + static_cast<size_t>(c0) * (K + 1),
            reinterpret_cast<const float *>(base + L.tau) + c0, nullptr, F_host, budget,
            reinterpret_cast<int32_t *>(base + L.acc) + c0, reinterpret_cast<int32_t *>(base + L.bon) + c0,
            nullptr, nullptr, reinterpret_cast<int32_t *>(base + L.cache) + static_cast<size_t>(c0) * budget,
            reinterpret_cast<uint8_t *>(base + L.hit) + c0, reinterpret_cast<int32_t *>(base + L.slot) + c0,
            workspace, workspace_bytes, dev_status, stream);
        if (rc != SSD_OK) return rc;
        d2h(accept_len + c0, L.acc + static_cast<size_t>(c0) * 4, static_cast<size_t>(nb) * 4);
        d2h(bonus + c0, L.bon + static_cast<size_t>(c0) * 4, static_cast<size_t>(nb) * 4);
        d2h(cache_tok + static_cast<size_t>(c0) * budget, L.cache + static_cast<size_t>(c0) * budget * 4,
            static_cast<size_t>(nb) * budget * 4);
        d2h(hit + c0, L.hit + static_cast<size_t>(c0), static_cast<size_t>(nb));
        d2h(slot + c0, L.slot + static_cast<size_t>(c0) * 4, static_cast<size_t>(nb) * 4);
    }
    if (!ok) {
        cudaGetLastError();
        return SSD_ERR_CUDA;
    }
    if (h2d_bytes) *h2d_bytes = moved;
    return SSD_OK;
}

}  // extern "C"
