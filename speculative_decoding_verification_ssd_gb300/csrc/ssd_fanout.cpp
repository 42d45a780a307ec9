// ssd_fanout.cpp -- Saguaro's geometric fan-out (host only).
//
// [SSD] "Speculative Speculative Decoding" notes (papernotes.org), "关键设计"
// item 1: under a power-law cache-miss model the budget-optimal fan-out is
//   F_k = F_0 a_p^{k/(1+r)}                          for k < K,
//   F_K = F_0 a_p^{K/(1+r)} (1 - a_p)^{-1/(1+r)}     (the all-accepted outcome),
// subject to sum_k F_k <= budget.  F_0 takes the whole budget; the real values
// are made integers by the largest-remainder method and clamped to V.
#include <cmath>
#include <cstdint>
#include <vector>

#include "../../include/ssd.h"

extern "C" int ssd_fanout(int K, int budget, double a_p, double r, int V, int32_t *F_host,
                          int32_t *off_host) {
    if (K < 1 || K > SSD_MAX_K || budget < 0 || V < 1 || !F_host || !off_host)
        return SSD_ERR_INVALID_ARG;
    if (!(a_p > 0.0 && a_p < 1.0) || !(r > -1.0) || !std::isfinite(r)) return SSD_ERR_INVALID_ARG;
    const double e = 1.0 / (1.0 + r);
    std::vector<double> shape(K + 1);
    double total = 0.0;
    for (int k = 0; k <= K; ++k) {
        shape[k] = std::pow(a_p, k * e);
        if (k == K) shape[k] *= std::pow(1.0 - a_p, -e);
        total += shape[k];
    }
    // Largest remainder: floors first, then one extra slot to each of the
    // largest fractional parts (ties to the smaller k) until the budget is met.
    std::vector<double> real(K + 1), frac(K + 1);
    std::vector<int> F(K + 1);
    long used = 0;
    for (int k = 0; k <= K; ++k) {
        real[k] = budget * shape[k] / total;
        const double fl = std::floor(real[k]);
        F[k] = static_cast<int>(fl);
        frac[k] = real[k] - fl;
        used += F[k];
    }
    std::vector<bool> taken(K + 1, false);
    for (long left = budget - used; left > 0; --left) {
        int pick = -1;
        for (int k = 0; k <= K; ++k)
            if (!taken[k] && (pick < 0 || frac[k] > frac[pick])) pick = k;
        if (pick < 0) break;
        taken[pick] = true;
        ++F[pick];
    }
    off_host[0] = 0;
    for (int k = 0; k <= K; ++k) {
        F_host[k] = F[k] > V ? V : F[k];
        off_host[k + 1] = off_host[k] + F_host[k];
    }
    return SSD_OK;
}

// The uniform fan-out the geometric shape is compared against in [SSD] item 1:
// an equal share of the budget for every accepted length, the remainder going
// one slot each to the lowest k, each share clamped to V.
extern "C" int ssd_fanout_uniform(int K, int budget, int V, int32_t *F_host, int32_t *off_host) {
    if (K < 1 || K > SSD_MAX_K || budget < 0 || V < 1 || !F_host || !off_host)
        return SSD_ERR_INVALID_ARG;
    const int share = budget / (K + 1);
    const int extra = budget % (K + 1);
    off_host[0] = 0;
    for (int k = 0; k <= K; ++k) {
        const int f = share + (k < extra ? 1 : 0);
        F_host[k] = f > V ? V : f;
        off_host[k + 1] = off_host[k] + F_host[k];
    }
    return SSD_OK;
}
