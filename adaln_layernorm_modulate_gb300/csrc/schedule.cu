// Host-side scheduling half of the AdaptiveLoad technical summary, section 2.A ("adaptive
// load balancing with a dual constraint"): the bucket size for a real (fitted) exponent, the
// Shape-Benchmarking fit of the step-time model t = a + b * B * S^p, and the compute-load
// imbalance a bucketing rule leaves. Plain host C++, no device work; see include/adaln.h.
#include "adaln.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

namespace {

bool finite_positive(double v) { return std::isfinite(v) && v > 0.0; }

// For a fixed exponent p the model t = a + b * u, u = B * S^p, is linear: the exact
// least-squares (a, b) and the residual sum of squares.
struct LinearFit {
    double a, b, rss;
};

LinearFit fit_at(const int64_t* B, const int64_t* S, const double* t, int64_t n, double p) {
    std::vector<double> u((size_t)n);
    double su = 0.0, st = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        u[(size_t)i] = (double)B[i] * std::pow((double)S[i], p);
        su += u[(size_t)i];
        st += t[i];
    }
    const double mu = su / (double)n, mt = st / (double)n;
    double suu = 0.0, sut = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double du = u[(size_t)i] - mu;
        suu += du * du;
        sut += du * (t[i] - mt);
    }
    LinearFit f{mt, 0.0, 0.0};
    if (suu > 0.0) {
        f.b = sut / suu;
        f.a = mt - f.b * mu;
    }
    for (int64_t i = 0; i < n; ++i) {
        const double r = t[i] - f.a - f.b * u[(size_t)i];
        f.rss += r * r;
    }
    return f;
}

}  // namespace

extern "C" {

int64_t adaln_bucket_batch_real(int64_t S, int64_t M_mem, int64_t M_comp, double p) {
    if (S <= 0 || M_mem <= 0 || M_comp <= 0 || !finite_positive(p)) return -(int64_t)ADALN_ERR_INVALID_ARG;
    if (p >= 1.0 && p <= 64.0 && p == std::floor(p)) return adaln_bucket_batch(S, M_mem, M_comp, (int32_t)p);
    const int64_t by_memory = M_mem / S;
    const double q = (double)M_comp / std::pow((double)S, p);
    const int64_t by_compute = q >= 9.2e18 ? INT64_MAX : (int64_t)std::floor(q);
    const int64_t b = std::min(by_memory, by_compute);
    return b > 1 ? b : 1;
}

int adaln_fit_step_cost(const int64_t* B, const int64_t* S, const double* t, int64_t n,
                        double p_lo, double p_hi, double t_budget, double* out) {
    if (!B || !S || !t || !out || n < 3) return ADALN_ERR_INVALID_ARG;
    if (!finite_positive(p_lo) || !std::isfinite(p_hi) || !(p_lo < p_hi) || !std::isfinite(t_budget))
        return ADALN_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n; ++i)
        if (B[i] <= 0 || S[i] <= 0 || !std::isfinite(t[i])) return ADALN_ERR_INVALID_ARG;

    // Bracket the best exponent on a grid, then refine by golden-section search.
    constexpr int kGrid = 200;
    int best = 0;
    double best_rss = INFINITY;
    for (int j = 0; j <= kGrid; ++j) {
        const double p = p_lo + (p_hi - p_lo) * (double)j / kGrid;
        const double r = fit_at(B, S, t, n, p).rss;
        if (r < best_rss) {
            best_rss = r;
            best = j;
        }
    }
    double lo = p_lo + (p_hi - p_lo) * (double)std::max(best - 1, 0) / kGrid;
    double hi = p_lo + (p_hi - p_lo) * (double)std::min(best + 1, kGrid) / kGrid;
    const double g = 0.5 * (std::sqrt(5.0) - 1.0);
    double x1 = hi - g * (hi - lo), x2 = lo + g * (hi - lo);
    double f1 = fit_at(B, S, t, n, x1).rss, f2 = fit_at(B, S, t, n, x2).rss;
    for (int it = 0; it < 200 && hi - lo > 1e-12; ++it) {
        if (f1 <= f2) {
            hi = x2;
            x2 = x1;
            f2 = f1;
            x1 = hi - g * (hi - lo);
            f1 = fit_at(B, S, t, n, x1).rss;
        } else {
            lo = x1;
            x1 = x2;
            f1 = f2;
            x2 = lo + g * (hi - lo);
            f2 = fit_at(B, S, t, n, x2).rss;
        }
    }
    double p = 0.5 * (lo + hi);
    LinearFit f = fit_at(B, S, t, n, p);
    // Keep the grid point if the refinement ended on a worse value (a flat residual).
    const double p_grid = p_lo + (p_hi - p_lo) * (double)best / kGrid;
    const LinearFit fg = fit_at(B, S, t, n, p_grid);
    if (fg.rss < f.rss) {
        f = fg;
        p = p_grid;
    }
    out[0] = f.a;
    out[1] = f.b;
    out[2] = p;
    out[3] = std::sqrt(f.rss / (double)n);
    out[4] = (f.b > 0.0 && t_budget > f.a) ? std::floor((t_budget - f.a) / f.b) : 0.0;
    return ADALN_OK;
}

int adaln_bucket_load_cv(const int64_t* lengths, int64_t n, const int64_t* buckets,
                         int32_t nbuckets, int64_t M_mem, int64_t M_comp, double p, int32_t rule,
                         double* out) {
    if (!lengths || !buckets || !out || n < 1 || nbuckets < 1) return ADALN_ERR_INVALID_ARG;
    if (M_mem <= 0 || M_comp <= 0 || !finite_positive(p) || (rule != 0 && rule != 1))
        return ADALN_ERR_INVALID_ARG;
    for (int32_t k = 0; k < nbuckets; ++k)
        if (buckets[k] <= 0 || (k > 0 && buckets[k] <= buckets[k - 1])) return ADALN_ERR_INVALID_ARG;
    std::vector<int64_t> count((size_t)nbuckets, 0);
    for (int64_t i = 0; i < n; ++i) {
        const int64_t L = lengths[i];
        const int64_t* it = std::lower_bound(buckets, buckets + nbuckets, L);
        if (L <= 0 || it == buckets + nbuckets) return ADALN_ERR_INVALID_ARG;
        ++count[(size_t)(it - buckets)];
    }
    // Batches per bucket: `full` of its batch size, plus one of the remainder.
    struct Group {
        double cost;
        int64_t batches;
    };
    std::vector<Group> groups;
    double total = 0.0;
    int64_t nb = 0;
    for (int32_t k = 0; k < nbuckets; ++k) {
        const int64_t c = count[(size_t)k];
        if (c == 0) continue;
        const int64_t S = buckets[k];
        const int64_t bs = rule == 0 ? std::max<int64_t>(1, M_mem / S) : adaln_bucket_batch_real(S, M_mem, M_comp, p);
        const double unit = std::pow((double)S, p);
        const int64_t full = c / bs, rem = c % bs;
        if (full > 0) groups.push_back({(double)bs * unit, full});
        if (rem > 0) groups.push_back({(double)rem * unit, 1});
    }
    for (const Group& g : groups) {
        total += g.cost * (double)g.batches;
        nb += g.batches;
    }
    const double mean = total / (double)nb;
    double ss = 0.0;
    for (const Group& g : groups) ss += (double)g.batches * (g.cost - mean) * (g.cost - mean);
    out[0] = mean > 0.0 ? std::sqrt(ss / (double)nb) / mean : 0.0;
    out[1] = (double)nb;
    out[2] = mean;
    return ADALN_OK;
}

}  // extern "C"
