// TEST INFRASTRUCTURE ONLY -- not part of the product path.
//
// A plain, slow, obviously-correct CPU statement of the fused AdaLN
// (LayerNorm-Modulate) operator, used to check the CUDA kernels. Only the test
// suite, the package smoke check and the benchmark's CPU-baseline leg may load
// it. It shares no code, header or constant with the CUDA library.
//
// Source: "AdaptiveLoad: Towards Efficient Video Diffusion Transformer
// Training", technical summary, section 2.B "Fused LayerNorm-Modulate CUDA
// kernels" (forward-pass and backward-pass bullets). The pages name the operator
// (normalisation followed by modulation; statistics = mean and variance over the
// feature dimension D; modulation gradients reduced along the sequence) but print
// no formula. This file takes the standard DiT "modulate" reading:
//
//   mu    = (1/D) sum_d x_d
//   var   = (1/D) sum_d (x_d - mu)^2            (biased; two passes)
//   rstd  = 1 / sqrt(var + eps)
//   xhat  = (x - mu) * rstd                      (no LayerNorm affine)
//   y     = xhat * (1 + scale[m]) + shift[m]     (m = modulation row of the token)
//
// and its exact gradient for L = sum dy * y, with the statistics given:
//
//   g      = dy * (1 + scale[m])
//   dx     = rstd * (g - mean_d(g) - xhat * mean_d(g * xhat))
//   dshift[m] += dy,   dscale[m] += dy * xhat     (summed over all tokens of m)
//
// Everything is accumulated in double, in plain sequential loops, one row at a
// time. Inputs are read as the exact values of their stored bits (fp32, bf16 or
// fp64), widened to double.
//
// Rows are packed: a segment table cu_seqlens[0..nseg] (cu_seqlens[0] = 0,
// non-decreasing) splits the rows into segments, and segment s uses modulation
// row mod_idx[s]. A dense [Bt, N, D] batch is the table {0, N, 2N, ...} with
// mod_idx[b] = b. Work is limited to rows [row_begin, row_end); per-row outputs
// are indexed relative to row_begin, and dshift/dscale are accumulated (+=) so a
// caller may feed the rows of one modulation row in several calls.

#include <cmath>
#include <cstdint>
#include <cstring>

namespace {

enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };

double element(const void* p, int dtype, int64_t i) {
    if (dtype == OR_F32) return (double)((const float*)p)[i];
    if (dtype == OR_F64) return ((const double*)p)[i];
    // bf16: the upper half of an IEEE binary32 with the same sign and exponent.
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    std::memcpy(&f, &bits, sizeof f);
    return (double)f;
}

bool valid_table(const int64_t* cu, const int64_t* mod, int64_t nseg, int64_t nmod) {
    if (!cu || nseg < 0 || cu[0] != 0) return false;
    for (int64_t s = 0; s < nseg; ++s) {
        if (cu[s + 1] < cu[s]) return false;
        if (!mod || mod[s] < 0 || mod[s] >= nmod) return false;
    }
    return true;
}

// The segment s with cu[s] <= row < cu[s+1] (a plain linear search).
int64_t segment_of(const int64_t* cu, int64_t nseg, int64_t row) {
    for (int64_t s = 0; s < nseg; ++s)
        if (cu[s] <= row && row < cu[s + 1]) return s;
    return -1;
}

}  // namespace

extern "C" {

// Forward over rows [row_begin, row_end). y: (row_end-row_begin) x D; mean, rstd:
// (row_end-row_begin). Returns 0, or -1 on invalid arguments.
int oracle_adaln_fwd(const void* x, const void* shift, const void* scale, int dtype, int64_t D,
                     const int64_t* cu_seqlens, const int64_t* mod_idx, int64_t nseg, int64_t nmod,
                     int64_t row_begin, int64_t row_end, double eps, double* y, double* mean,
                     double* rstd) {
    if (dtype < 0 || dtype > 2 || D <= 0 || !(eps > 0.0)) return -1;
    if (!valid_table(cu_seqlens, mod_idx, nseg, nmod)) return -1;
    if (row_begin < 0 || row_end < row_begin || row_end > cu_seqlens[nseg]) return -1;
    for (int64_t r = row_begin; r < row_end; ++r) {
        const int64_t m = mod_idx[segment_of(cu_seqlens, nseg, r)];
        const int64_t base = r * D;
        double sum = 0.0;
        for (int64_t d = 0; d < D; ++d) sum += element(x, dtype, base + d);
        const double mu = sum / (double)D;
        double ss = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            const double c = element(x, dtype, base + d) - mu;
            ss += c * c;
        }
        const double var = ss / (double)D;
        const double rho = 1.0 / std::sqrt(var + eps);
        const int64_t o = r - row_begin;
        for (int64_t d = 0; d < D; ++d) {
            const double xhat = (element(x, dtype, base + d) - mu) * rho;
            const double a = 1.0 + element(scale, dtype, m * D + d);
            const double b = element(shift, dtype, m * D + d);
            y[o * D + d] = xhat * a + b;
        }
        mean[o] = mu;
        rstd[o] = rho;
    }
    return 0;
}

// Backward over rows [row_begin, row_end) given that range's statistics
// (mean, rstd indexed relative to row_begin). dx: (row_end-row_begin) x D.
// dshift, dscale: nmod x D, accumulated into (+=). Returns 0, or -1.
int oracle_adaln_bwd(const void* dy, const void* x, const double* mean, const double* rstd,
                     const void* scale, int dtype, int64_t D, const int64_t* cu_seqlens,
                     const int64_t* mod_idx, int64_t nseg, int64_t nmod, int64_t row_begin,
                     int64_t row_end, double* dx, double* dshift, double* dscale) {
    if (dtype < 0 || dtype > 2 || D <= 0) return -1;
    if (!valid_table(cu_seqlens, mod_idx, nseg, nmod)) return -1;
    if (row_begin < 0 || row_end < row_begin || row_end > cu_seqlens[nseg]) return -1;
    for (int64_t r = row_begin; r < row_end; ++r) {
        const int64_t m = mod_idx[segment_of(cu_seqlens, nseg, r)];
        const int64_t base = r * D;
        const int64_t o = r - row_begin;
        const double mu = mean[o], rho = rstd[o];
        double sum_g = 0.0, sum_gx = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            const double xhat = (element(x, dtype, base + d) - mu) * rho;
            const double g = element(dy, dtype, base + d) * (1.0 + element(scale, dtype, m * D + d));
            sum_g += g;
            sum_gx += g * xhat;
        }
        const double mean_g = sum_g / (double)D;
        const double mean_gx = sum_gx / (double)D;
        for (int64_t d = 0; d < D; ++d) {
            const double xhat = (element(x, dtype, base + d) - mu) * rho;
            const double gy = element(dy, dtype, base + d);
            const double g = gy * (1.0 + element(scale, dtype, m * D + d));
            dx[o * D + d] = rho * (g - mean_g - xhat * mean_gx);
            dshift[m * D + d] += gy;
            dscale[m * D + d] += gy * xhat;
        }
    }
    return 0;
}

// double -> bf16 bits, round to nearest with ties to even, in one step (no
// intermediate fp32). bf16 keeps 8 significant bits; in the binade [2^(e-1), 2^e)
// its grid spacing is 2^(e-8), and below 2^-126 the spacing is fixed at 2^-133.
void oracle_round_to_bf16(const double* v, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        const double a = v[i];
        uint16_t sign = std::signbit(a) ? 0x8000 : 0x0000;
        if (std::isnan(a)) { out[i] = 0x7FC0; continue; }
        const double mag = std::fabs(a);
        if (std::isinf(mag)) { out[i] = sign | 0x7F80; continue; }
        if (mag == 0.0) { out[i] = sign; continue; }
        int e = 0;
        std::frexp(mag, &e);
        const double spacing = std::ldexp(1.0, e - 8 < -133 ? -133 : e - 8);
        const double units = mag / spacing;              // exact: divide by a power of two
        const double rounded = std::nearbyint(units);    // nearest, ties to even
        const double value = rounded * spacing;          // exact
        if (value >= std::ldexp(1.0, 128)) { out[i] = sign | 0x7F80; continue; }
        const float f = (float)value;                    // exact: <= 8 significant bits
        uint32_t bits;
        std::memcpy(&bits, &f, sizeof bits);
        out[i] = (uint16_t)(sign | (bits >> 16));
    }
}

}  // extern "C"
