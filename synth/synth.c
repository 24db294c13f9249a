/*
 * Seeded synthetic inputs for the fused AdaLN operator.
 *
 * This module is the ONLY code shared by the CPU oracle side and the CUDA side:
 * both consume the exact bits it writes. It holds random-number generation and
 * rounding to the I/O dtype, and none of the operator's arithmetic.
 *
 * Generator: counter-based SplitMix64 (Steele, Lea & Flood, "Fast Splittable
 * Pseudorandom Number Generators", OOPSLA 2014): the k-th output of a stream is
 * the SplitMix64 finaliser applied to key + (k+1)*gamma, so any element can be
 * produced independently of the others (parallel fills are deterministic).
 * Normals: Box-Muller transform (Box & Muller, 1958) in double precision; element
 * 2j uses the cosine branch and element 2j+1 the sine branch of pair j.
 * Rounding: double -> bf16 and double -> fp32, both round-to-nearest-even, done
 * once, straight from double.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

enum { SYNTH_F32 = 0, SYNTH_BF16 = 1, SYNTH_F64 = 2 };

/* Row recipes for synth_rows(). */
enum {
    SYNTH_ROWS_NORMAL = 0,      /* x = mean + std * z                                         */
    SYNTH_ROWS_SCALED = 1,      /* x = o_r + s_r * z, s_r ~ LogNormal(0, 0.5), o_r ~ N(0, 0.5) */
    SYNTH_ROWS_ADVERSARIAL = 2  /* SCALED, with every 16th-row class replaced (see below)     */
};

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of one named stream of one seed. */
static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GAMMA) ^ mix64(stream * GAMMA + 0x632BE59BD9B4E019ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t k) { return mix64(key + (k + 1) * GAMMA); }

/* Uniform on the open interval (0, 1) with 53 random bits. */
static inline double unif_open(uint64_t r) { return ((double)(r >> 11) + 0.5) * 0x1.0p-53; }

static inline double normal_at(uint64_t key, uint64_t i) {
    uint64_t j = i >> 1;
    double u1 = unif_open(draw(key, 2 * j));
    double u2 = unif_open(draw(key, 2 * j + 1));
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586476925 * u2;
    return (i & 1) ? rad * sin(ang) : rad * cos(ang);
}

/* double -> bf16 bits, round to nearest, ties to even (bf16: 8 exponent bits, 7 stored
 * mantissa bits). Works on the double's bit pattern: keep the top 8 significant bits of
 * the value expressed on the bf16 grid of its binade. */
static uint16_t to_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                      /* a = f * 2^e, f in [0.5, 1) -> unit in last place 2^(e-8) */
    int q = e - 8;
    if (q < -133) q = -133;            /* below the normal range the grid spacing is fixed at 2^-133 */
    double k = ldexp(a, -q);           /* exact: power-of-two scaling */
    double kr = nearbyint(k);          /* default mode: nearest, ties to even */
    double r = ldexp(kr, q);
    if (r >= 0x1.0p128) return sign | 0x7F80;
    float f = (float)r;                /* exact: r has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return (uint16_t)(sign | (bits >> 16));
}

static inline void store(void* out, int dtype, int64_t i, double v) {
    if (dtype == SYNTH_F32) ((float*)out)[i] = (float)v;
    else if (dtype == SYNTH_BF16) ((uint16_t*)out)[i] = to_bf16(v);
    else ((double*)out)[i] = v;
}

/* out[i] = mean + std * z_i for i in [0, n), z from (seed, stream). */
int synth_normal(uint64_t seed, uint64_t stream, int64_t n, double mean, double std, int dtype,
                 void* out) {
    if (n < 0 || dtype < 0 || dtype > 2 || (n > 0 && !out)) return -1;
    uint64_t key = stream_key(seed, stream * 8 + 0);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) store(out, dtype, i, mean + std * normal_at(key, (uint64_t)i));
    return 0;
}

/* Row-structured activations for a packed tensor of cu_seqlens[nseg] rows of width D.
 *   NORMAL:      x = mean + std * z.
 *   SCALED:      per global row g, o = 0.5 * z_o(g), s = exp(0.5 * z_s(g)); x = o + s * z.
 *   ADVERSARIAL: SCALED, except by the row's index r inside its segment:
 *       r == 0          -> all zeros
 *       r % 16 == 1     -> mean U(-1e3, 1e3), std 1e-2
 *       r % 16 == 2     -> constant row, value U(-1e3, 1e3)
 *       r % 16 == 3     -> (fp32 only) 65504 * z when (r / 16) is even, else exact +-65504
 *                          with a random sign per element.
 * mean/std are used by NORMAL only. */
int synth_rows(uint64_t seed, uint64_t stream, int mode, const int64_t* cu_seqlens, int64_t nseg,
               int64_t D, double mean, double std, int dtype, void* out) {
    if (!cu_seqlens || nseg < 0 || D <= 0 || dtype < 0 || dtype > 2 || mode < 0 || mode > 2) return -1;
    for (int64_t s = 0; s < nseg; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s] || cu_seqlens[0] != 0) return -1;
    if (cu_seqlens[nseg] > 0 && !out) return -1;
    uint64_t kx = stream_key(seed, stream * 8 + 0);
    uint64_t ko = stream_key(seed, stream * 8 + 1);
    uint64_t ks = stream_key(seed, stream * 8 + 2);
    uint64_t ku = stream_key(seed, stream * 8 + 3);
    uint64_t kb = stream_key(seed, stream * 8 + 4);
    for (int64_t s = 0; s < nseg; ++s) {
        int64_t g0 = cu_seqlens[s], g1 = cu_seqlens[s + 1];
#pragma omp parallel for schedule(static)
        for (int64_t g = g0; g < g1; ++g) {
            int64_t r = g - g0;
            int64_t base = g * D;
            int cls = (mode == SYNTH_ROWS_ADVERSARIAL) ? (r == 0 ? -1 : (int)(r % 16)) : 0;
            if (mode == SYNTH_ROWS_NORMAL) {
                for (int64_t d = 0; d < D; ++d)
                    store(out, dtype, base + d, mean + std * normal_at(kx, (uint64_t)(base + d)));
            } else if (cls == -1) {
                for (int64_t d = 0; d < D; ++d) store(out, dtype, base + d, 0.0);
            } else if (cls == 1) {
                double mu = -1e3 + 2e3 * unif_open(draw(ku, (uint64_t)g));
                for (int64_t d = 0; d < D; ++d)
                    store(out, dtype, base + d, mu + 1e-2 * normal_at(kx, (uint64_t)(base + d)));
            } else if (cls == 2) {
                double c = -1e3 + 2e3 * unif_open(draw(ku, (uint64_t)g));
                for (int64_t d = 0; d < D; ++d) store(out, dtype, base + d, c);
            } else if (cls == 3 && dtype == SYNTH_F32) {
                int exact = (int)((r / 16) % 2);
                for (int64_t d = 0; d < D; ++d) {
                    double v = exact ? ((draw(kb, (uint64_t)(base + d)) >> 63) ? -65504.0 : 65504.0)
                                     : 65504.0 * normal_at(kx, (uint64_t)(base + d));
                    store(out, dtype, base + d, v);
                }
            } else {
                double o = 0.5 * normal_at(ko, (uint64_t)g);
                double sc = exp(0.5 * normal_at(ks, (uint64_t)g));
                for (int64_t d = 0; d < D; ++d)
                    store(out, dtype, base + d, o + sc * normal_at(kx, (uint64_t)(base + d)));
            }
        }
    }
    return 0;
}

/* Round an array of doubles to bf16 bits (exposed for the generator's own tests). */
void synth_round_bf16(const double* v, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = to_bf16(v[i]);
}
