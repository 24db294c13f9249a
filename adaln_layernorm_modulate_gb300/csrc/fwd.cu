// Fused AdaLN forward: per-row statistics + modulation in one launch.
//
// AdaptiveLoad technical summary, section 2.B, forward-pass bullet: mean and variance
// are kept on chip and reduced by warp shuffles followed by a block reduction, and the
// modulation is applied on a further pass over D. Here one CTA owns a contiguous tile of
// rows; each thread owns the same 16-byte column vectors of every row, so the row is held
// in registers and the three passes (sum, centred sum of squares, modulated write) run
// over registers, touching HBM once for x and once for y.
//
// Variance: sum and centred sum of squares of d = x - x[row, 0]. Subtracting the row's
// first element first (shifted data, Chan, Golub & LeVeque 1983) keeps the fp32 sums of
// rows with a large mean and a tiny spread exact enough; the second pass is centred on
// the mean of d (two-pass), never E[x^2] - E[x]^2.
#include "common.cuh"
#include "launch.h"

namespace adaln {

template <typename T, int NV, bool VARLEN>
__global__ void __launch_bounds__(RowShape<NV>::kMaxThreads) fwd_kernel(const FwdArgs a) {
    using IO = Io<T>;
    constexpr int VE = IO::VE;
    constexpr int RB = RowShape<NV>::kRows;
    __shared__ float red1[RB][32];
    __shared__ float red2[RB][32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t R = a.seg.R, D = a.D, V = D / VE;
    const int64_t r0 = tile_begin(b, R, G), r1 = tile_begin(b + 1, R, G);
    const T* __restrict__ x = static_cast<const T*>(a.x);
    T* __restrict__ y = static_cast<T*>(a.y);
    const float invD = 1.0f / (float)D;

    uint32_t err = validate_segments<VARLEN>(a.seg, b, G);

    int64_t col[NV];
    bool ok[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int64_t v = tid + (int64_t)k * blockDim.x;
        ok[k] = v < V;
        col[k] = v * VE;
    }

    int64_t row = r0;
    int64_t s = R > 0 ? seg_find<VARLEN>(a.seg, r0) : 0;
    while (row < r1) {
        while (s < a.seg.nseg && seg_start<VARLEN>(a.seg, s + 1) <= row) ++s;
        if (s >= a.seg.nseg) {
            err |= kErrSeqlens;
            break;
        }
        const int64_t pend = min(seg_start<VARLEN>(a.seg, s + 1), r1);
        const int64_t m = seg_mod<VARLEN>(a.seg, s);
        if (m < 0 || m >= a.seg.nmod) {
            err |= kErrModIdx;
            row = pend;
            continue;
        }
        // This segment's modulation for my columns: shift and (1 + scale) in fp32.
        float sh[NV][VE], sc1[NV][VE];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            uint4 vs = make_uint4(0, 0, 0, 0), vc = make_uint4(0, 0, 0, 0);
            if (ok[k]) {
                vs = ld_keep(static_cast<const T*>(a.shift) + m * D + col[k]);
                vc = ld_keep(static_cast<const T*>(a.scale) + m * D + col[k]);
            }
            IO::unpack(vs, sh[k]);
            IO::unpack(vc, sc1[k]);
#pragma unroll
            for (int j = 0; j < VE; ++j) sc1[k][j] += 1.0f;
        }

        while (row < pend) {
            const int nr = (int)min((int64_t)RB, pend - row);
            uint4 xv[RB][NV];
            float K[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const T* xr = x + (row + i) * D;
                K[i] = (i < nr) ? IO::first(xr) : 0.0f;
#pragma unroll
                for (int k = 0; k < NV; ++k)
                    xv[i][k] = (i < nr && ok[k]) ? ld_stream(xr + col[k]) : make_uint4(0, 0, 0, 0);
            }
            // Pass 1: sum of d = x - K.
            float s1[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                s1[i] = 0.0f;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    if (!ok[k]) continue;
                    float f[VE];
                    IO::unpack(xv[i][k], f);
#pragma unroll
                    for (int j = 0; j < VE; ++j) s1[i] += f[j] - K[i];
                }
            }
            warp_sum(s1);
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < RB; ++i) red1[i][warp] = s1[i];
            }
            __syncthreads();
            float md[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                float t = 0.0f;
                for (int w = 0; w < nwarps; ++w) t += red1[i][w];
                md[i] = t * invD;
            }
            // Pass 2: centred sum of squares.
            float s2[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                s2[i] = 0.0f;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    if (!ok[k]) continue;
                    float f[VE];
                    IO::unpack(xv[i][k], f);
#pragma unroll
                    for (int j = 0; j < VE; ++j) {
                        const float c = (f[j] - K[i]) - md[i];
                        s2[i] = fmaf(c, c, s2[i]);
                    }
                }
            }
            warp_sum(s2);
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < RB; ++i) red2[i][warp] = s2[i];
            }
            __syncthreads();
            // Pass 3: modulated write.
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                if (i >= nr) continue;
                float t = 0.0f;
                for (int w = 0; w < nwarps; ++w) t += red2[i][w];
                const float rs = rsqrtf(t * invD + a.eps);
                T* yr = y + (row + i) * D;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    if (!ok[k]) continue;
                    float f[VE];
                    IO::unpack(xv[i][k], f);
#pragma unroll
                    for (int j = 0; j < VE; ++j) {
                        const float xhat = ((f[j] - K[i]) - md[i]) * rs;
                        f[j] = fmaf(xhat, sc1[k][j], sh[k][j]);
                    }
                    st_vec(yr + col[k], IO::pack(f));
                }
                if (tid == 0) {
                    a.mean[row + i] = K[i] + md[i];
                    a.rstd[row + i] = rs;
                }
            }
            row += nr;
        }
    }
    publish_status(err, a.status, a.header);
}

template <typename T, int NV, bool VARLEN>
static const void* fwd_fn() {
    return reinterpret_cast<const void*>(&fwd_kernel<T, NV, VARLEN>);
}

static const void* pick_fwd(int dtype, int nv, bool varlen) {
#define ADALN_PICK(T)                                                            \
    switch (nv) {                                                                \
        case 1: return varlen ? fwd_fn<T, 1, true>() : fwd_fn<T, 1, false>();     \
        case 2: return varlen ? fwd_fn<T, 2, true>() : fwd_fn<T, 2, false>();     \
        case 3: return varlen ? fwd_fn<T, 3, true>() : fwd_fn<T, 3, false>();     \
        case 4: return varlen ? fwd_fn<T, 4, true>() : fwd_fn<T, 4, false>();     \
        default: return nullptr;                                                 \
    }
    if (dtype == 0) { ADALN_PICK(float) }
    if (dtype == 1) { ADALN_PICK(__nv_bfloat16) }
#undef ADALN_PICK
    return nullptr;
}

cudaError_t fwd_blocks_per_sm(int dtype, int nv, bool varlen, int tpb, int* out) {
    const void* fn = pick_fwd(dtype, nv, varlen);
    if (!fn) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, fn, tpb, 0);
}

cudaError_t launch_fwd(const FwdArgs& args, int dtype, int nv, bool varlen, int64_t G, int tpb,
                       cudaStream_t stream) {
    const void* fn = pick_fwd(dtype, nv, varlen);
    if (!fn) return cudaErrorInvalidValue;
    FwdArgs a = args;
    void* params[] = {&a};
    return cudaLaunchKernel(fn, dim3((unsigned)G), dim3((unsigned)tpb), params, 0, stream);
}

}  // namespace adaln
