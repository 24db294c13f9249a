// Fused AdaLN backward: dx plus the "D-tile coalesced reduction" of dshift/dscale.
//
// AdaptiveLoad technical summary, section 2.B, backward-pass bullet: instead of reducing
// the modulation gradients along the sequence with strided loads, threads are pinned to a
// feature index d and accumulate vertically down a tile of sequence rows, so every warp
// access is contiguous in D. Here that accumulation is fused with dx: a CTA walks its
// tile of rows once, each thread owning the same column vectors of every row; for each
// row it forms g = dy * (1 + scale), reduces sum(g) and sum(g * xhat) across the CTA
// (warp shuffles, then shared memory), writes dx, and adds dy and dy * xhat into its
// column accumulators. At the end of each (tile, segment) piece the accumulators are
// written as one fp32 partial; stage 2 sums the partials of each modulation row in a
// fixed order. No float atomics; dy and x are read from HBM exactly once.
#include "common.cuh"
#include "launch.h"

namespace adaln {

template <typename T, int NV, bool VARLEN>
__global__ void __launch_bounds__(RowShape<NV>::kMaxThreads) bwd_kernel(const BwdArgs a) {
    using IO = Io<T>;
    constexpr int VE = IO::VE;
    constexpr int RB = RowShape<NV>::kRows;
    __shared__ float red[2][RB][2][32];   // double-buffered per-warp sums of g and g*xhat

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t R = a.seg.R, D = a.D, V = D / VE;
    const int64_t r0 = tile_begin(b, R, G), r1 = tile_begin(b + 1, R, G);
    const T* __restrict__ x = static_cast<const T*>(a.x);
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    T* __restrict__ dx = static_cast<T*>(a.dx);
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

    int buf = 0;
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
        float sc1[NV][VE];
        float acc_dy[NV][VE], acc_dyx[NV][VE];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            uint4 vc = make_uint4(0, 0, 0, 0);
            if (ok[k]) vc = ld_keep(static_cast<const T*>(a.scale) + m * D + col[k]);
            IO::unpack(vc, sc1[k]);
#pragma unroll
            for (int j = 0; j < VE; ++j) {
                sc1[k][j] += 1.0f;
                acc_dy[k][j] = 0.0f;
                acc_dyx[k][j] = 0.0f;
            }
        }

        while (row < pend) {
            const int nr = (int)min((int64_t)RB, pend - row);
            uint4 xv[RB][NV], gv[RB][NV];
            float mu[RB], rs[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const bool live = i < nr;
                mu[i] = live ? __ldg(a.mean + row + i) : 0.0f;
                rs[i] = live ? __ldg(a.rstd + row + i) : 0.0f;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const bool on = live && ok[k];
                    xv[i][k] = on ? ld_stream(x + (row + i) * D + col[k]) : make_uint4(0, 0, 0, 0);
                    gv[i][k] = on ? ld_stream(dy + (row + i) * D + col[k]) : make_uint4(0, 0, 0, 0);
                }
            }
            // Row sums of g and g*xhat; column sums of dy and dy*xhat.
            float sums[2 * RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                float sg = 0.0f, sgx = 0.0f;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    if (!ok[k]) continue;
                    float fx[VE], fd[VE];
                    IO::unpack(xv[i][k], fx);
                    IO::unpack(gv[i][k], fd);
#pragma unroll
                    for (int j = 0; j < VE; ++j) {
                        const float xhat = (fx[j] - mu[i]) * rs[i];
                        const float g = fd[j] * sc1[k][j];
                        sg += g;
                        sgx = fmaf(g, xhat, sgx);
                        if (i < nr) {
                            acc_dy[k][j] += fd[j];
                            acc_dyx[k][j] = fmaf(fd[j], xhat, acc_dyx[k][j]);
                        }
                    }
                }
                sums[2 * i] = sg;
                sums[2 * i + 1] = sgx;
            }
            warp_sum(sums);
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                    red[buf][i][0][warp] = sums[2 * i];
                    red[buf][i][1][warp] = sums[2 * i + 1];
                }
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                if (i >= nr) continue;
                float tg = 0.0f, tgx = 0.0f;
                for (int w = 0; w < nwarps; ++w) {
                    tg += red[buf][i][0][w];
                    tgx += red[buf][i][1][w];
                }
                const float mg = tg * invD, mgx = tgx * invD;
                T* dxr = dx + (row + i) * D;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    if (!ok[k]) continue;
                    float fx[VE], fd[VE];
                    IO::unpack(xv[i][k], fx);
                    IO::unpack(gv[i][k], fd);
#pragma unroll
                    for (int j = 0; j < VE; ++j) {
                        const float xhat = (fx[j] - mu[i]) * rs[i];
                        const float g = fd[j] * sc1[k][j];
                        fd[j] = rs[i] * (g - mg - xhat * mgx);
                    }
                    st_vec(dxr + col[k], IO::pack(fd));
                }
            }
            buf ^= 1;
            row += nr;
        }
        // Piece (tile b, segment s) done: one fp32 partial row pair in slot b + s.
        float* P = a.partials + (b + s) * 2 * D;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (!ok[k]) continue;
#pragma unroll
            for (int j = 0; j < VE; j += 4) {
                *reinterpret_cast<float4*>(P + col[k] + j) =
                    make_float4(acc_dy[k][j], acc_dy[k][j + 1], acc_dy[k][j + 2], acc_dy[k][j + 3]);
                *reinterpret_cast<float4*>(P + D + col[k] + j) = make_float4(
                    acc_dyx[k][j], acc_dyx[k][j + 1], acc_dyx[k][j + 2], acc_dyx[k][j + 3]);
            }
        }
    }
    publish_status(err, a.status, a.header);
}

// Stage 2: dshift[m] / dscale[m] = sum of the partials of every piece of every segment
// whose modulation row is m, in a fixed order. CTA (blockIdx.x, m) covers `cw` float4
// columns; its 256 threads form cw columns x (256 / cw) splits of m's piece list (piece j
// goes to split j mod splits), combined by a fixed shared-memory tree.
template <bool VARLEN>
__global__ void __launch_bounds__(kStage2Threads) stage2_kernel(const Stage2Args a) {
    __shared__ float4 red[2][kStage2Threads];
    __shared__ int32_t list[kStage2Threads];
    __shared__ int32_t warp_count[kStage2Threads / 32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cw = a.cw, splits = kStage2Threads / cw;
    const int ci = tid % cw, k = tid / cw;
    const int64_t D4 = a.D / 4;
    const int64_t c4 = (int64_t)blockIdx.x * cw + ci;
    const bool cok = c4 < D4;
    const int64_t R = a.seg.R, G = a.G;
    const float4* P = reinterpret_cast<const float4*>(a.partials);

    for (int64_t m = blockIdx.y; m < a.seg.nmod; m += gridDim.y) {
        float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
        int64_t J = 0;  // pieces of row m seen so far, in segment order

        auto add_segment = [&](int64_t s) {
            const int64_t lo = max((int64_t)0, min(seg_start<VARLEN>(a.seg, s), R));
            const int64_t hi = max((int64_t)0, min(seg_start<VARLEN>(a.seg, s + 1), R));
            if (hi <= lo) return;
            const int64_t blo = tile_of_row(lo, R, G), bhi = tile_of_row(hi - 1, R, G);
            const int64_t n = bhi - blo + 1;
            for (int64_t j = ((k - J) % splits + splits) % splits; j < n; j += splits) {
                const int64_t slot = blo + j + s;
                if (cok) {
                    const float4 u = P[(slot * 2 + 0) * D4 + c4];
                    const float4 v = P[(slot * 2 + 1) * D4 + c4];
                    acc0.x += u.x; acc0.y += u.y; acc0.z += u.z; acc0.w += u.w;
                    acc1.x += v.x; acc1.y += v.y; acc1.z += v.z; acc1.w += v.w;
                }
            }
            J += n;
        };

        if constexpr (!VARLEN) {
            add_segment(m);
        } else {
            // Ordered scan of the segment table for the segments that use row m.
            for (int64_t base = 0; base < a.seg.nseg; base += kStage2Threads) {
                const int64_t s = base + tid;
                const bool hit = s < a.seg.nseg && (int64_t)__ldg(a.seg.mod + s) == m;
                const unsigned mask = __ballot_sync(0xFFFFFFFFu, hit);
                if (lane == 0) warp_count[warp] = __popc(mask);
                __syncthreads();
                int offset = 0, total = 0;
                for (int w = 0; w < kStage2Threads / 32; ++w) {
                    if (w < warp) offset += warp_count[w];
                    total += warp_count[w];
                }
                if (hit) list[offset + __popc(mask & ((1u << lane) - 1u))] = (int32_t)s;
                __syncthreads();
                for (int i = 0; i < total; ++i) add_segment(list[i]);
                __syncthreads();
            }
        }

        red[0][tid] = acc0;
        red[1][tid] = acc1;
        __syncthreads();
        for (int st = splits / 2; st >= 1; st >>= 1) {
            if (k < st) {
                const float4 u = red[0][tid + st * cw], v = red[1][tid + st * cw];
                float4& p = red[0][tid];
                float4& q = red[1][tid];
                p.x += u.x; p.y += u.y; p.z += u.z; p.w += u.w;
                q.x += v.x; q.y += v.y; q.z += v.z; q.w += v.w;
            }
            __syncthreads();
        }
        if (k == 0 && cok) {
            reinterpret_cast<float4*>(a.dshift)[m * D4 + c4] = red[0][tid];
            reinterpret_cast<float4*>(a.dscale)[m * D4 + c4] = red[1][tid];
        }
        __syncthreads();
    }
}

template <typename T, int NV, bool VARLEN>
static const void* bwd_fn() {
    return reinterpret_cast<const void*>(&bwd_kernel<T, NV, VARLEN>);
}

static const void* pick_bwd(int dtype, int nv, bool varlen) {
#define ADALN_PICK(T)                                                            \
    switch (nv) {                                                                \
        case 1: return varlen ? bwd_fn<T, 1, true>() : bwd_fn<T, 1, false>();     \
        case 2: return varlen ? bwd_fn<T, 2, true>() : bwd_fn<T, 2, false>();     \
        case 3: return varlen ? bwd_fn<T, 3, true>() : bwd_fn<T, 3, false>();     \
        case 4: return varlen ? bwd_fn<T, 4, true>() : bwd_fn<T, 4, false>();     \
        default: return nullptr;                                                 \
    }
    if (dtype == 0) { ADALN_PICK(float) }
    if (dtype == 1) { ADALN_PICK(__nv_bfloat16) }
#undef ADALN_PICK
    return nullptr;
}

cudaError_t bwd_blocks_per_sm(int dtype, int nv, bool varlen, int tpb, int* out) {
    const void* fn = pick_bwd(dtype, nv, varlen);
    if (!fn) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, fn, tpb, 0);
}

cudaError_t launch_bwd(const BwdArgs& args, int dtype, int nv, bool varlen, int64_t G, int tpb,
                       cudaStream_t stream) {
    const void* fn = pick_bwd(dtype, nv, varlen);
    if (!fn) return cudaErrorInvalidValue;
    BwdArgs a = args;
    void* params[] = {&a};
    return cudaLaunchKernel(fn, dim3((unsigned)G), dim3((unsigned)tpb), params, 0, stream);
}

cudaError_t launch_stage2(const Stage2Args& args, bool varlen, cudaStream_t stream) {
    const int64_t D4 = args.D / 4;
    const int64_t gy = args.seg.nmod < 65535 ? args.seg.nmod : 65535;
    const dim3 grid((unsigned)((D4 + args.cw - 1) / args.cw), (unsigned)gy);
    Stage2Args a = args;
    void* params[] = {&a};
    const void* fn = varlen ? reinterpret_cast<const void*>(&stage2_kernel<true>)
                            : reinterpret_cast<const void*>(&stage2_kernel<false>);
    return cudaLaunchKernel(fn, grid, dim3(kStage2Threads), params, 0, stream);
}

}  // namespace adaln
