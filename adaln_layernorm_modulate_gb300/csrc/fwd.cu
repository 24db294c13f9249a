// Fused AdaLN forward: per-row statistics + modulation in one launch.
//
// AdaptiveLoad technical summary, section 2.B, forward-pass bullet: mean and variance
// are kept on chip and reduced by warp shuffles followed by a block reduction, and the
// modulation is applied on a further pass over D. Here one CTA owns a contiguous tile of
// rows; each thread owns the same 16-byte column vectors of every row, so a row is held
// in registers and the three passes (sum, centred sum of squares, modulated write) run
// over registers, touching HBM once for x and once for y.
//
// Memory-level parallelism, three staging modes:
//  - bulk ring: one thread copies whole rows into a shared-memory ring of `stages` rounds
//    with bulk (TMA) copies, one instruction per row, completing on a per-slot mbarrier; it
//    refills the previous round's slot at the top of each round, when every thread has
//    passed that round's barriers. It gets rows flowing fastest after launch: the choice
//    for short tiles.
//  - copy ring: every thread copies its own 16-byte vectors (and the row's first word) of
//    the round `stages` ahead with cp.async and waits only on its own copy groups: no
//    single producer on the CTA's critical path. It sustains a few percent more bandwidth
//    on long tiles of bf16 rows mapped three vectors a thread (the one form planned).
//  - plain: rows too wide for a ring of two rounds load straight into registers.
// FULL: the CTA's threads cover the row exactly (no idle vector slots), so no lane masking.
//
// Variance: sum and centred sum of squares of d = x - x[row, 0]. Subtracting the row's
// first element first (shifted data, Chan, Golub & LeVeque 1983) keeps the fp32 sums of
// rows with a large mean and a tiny spread accurate; the second pass is centred on the
// mean of d (two-pass), never E[x^2] - E[x]^2. Elementwise math runs on fp32 pairs.
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace adaln {

template <typename T, int NV, bool VARLEN, int RING, bool FULL>
__global__ void __launch_bounds__(max_threads(NV, Io<T>::VE)) fwd_kernel(const FwdArgs a) {
    pdl_begin();
    constexpr bool BULK = RING == kRingBulk, COPY = RING == kRingCopy;
    using IO = Io<T>;
    constexpr int VE = IO::VE;
    constexpr int PV = VE / 2;  // fp32 pairs per 16-byte vector
    constexpr int RB = RowShape<NV>::kFwdRows;
    extern __shared__ uint4 ring[];
    __shared__ __align__(16) float red1[RB][32];
    __shared__ __align__(16) float red2[RB][32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int TPB = blockDim.x;
    const int nwarps = TPB >> 5;
    int ng = 1;  // warps rounded up to a power of two
    while (ng < nwarps) ng <<= 1;
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t R = a.seg.R, D = a.D, V = D / VE;
    const int64_t r0 = tile_begin(b, R, G), r1 = tile_begin(b + 1, R, G);
    const char* __restrict__ xb = static_cast<const char*>(a.x);
    char* __restrict__ yb = static_cast<char*>(a.y);
    const int64_t row_bytes = D * (int64_t)sizeof(T);
    const float invD = 1.0f / (float)D;
    const int ns = a.stages;

    // Ring layout (32-bit shared addresses): ns mbarriers (first 128 bytes, bulk ring), then
    // [ns][RB] rows, each row at the offsets it has in global memory (thread t's vector k at
    // (t + k*TPB)*16), so a bulk copy lands every thread's vectors where it reads them; the
    // copy ring then keeps [ns][RB][TPB] words, each thread's copy of the row's first word.
    __shared__ int abort_flag;
    const uint32_t vk = (uint32_t)TPB * 16u;           // one vector index k across the CTA
    const uint32_t vrow = (uint32_t)NV * vk;           // one row slot
    const uint32_t vslot = (uint32_t)RB * vrow;        // one round
    const uint32_t bars = smem_addr(ring);
    const uint32_t data = bars + 128u;
    const uint32_t my_vec = data + (uint32_t)tid * 16u;
    const uint32_t krow = (uint32_t)TPB * 4u, kslot = (uint32_t)RB * krow;
    const uint32_t my_k = data + (uint32_t)ns * vslot + (uint32_t)tid * 4u;

    zero_absent_warps<RB>(red1, nwarps);
    zero_absent_warps<RB>(red2, nwarps);
    uint32_t err = validate_segments<VARLEN>(a.seg, b, G);
    if constexpr (BULK) {
        if (tid == 0) {
            for (int q = 0; q < ns; ++q) mbar_init(bars + 8u * q, 1);
            abort_flag = 0;
            mbar_fence_init();
        }
        __syncthreads();
    }

    uint32_t colb[NV];  // byte offset of my vector k within a row
    bool ok[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int64_t v = tid + (int64_t)k * TPB;
        ok[k] = FULL || v < V;
        colb[k] = (uint32_t)(v * 16);
    }

    const int64_t s0 = R > 0 ? seg_find<VARLEN>(a.seg, r0) : 0;
    Walker<VARLEN, RB> cw{r0, s0, -1, false};
    Walker<VARLEN, RB> pw{r0, s0, -1, false};  // the copies' walker, ns rounds ahead

    // Thread 0: copy the producer walker's next round into ring slot `slot`.
    auto issue = [&](int slot) {
        int64_t rs, sg;
        int nr;
        if (pw.next(a.seg, r1, rs, nr, sg)) {
            const uint32_t bar = bars + 8u * (uint32_t)slot;
            mbar_arrive_expect_tx(bar, (uint32_t)(nr * row_bytes));
#pragma unroll
            for (int i = 0; i < RB; ++i)
                if (i < nr && ADALN_IN_ROW(rs + i, R, 0, row_bytes, row_bytes) &&
                    ADALN_IN_RING(bars, data + (uint32_t)slot * vslot + (uint32_t)i * vrow, row_bytes))
                    bulk_load(data + (uint32_t)slot * vslot + (uint32_t)i * vrow, xb + (rs + i) * row_bytes,
                              (uint32_t)row_bytes, bar);
        }
    };
    // Copy ring: this thread's vectors of the walker's next round into ring slot `slot`.
    auto prefetch = [&](int slot) {
        int64_t rs, sg;
        int nr;
        if (pw.next(a.seg, r1, rs, nr, sg)) {
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                if (i >= nr || !ADALN_IN_ROW(rs + i, R, 0, 4, row_bytes)) continue;
                const char* src = xb + (rs + i) * row_bytes;
                const uint32_t dst = my_vec + (uint32_t)slot * vslot + (uint32_t)i * vrow;
                if (ADALN_IN_RING(bars, my_k + (uint32_t)slot * kslot + (uint32_t)i * krow, 4))
                    cp_async4_sa(my_k + (uint32_t)slot * kslot + (uint32_t)i * krow, src);
#pragma unroll
                for (int k = 0; k < NV; ++k)
                    if (ok[k] && ADALN_IN_ROW(rs + i, R, colb[k], 16, row_bytes) &&
                        ADALN_IN_RING(bars, dst + (uint32_t)k * vk, 16))
                        cp_async16_sa(dst + (uint32_t)k * vk, src + colb[k]);
            }
        }
        cp_async_commit();
    };
    if constexpr (BULK) {
        if (tid == 0)
            for (int q = 0; q < ns; ++q) issue(q);
    }
    if constexpr (COPY) {
        for (int q = 0; q < ns; ++q) prefetch(q);
    }

    int slot = 0;
    uint32_t lap = 0;  // completed passes over the ring: the parity of the slot's phase
    bool started = false;  // a previous round exists whose slot can be refilled
    int64_t cur_s = -1;
    bool cur_ok = false;
    f2r sh[NV][PV], sc1[NV][PV];
    int64_t row, s;
    int nr;
    while (cw.next(a.seg, r1, row, nr, s)) {
        uint4 xv[RB][NV];
        float K[RB];
        if constexpr (BULK) {
            // The previous round's slot has been read by every thread (they all passed that
            // round's barriers): refill it ns rounds ahead before waiting on this one.
            if (tid == 0 && started) issue(slot == 0 ? ns - 1 : slot - 1);
            started = true;
            if (!mbar_wait_bounded(bars + 8u * (uint32_t)slot, lap & 1u, &abort_flag)) err |= kErrTimeout;
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const uint32_t rowsa = (uint32_t)slot * vslot + (uint32_t)i * vrow;
#pragma unroll
                for (int k = 0; k < NV; ++k)
                    xv[i][k] = (i < nr && ok[k] && ADALN_IN_RING(bars, my_vec + rowsa + (uint32_t)k * vk, 16))
                                   ? lds128(my_vec + rowsa + (uint32_t)k * vk)
                                   : make_uint4(0, 0, 0, 0);
                K[i] = (i < nr && ADALN_IN_RING(bars, data + rowsa, 4)) ? IO::first_of_word(lds32(data + rowsa))
                                                                          : 0.0f;
            }
        } else if constexpr (COPY) {
            cp_async_wait(ns - 1);  // this thread's copies of this round have landed
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const uint32_t src = my_vec + (uint32_t)slot * vslot + (uint32_t)i * vrow;
#pragma unroll
                for (int k = 0; k < NV; ++k)
                    xv[i][k] = (i < nr && ok[k] && ADALN_IN_RING(bars, src + (uint32_t)k * vk, 16))
                                   ? lds128(src + (uint32_t)k * vk)
                                   : make_uint4(0, 0, 0, 0);
                K[i] = (i < nr && ADALN_IN_RING(bars, my_k + (uint32_t)slot * kslot + (uint32_t)i * krow, 4))
                           ? IO::first_of_word(lds32(my_k + (uint32_t)slot * kslot + (uint32_t)i * krow))
                           : 0.0f;
            }
        } else {
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const char* src = xb + (row + i) * row_bytes;
#pragma unroll
                for (int k = 0; k < NV; ++k)
                    xv[i][k] = (i < nr && ok[k] && ADALN_IN_ROW(row + i, R, colb[k], 16, row_bytes))
                                   ? ld_stream(src + colb[k])
                                   : make_uint4(0, 0, 0, 0);
                K[i] = (i < nr && ADALN_IN_ROW(row + i, R, 0, 4, row_bytes)) ? IO::first(src) : 0.0f;
            }
        }

        if (s != cur_s) {
            // A new segment: its modulation for my columns, shift and (1 + scale) in fp32.
            cur_s = s;
            const int64_t m = seg_mod<VARLEN>(a.seg, s);
            cur_ok = m >= 0 && m < a.seg.nmod;
            if (!cur_ok) err |= kErrModIdx;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                uint4 vs = make_uint4(0, 0, 0, 0), vc = make_uint4(0, 0, 0, 0);
                if (cur_ok && ok[k] && ADALN_IN(kDbgMod, m >= 0 && m < a.seg.nmod && colb[k] + 16 <= row_bytes)) {
                    vs = ld_keep(static_cast<const char*>(a.shift) + m * row_bytes + colb[k]);
                    vc = ld_keep(static_cast<const char*>(a.scale) + m * row_bytes + colb[k]);
                }
                IO::unpackp(vs, sh[k]);
                IO::unpackp(vc, sc1[k]);
                const f2r one = p_splat(1.0f);
#pragma unroll
                for (int p = 0; p < PV; ++p) sc1[k][p] = p_add(sc1[k][p], one);
            }
        }

        if (cur_ok) {  // uniform across the CTA
            // d = x - K, kept for all three passes; idle lanes hold d = 0.
            f2r d[RB][NV][PV];
            float s1[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const f2r kk = p_splat(K[i]);
                f2r acc0 = kPairZero, acc1 = kPairZero;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    IO::unpackp(xv[i][k], d[i][k]);
#pragma unroll
                    for (int p = 0; p < PV; ++p) {
                        d[i][k][p] = p_sub(d[i][k][p], kk);
                        if (!FULL && !ok[k]) d[i][k][p] = kPairZero;
                        if (p & 1) acc1 = p_add(acc1, d[i][k][p]);
                        else acc0 = p_add(acc0, d[i][k][p]);
                    }
                }
                s1[i] = p_hsum(p_add(acc0, acc1));
            }
            // Pass 1: mean of d.
            warp_sum(s1);
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < RB; ++i) red1[i][warp] = s1[i];
            }
            __syncthreads();
            cta_sum(red1, ng, lane, s1);
            // Pass 2: centred sum of squares.
            float s2[RB], md[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                md[i] = s1[i] * invD;
                const f2r pm = p_splat(md[i]);
                f2r acc0 = kPairZero, acc1 = kPairZero;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
#pragma unroll
                    for (int p = 0; p < PV; ++p) {
                        d[i][k][p] = p_sub(d[i][k][p], pm);
                        if (!FULL && !ok[k]) d[i][k][p] = kPairZero;
                        if (p & 1) acc1 = p_fma(d[i][k][p], d[i][k][p], acc1);
                        else acc0 = p_fma(d[i][k][p], d[i][k][p], acc0);
                    }
                }
                s2[i] = p_hsum(p_add(acc0, acc1));
            }
            warp_sum(s2);
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < RB; ++i) red2[i][warp] = s2[i];
            }
            __syncthreads();
            cta_sum(red2, ng, lane, s2);
            // Pass 3: y = (d - mean_d) * rstd * (1 + scale) + shift.
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                if (i >= nr) continue;
                const float rs = rsqrtf(s2[i] * invD + a.eps);
                const f2r prs = p_splat(rs);
                char* yr = yb + (row + i) * row_bytes;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    if (!ok[k]) continue;
                    f2r o[PV];
#pragma unroll
                    for (int p = 0; p < PV; ++p) o[p] = p_fma(p_mul(d[i][k][p], prs), sc1[k][p], sh[k][p]);
                    if (ADALN_IN_ROW(row + i, R, colb[k], 16, row_bytes)) st_vec(yr + colb[k], IO::packp(o));
                }
                if (tid == 0 && ADALN_IN(kDbgStats, row + i >= 0 && row + i < R)) {
                    a.mean[row + i] = K[i] + md[i];
                    a.rstd[row + i] = rs;
                }
            }
        }
        if constexpr (BULK) {
            if (!cur_ok) __syncthreads();  // a skipped round still fences the slot's readers
            if (++slot == ns) {
                slot = 0;
                ++lap;
            }
        }
        if constexpr (COPY) {
            prefetch(slot);  // this slot's data is in my registers: refill it ns rounds ahead
            slot = slot + 1 == ns ? 0 : slot + 1;
        }
    }
    if (cw.bad) err |= kErrSeqlens;
    if constexpr (COPY) cp_async_wait_all();
    if constexpr (BULK) {
        // After a timed-out wait, copies may still be in flight into this CTA's shared
        // memory: give each slot's outstanding phase one more bounded wait before exiting.
        __syncthreads();
        if (tid == 0 && abort_flag) {
            volatile int never = 0;
            for (int q = 0; q < ns; ++q) {
                if (q >= slot && lap == 0) continue;  // never used
                const uint32_t last = q < slot ? lap : lap - 1;  // pass of the slot's last round
                mbar_wait_bounded(bars + 8u * q, last & 1u, &never);
            }
        }
    }
    publish_status(err, a.status, a.header);
}

template <typename T, int NV, bool VARLEN, int RING, bool FULL>
static const void* fwd_fn() {
    return reinterpret_cast<const void*>(&fwd_kernel<T, NV, VARLEN, RING, FULL>);
}

// Instantiated variants: the bulk ring with a full or a partial row; the copy ring only with
// the one mapping the host plans it with (bf16, three vectors a thread, full rows); plain
// loads (partial row).
template <typename T, int NV, bool VARLEN>
static const void* pick_variant(int ring, bool full) {
    if (ring == kRingBulk)
        return full ? fwd_fn<T, NV, VARLEN, kRingBulk, true>() : fwd_fn<T, NV, VARLEN, kRingBulk, false>();
    if (ring == kRingCopy) {
        if constexpr (NV == 3 && std::is_same<T, __nv_bfloat16>::value)
            if (full) return fwd_fn<T, NV, VARLEN, kRingCopy, true>();
        return nullptr;
    }
    return fwd_fn<T, NV, VARLEN, kRingNone, false>();
}

template <typename T, bool VARLEN>
static const void* pick_nv(int nv, int ring, bool full) {
    switch (nv) {
        case 1: return pick_variant<T, 1, VARLEN>(ring, full);
        case 2: return pick_variant<T, 2, VARLEN>(ring, full);
        case 3: return pick_variant<T, 3, VARLEN>(ring, full);
        case 4: return pick_variant<T, 4, VARLEN>(ring, full);
        case 6: return pick_variant<T, 6, VARLEN>(ring, full);
        case 8: return pick_variant<T, 8, VARLEN>(ring, full);
        default: return nullptr;
    }
}

static const void* pick_fwd(int dtype, int nv, bool varlen, int ring, bool full) {
    if (dtype == 0) return varlen ? pick_nv<float, true>(nv, ring, full) : pick_nv<float, false>(nv, ring, full);
    if (dtype == 1)
        return varlen ? pick_nv<__nv_bfloat16, true>(nv, ring, full)
                      : pick_nv<__nv_bfloat16, false>(nv, ring, full);
    return nullptr;
}

cudaError_t fwd_blocks_per_sm(int dtype, int nv, bool varlen, int ring, bool full, int tpb,
                              size_t smem, int* out) {
    const void* fn = pick_fwd(dtype, nv, varlen, ring, full);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = allow_dynamic_smem(fn);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, fn, tpb, smem);
}

cudaError_t launch_fwd(const FwdArgs& args, int dtype, int nv, bool varlen, int ring, bool full,
                       int64_t G, int tpb, size_t smem, cudaStream_t stream) {
    const void* fn = pick_fwd(dtype, nv, varlen, ring, full);
    if (!fn) return cudaErrorInvalidValue;
    FwdArgs a = args;
    void* params[] = {&a};
    return launch_dependent(fn, dim3((unsigned)G), dim3((unsigned)tpb), params, smem, stream);
}

// Row statistics alone, for a backward whose forward kept no statistics: the forward's row
// mapping (NV, blockDim) and its passes 1 and 2 verbatim (shifted sum, centred sum of
// squares, the same warp and CTA reductions), so every row gets bitwise the mean and rstd
// the forward computed. Rows are independent here: CTA b takes rows b*R/G ... in rounds of
// RB consecutive rows, loaded straight into registers.
template <typename T, int NV>
__global__ void __launch_bounds__(max_threads(NV, Io<T>::VE)) stats_kernel(const void* x, float* mean,
                                                                         float* rstd, int64_t R, int64_t D,
                                                                         float eps) {
    pdl_begin();
    using IO = Io<T>;
    constexpr int VE = IO::VE;
    constexpr int PV = VE / 2;
    constexpr int RB = RowShape<NV>::kFwdRows;
    __shared__ __align__(16) float red1[RB][32];
    __shared__ __align__(16) float red2[RB][32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int TPB = blockDim.x;
    const int nwarps = TPB >> 5;
    int ng = 1;
    while (ng < nwarps) ng <<= 1;
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t V = D / VE;
    const int64_t r0 = tile_begin(b, R, G), r1 = tile_begin(b + 1, R, G);
    const char* __restrict__ xb = static_cast<const char*>(x);
    const int64_t row_bytes = D * (int64_t)sizeof(T);
    const float invD = 1.0f / (float)D;
    zero_absent_warps<RB>(red1, nwarps);
    zero_absent_warps<RB>(red2, nwarps);
    uint32_t colb[NV];
    bool ok[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int64_t v = tid + (int64_t)k * TPB;
        ok[k] = v < V;
        colb[k] = (uint32_t)(v * 16);
    }
    __syncthreads();
    for (int64_t row = r0; row < r1; row += RB) {
        const int nr = (int)min((int64_t)RB, r1 - row);
        f2r d[RB][NV][PV];
        float K[RB], s1[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            const char* src = xb + (row + i) * row_bytes;
            K[i] = (i < nr && ADALN_IN_ROW(row + i, R, 0, 4, row_bytes)) ? IO::first(src) : 0.0f;
            const f2r kk = p_splat(K[i]);
            f2r acc0 = kPairZero, acc1 = kPairZero;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                IO::unpackp((i < nr && ok[k] && ADALN_IN_ROW(row + i, R, colb[k], 16, row_bytes))
                                ? ld_stream(src + colb[k])
                                : make_uint4(0, 0, 0, 0),
                            d[i][k]);
#pragma unroll
                for (int p = 0; p < PV; ++p) {
                    d[i][k][p] = p_sub(d[i][k][p], kk);
                    if (!ok[k]) d[i][k][p] = kPairZero;
                    if (p & 1) acc1 = p_add(acc1, d[i][k][p]);
                    else acc0 = p_add(acc0, d[i][k][p]);
                }
            }
            s1[i] = p_hsum(p_add(acc0, acc1));
        }
        warp_sum(s1);
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < RB; ++i) red1[i][warp] = s1[i];
        }
        __syncthreads();
        cta_sum(red1, ng, lane, s1);
        float s2[RB], md[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            md[i] = s1[i] * invD;
            const f2r pm = p_splat(md[i]);
            f2r acc0 = kPairZero, acc1 = kPairZero;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
#pragma unroll
                for (int p = 0; p < PV; ++p) {
                    d[i][k][p] = p_sub(d[i][k][p], pm);
                    if (!ok[k]) d[i][k][p] = kPairZero;
                    if (p & 1) acc1 = p_fma(d[i][k][p], d[i][k][p], acc1);
                    else acc0 = p_fma(d[i][k][p], d[i][k][p], acc0);
                }
            }
            s2[i] = p_hsum(p_add(acc0, acc1));
        }
        warp_sum(s2);
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < RB; ++i) red2[i][warp] = s2[i];
        }
        __syncthreads();
        cta_sum(red2, ng, lane, s2);
        if (tid == 0) {
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                if (i < nr && ADALN_IN(kDbgStats, row + i >= 0 && row + i < R)) {
                    mean[row + i] = K[i] + md[i];
                    rstd[row + i] = rsqrtf(s2[i] * invD + eps);
                }
            }
        }
    }
}

template <typename T>
static const void* pick_stats(int nv) {
    switch (nv) {
        case 1: return reinterpret_cast<const void*>(&stats_kernel<T, 1>);
        case 2: return reinterpret_cast<const void*>(&stats_kernel<T, 2>);
        case 3: return reinterpret_cast<const void*>(&stats_kernel<T, 3>);
        case 4: return reinterpret_cast<const void*>(&stats_kernel<T, 4>);
        case 6: return reinterpret_cast<const void*>(&stats_kernel<T, 6>);
        case 8: return reinterpret_cast<const void*>(&stats_kernel<T, 8>);
        default: return nullptr;
    }
}

cudaError_t debug_word_fwd(uint32_t* out, bool reset) { return debug_word(out, reset); }

cudaError_t launch_stats(const void* x, float* mean, float* rstd, int64_t R, int64_t D, float eps,
                         int dtype, int nv, int tpb, int64_t G, cudaStream_t stream) {
    const void* fn = dtype == 0 ? pick_stats<float>(nv) : dtype == 1 ? pick_stats<__nv_bfloat16>(nv) : nullptr;
    if (!fn || G < 1) return cudaErrorInvalidValue;
    void* params[] = {&x, &mean, &rstd, &R, &D, &eps};
    return launch_dependent(fn, dim3((unsigned)G), dim3((unsigned)tpb), params, 0, stream);
}

}  // namespace adaln
