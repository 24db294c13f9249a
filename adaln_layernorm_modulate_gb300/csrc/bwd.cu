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
//
// As in the forward, the ring variant has one thread copy whole rows of x and dy into a
// shared-memory ring with bulk (TMA) copies completing on per-slot mbarriers; the rows'
// saved mean/rstd are loaded one round ahead into registers; the elementwise math runs on
// fp32 pairs. Wide rows (6 or more vectors a thread) are read from the ring twice, once for
// the sums and accumulators and once for dx, instead of being held in registers.
#include "common.cuh"
#include "launch.h"

namespace adaln {

// WIDE: bf16 rows of four vectors a thread over more than max_threads(4, 8) threads (D of
// 14336 and 16384: 448 and 512 threads), which read x and dy from the ring twice so that only
// the column accumulators and (1 + scale) stay in registers (128 a thread at 512).
// SPLIT: fp32 rows too wide for a ring of two rounds (D > 14336). The grid is made of
// two-CTA clusters, a cluster per row tile; CTA r of a cluster stages and owns half r of
// every row (a ring of half rows), and the two CTAs add their row sums of g and g*xhat after
// exchanging them through distributed shared memory (the same bits in both).
template <typename T, int NV, bool VARLEN, bool RING, bool FULL, bool WIDE = false, bool SPLIT = false>
__global__ void __launch_bounds__(SPLIT ? kSplitThreads : WIDE ? kWideThreads : max_threads(NV, Io<T>::VE))
    bwd_kernel(const BwdArgs a) {
    pdl_begin();
    using IO = Io<T>;
    constexpr int VE = IO::VE;
    constexpr int PV = VE / 2;  // fp32 pairs per 16-byte vector
    constexpr int RB = RowShape<NV>::kRows;
    // Wide rows read x and dy from the ring twice instead of holding them in registers.
    constexpr bool REREAD = RING && (NV >= 6 || WIDE) && !SPLIT;
    static_assert(!REREAD || RB == 1, "wide rows are staged one a round");
    static_assert(!SPLIT || (RING && !WIDE), "the split form stages half rows in a ring");
    extern __shared__ uint4 ring[];
    __shared__ __align__(16) float red[2][2 * RB][32];  // double-buffered per-warp sums of g, g*xhat

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int TPB = blockDim.x;
    const int nwarps = TPB >> 5;
    int ng = 1;  // warps rounded up to a power of two
    while (ng < nwarps) ng <<= 1;
    // Row tiles: one per CTA, or per cluster in the split form (CTA `half` of it covering
    // vectors half * VC .. half * VC + VC - 1 of every row).
    const uint32_t half = SPLIT ? cluster_ctarank() : 0u;
    const int64_t G = SPLIT ? gridDim.x / 2 : gridDim.x, b = SPLIT ? blockIdx.x / 2 : blockIdx.x;
    const int64_t R = a.seg.R, D = a.D, V = D / VE;
    const int64_t VC = SPLIT ? V / 2 : V;
    const uint32_t copy_off = (uint32_t)((int64_t)half * VC * 16), copy_bytes = (uint32_t)(VC * 16);
    const int64_t r0 = tile_begin(b, R, G), r1 = tile_begin(b + 1, R, G);
    const char* __restrict__ xb = static_cast<const char*>(a.x);
    const char* __restrict__ gb = static_cast<const char*>(a.dy);
    char* __restrict__ dxb = static_cast<char*>(a.dx);
    const int64_t row_bytes = D * (int64_t)sizeof(T);
    const float invD = 1.0f / (float)D;
    const int ns = a.stages;

    // Ring layout (32-bit shared addresses): ns mbarriers (first 128 bytes), then [ns][RB]
    // row pairs (x, dy), each row at the offsets it has in global memory.
    __shared__ int abort_flag;
    // Split form: the peer CTA's row sums (double-buffered by round) and their mbarriers.
    __shared__ __align__(8) uint64_t xbar[2];
    __shared__ float xch[2][2 * RB];
    const uint32_t vk = (uint32_t)TPB * 16u;
    const uint32_t vrow = (uint32_t)NV * vk;           // one tensor's row slot
    const uint32_t vslot = (uint32_t)RB * 2u * vrow;   // one round: RB rows of x and dy
    const uint32_t bars = smem_addr(ring);
    const uint32_t data = bars + 128u;
    const uint32_t my_vec = data + (uint32_t)tid * 16u;

    zero_absent_warps<2 * RB>(red[0], nwarps);
    zero_absent_warps<2 * RB>(red[1], nwarps);
    uint32_t err = validate_segments<VARLEN>(a.seg, b, G);
    if constexpr (RING) {
        if (tid == 0) {
            for (int q = 0; q < ns; ++q) mbar_init(bars + 8u * q, 1);
            if constexpr (SPLIT) {
                mbar_init(smem_addr(&xbar[0]), 1);
                mbar_init(smem_addr(&xbar[1]), 1);
            }
            abort_flag = 0;
            mbar_fence_init();
        }
        // The split form: the peer's barriers are initialised before either CTA arrives on them.
        if constexpr (SPLIT)
            cluster_sync();
        else
            __syncthreads();
    }

    uint32_t colb[NV];
    bool ok[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int64_t v = tid + (int64_t)k * TPB;
        if constexpr (SPLIT) {
            ok[k] = FULL || v < VC;
            colb[k] = (uint32_t)(((int64_t)half * VC + v) * 16);
        } else {
            ok[k] = FULL || v < V;
            colb[k] = (uint32_t)(v * 16);
        }
    }

    const int64_t s0 = R > 0 ? seg_find<VARLEN>(a.seg, r0) : 0;
    Walker<VARLEN, RB> cw{r0, s0, -1, false};
    Walker<VARLEN, RB> pw{r0, s0, -1, false};  // producer's walker (thread 0), ns rounds ahead

    // Thread 0: copy the producer walker's next round (x and dy rows) into ring slot `slot`.
    auto issue = [&](int slot) {
        int64_t rs, sg;
        int nr;
        if (pw.next(a.seg, r1, rs, nr, sg)) {
            const uint32_t bar = bars + 8u * (uint32_t)slot;
            if constexpr (SPLIT)
                mbar_arrive_expect_tx(bar, (uint32_t)nr * 2u * copy_bytes);
            else
                mbar_arrive_expect_tx(bar, (uint32_t)(2 * nr * row_bytes));
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                if (i >= nr) continue;
                const uint32_t dst = data + (uint32_t)slot * vslot + (uint32_t)(2 * i) * vrow;
                if constexpr (SPLIT) {
                    const int64_t off = (rs + i) * row_bytes + copy_off;
                    if (ADALN_IN_ROW(rs + i, R, copy_off, copy_bytes, row_bytes) &&
                        ADALN_IN_RING(bars, dst, copy_bytes) && ADALN_IN_RING(bars, dst + vrow, copy_bytes)) {
                        bulk_load(dst, xb + off, copy_bytes, bar);
                        bulk_load(dst + vrow, gb + off, copy_bytes, bar);
                    }
                } else {
                    const int64_t off = (rs + i) * row_bytes;
                    if (ADALN_IN_ROW(rs + i, R, 0, row_bytes, row_bytes) && ADALN_IN_RING(bars, dst, row_bytes) &&
                        ADALN_IN_RING(bars, dst + vrow, row_bytes)) {
                        bulk_load(dst, xb + off, (uint32_t)row_bytes, bar);
                        bulk_load(dst + vrow, gb + off, (uint32_t)row_bytes, bar);
                    }
                }
            }
        }
    };
    if constexpr (RING) {
        if (tid == 0)
            for (int q = 0; q < ns; ++q) issue(q);
    }
    // The saved statistics of the next round's rows, loaded a round ahead (rounds are
    // consecutive rows of the tile).
    float mu_n[RB], rs_n[RB];
    auto load_stats = [&](int64_t first) {
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            const bool in = first + i < r1 && ADALN_IN(kDbgStats, first + i >= 0 && first + i < R);
            mu_n[i] = in ? __ldg(a.mean + first + i) : 0.0f;
            rs_n[i] = in ? __ldg(a.rstd + first + i) : 0.0f;
        }
    };
    if constexpr (RING) load_stats(r0);

    int slot = 0, buf = 0;
    uint32_t xr = 0;  // split form: row sums exchanged so far
    uint32_t lap = 0;  // completed passes over the ring: the parity of the slot's phase
    bool started = false;  // a previous round exists whose slot can be refilled
    int64_t cur_s = -1;
    bool cur_ok = false;
    f2r sc1[NV][PV];
    f2r acc_dy[NV][PV], acc_dyx[NV][PV];
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int p = 0; p < PV; ++p) acc_dy[k][p] = acc_dyx[k][p] = kPairZero;

    // Piece (tile b, segment cur_s) done: each thread writes its vectors' column sums into
    // slot b + cur_s, in the layout the launch chose (see BwdArgs).
    const int64_t S = G + a.seg.nseg;
    auto flush = [&]() {
        const int64_t slot = b + cur_s;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (ok[k] && ADALN_IN(kDbgPartials, slot >= 0 && slot < S && (int64_t)colb[k] / 16 < V)) {
                const int64_t v = colb[k] / 16;  // my vector k
                float* p0 = a.vec_major ? a.partials + ((v * 2 + 0) * S + slot) * VE
                                        : a.partials + slot * 2 * D + v * VE;
                float* p1 = a.vec_major ? a.partials + ((v * 2 + 1) * S + slot) * VE : p0 + D;
#pragma unroll
                for (int p = 0; p < PV; p += 2) {
                    const float2 a0 = p_get(acc_dy[k][p]), a1 = p_get(acc_dy[k][p + 1]);
                    const float2 b0 = p_get(acc_dyx[k][p]), b1 = p_get(acc_dyx[k][p + 1]);
                    *reinterpret_cast<float4*>(p0 + 2 * p) = make_float4(a0.x, a0.y, a1.x, a1.y);
                    *reinterpret_cast<float4*>(p1 + 2 * p) = make_float4(b0.x, b0.y, b1.x, b1.y);
                }
            }
#pragma unroll
            for (int p = 0; p < PV; ++p) acc_dy[k][p] = acc_dyx[k][p] = kPairZero;
        }
    };

    int64_t row, s;
    int nr;
    while (cw.next(a.seg, r1, row, nr, s)) {
        uint4 xv[RB][NV], gv[RB][NV];
        float mu[RB], rs[RB];
        if constexpr (RING) {
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                mu[i] = mu_n[i];
                rs[i] = rs_n[i];
            }
            load_stats(cw.row);
            // The previous round's slot has been read by every thread (they all passed that
            // round's barriers): refill it ns rounds ahead before waiting on this one.
            if (tid == 0 && started) issue(slot == 0 ? ns - 1 : slot - 1);
            started = true;
            if (!mbar_wait_bounded(bars + 8u * (uint32_t)slot, lap & 1u, &abort_flag)) err |= kErrTimeout;
            if constexpr (!REREAD) {
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                    const uint32_t xs = my_vec + (uint32_t)slot * vslot + (uint32_t)(2 * i) * vrow;
#pragma unroll
                    for (int k = 0; k < NV; ++k) {
                        const bool on = i < nr && ok[k] && ADALN_IN_RING(bars, xs + (uint32_t)k * vk, 16) &&
                                        ADALN_IN_RING(bars, xs + vrow + (uint32_t)k * vk, 16);
                        xv[i][k] = on ? lds128(xs + (uint32_t)k * vk) : make_uint4(0, 0, 0, 0);
                        gv[i][k] = on ? lds128(xs + vrow + (uint32_t)k * vk) : make_uint4(0, 0, 0, 0);
                    }
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const int64_t off = (row + i) * row_bytes;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const bool on = i < nr && ok[k] && ADALN_IN_ROW(row + i, R, colb[k], 16, row_bytes);
                    xv[i][k] = on ? ld_stream(xb + off + colb[k]) : make_uint4(0, 0, 0, 0);
                    gv[i][k] = on ? ld_stream(gb + off + colb[k]) : make_uint4(0, 0, 0, 0);
                }
                const bool in = i < nr && ADALN_IN(kDbgStats, row + i >= 0 && row + i < R);
                mu[i] = in ? __ldg(a.mean + row + i) : 0.0f;
                rs[i] = in ? __ldg(a.rstd + row + i) : 0.0f;
            }
        }

        if (s != cur_s) {
            if (cur_ok) flush();
            cur_s = s;
            const int64_t m = seg_mod<VARLEN>(a.seg, s);
            cur_ok = m >= 0 && m < a.seg.nmod;
            if (!cur_ok) err |= kErrModIdx;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                uint4 vc = make_uint4(0, 0, 0, 0);
                if (cur_ok && ok[k] && ADALN_IN(kDbgMod, m >= 0 && m < a.seg.nmod && colb[k] + 16 <= row_bytes))
                    vc = ld_keep(static_cast<const char*>(a.scale) + m * row_bytes + colb[k]);
                IO::unpackp(vc, sc1[k]);
                const f2r one = p_splat(1.0f);
#pragma unroll
                for (int p = 0; p < PV; ++p) sc1[k][p] = p_add(sc1[k][p], one);
            }
        }

        if (REREAD && cur_ok) {
            // Wide rows (RB = 1): x and dy stay in the ring slot. Pass 1 reads them for the row
            // sums and the column accumulators, pass 2 reads them again for dx, so only the
            // accumulators and (1 + scale) stay in registers across the row.
            const uint32_t xs = my_vec + (uint32_t)slot * vslot;
            const f2r rs2 = p_splat(rs[0]), mu2 = p_splat(mu[0]);
            f2r sg[2] = {kPairZero, kPairZero}, sgx[2] = {kPairZero, kPairZero};
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const bool on = ok[k] && ADALN_IN_RING(bars, xs + (uint32_t)k * vk, 16) &&
                                ADALN_IN_RING(bars, xs + vrow + (uint32_t)k * vk, 16);
                const uint4 xq = on ? lds128(xs + (uint32_t)k * vk) : make_uint4(0, 0, 0, 0);
                const uint4 gq = on ? lds128(xs + vrow + (uint32_t)k * vk) : make_uint4(0, 0, 0, 0);
                f2r xh[PV], fd[PV];
                IO::unpackp(xq, xh);
                IO::unpackp(gq, fd);
#pragma unroll
                for (int p = 0; p < PV; ++p) {
                    xh[p] = p_mul(p_sub(xh[p], mu2), rs2);
                    const f2r g = p_mul(fd[p], sc1[k][p]);
                    sg[p & 1] = p_add(sg[p & 1], g);
                    sgx[p & 1] = p_fma(g, xh[p], sgx[p & 1]);
                    acc_dy[k][p] = p_add(acc_dy[k][p], fd[p]);
                    acc_dyx[k][p] = p_fma(fd[p], xh[p], acc_dyx[k][p]);
                }
            }
            float sums[2] = {p_hsum(p_add(sg[0], sg[1])), p_hsum(p_add(sgx[0], sgx[1]))};
            warp_sum(sums);
            if (lane == 0) {
                red[buf][0][warp] = sums[0];
                red[buf][1][warp] = sums[1];
            }
            __syncthreads();
            cta_sum(red[buf], ng, lane, sums);
            const float mg = sums[0] * invD, mgx = sums[1] * invD;
            const f2r nmgx = p_splat(-mgx), nmgr = p_splat(-mg * rs[0]);
            char* dxr = dxb + row * row_bytes;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                if (!ok[k] || !ADALN_IN_RING(bars, xs + (uint32_t)k * vk, 16) ||
                    !ADALN_IN_RING(bars, xs + vrow + (uint32_t)k * vk, 16))
                    continue;
                f2r xh[PV], fd[PV], o[PV];
                IO::unpackp(lds128(xs + (uint32_t)k * vk), xh);
                IO::unpackp(lds128(xs + vrow + (uint32_t)k * vk), fd);
#pragma unroll
                for (int p = 0; p < PV; ++p) {
                    xh[p] = p_mul(p_sub(xh[p], mu2), rs2);
                    o[p] = p_fma(p_fma(xh[p], nmgx, p_mul(fd[p], sc1[k][p])), rs2, nmgr);
                }
                if (ADALN_IN_ROW(row, R, colb[k], 16, row_bytes)) st_vec(dxr + colb[k], IO::packp(o));
            }
            buf ^= 1;
        } else if (cur_ok) {  // uniform across the CTA
            // xhat = (x - mean) * rstd, g = dy * (1 + scale); row sums of g and g*xhat;
            // column sums of dy and dy*xhat. Rows past nr and idle lanes load dy = 0, so they
            // add nothing anywhere.
            f2r xh[RB][NV][PV], g[RB][NV][PV];
            float sums[2 * RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const f2r rs2 = p_splat(rs[i]), mu2 = p_splat(mu[i]);
                f2r sg[2] = {kPairZero, kPairZero}, sgx[2] = {kPairZero, kPairZero};
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    f2r fd[PV];
                    IO::unpackp(xv[i][k], xh[i][k]);
                    IO::unpackp(gv[i][k], fd);
#pragma unroll
                    for (int p = 0; p < PV; ++p) {
                        // x - mean first: exact for rows whose mean dwarfs their spread.
                        xh[i][k][p] = p_mul(p_sub(xh[i][k][p], mu2), rs2);
                        g[i][k][p] = p_mul(fd[p], sc1[k][p]);
                        sg[p & 1] = p_add(sg[p & 1], g[i][k][p]);
                        sgx[p & 1] = p_fma(g[i][k][p], xh[i][k][p], sgx[p & 1]);
                        acc_dy[k][p] = p_add(acc_dy[k][p], fd[p]);
                        acc_dyx[k][p] = p_fma(fd[p], xh[i][k][p], acc_dyx[k][p]);
                    }
                }
                sums[2 * i] = p_hsum(p_add(sg[0], sg[1]));
                sums[2 * i + 1] = p_hsum(p_add(sgx[0], sgx[1]));
            }
            warp_sum(sums);
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < 2 * RB; ++i) red[buf][i][warp] = sums[i];
            }
            __syncthreads();
            cta_sum(red[buf], ng, lane, sums);
            if constexpr (SPLIT) {
                // Send this half's sums to the other CTA, take its sums, add them in CTA order
                // (so both CTAs hold the same bits). A round's buffer is written again two
                // rounds later, after its reader has sent the round in between.
                const uint32_t par = xr & 1u;
                if (tid == 0) {
                    const uint32_t dst = cluster_map(smem_addr(&xch[par][0]), half ^ 1u);
#pragma unroll
                    for (int i = 0; i < 2 * RB; ++i) st_cluster_f32(dst + 4u * (uint32_t)i, sums[i]);
                    mbar_arrive_remote(cluster_map(smem_addr(&xbar[par]), half ^ 1u));
                }
                if (!mbar_wait_cluster_bounded(smem_addr(&xbar[par]), (xr >> 1) & 1u, &abort_flag))
                    err |= kErrTimeout;
                const volatile float* peer = xch[par];
#pragma unroll
                for (int i = 0; i < 2 * RB; ++i) {
                    const float o = peer[i];
                    sums[i] = half == 0 ? sums[i] + o : o + sums[i];
                }
                ++xr;
            }
            // dx = rstd * (g - mean(g) - xhat * mean(g*xhat))
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                if (i >= nr) continue;
                const float mg = sums[2 * i] * invD, mgx = sums[2 * i + 1] * invD;
                const f2r rs2 = p_splat(rs[i]), nmgx = p_splat(-mgx), nmgr = p_splat(-mg * rs[i]);
                char* dxr = dxb + (row + i) * row_bytes;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    if (!ok[k]) continue;
                    f2r o[PV];
#pragma unroll
                    for (int p = 0; p < PV; ++p) o[p] = p_fma(p_fma(xh[i][k][p], nmgx, g[i][k][p]), rs2, nmgr);
                    if (ADALN_IN_ROW(row + i, R, colb[k], 16, row_bytes)) st_vec(dxr + colb[k], IO::packp(o));
                }
            }
            buf ^= 1;
        }
        if constexpr (RING) {
            // A skipped round, and a wide row read again after its barrier, still fence the
            // slot's readers before the slot is refilled.
            if (REREAD || !cur_ok) __syncthreads();
            if (++slot == ns) {
                slot = 0;
                ++lap;
            }
        }
    }
    if (cur_ok) flush();
    if (cw.bad) err |= kErrSeqlens;
    if constexpr (RING) {
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
    // The split form: neither CTA leaves while the other may still write into its memory.
    if constexpr (SPLIT) cluster_sync();
}

// Stage 2: dshift[m] / dscale[m] = sum of the partials of every piece of every segment
// whose modulation row is m, in a fixed order. The pieces of m form a flat list in segment
// order (piece = tile b of segment s, partial slot b + s). CTA (blockIdx.x, m) covers `cw`
// float4 columns; its 256 threads form cw columns x (256 / cw) splits, piece j going to
// split j mod splits; each split adds its pieces in list order (kStage2Unroll loads in
// flight at a time), and a fixed shared-memory tree combines the splits.
//
// Packed batches find m's segments by compacting the segment table a chunk at a time:
// every thread tests kStage2Per consecutive entries, and one block-wide scan places the
// hits, in order, with the flat index of their first piece.
constexpr int kStage2Per = 4;
constexpr int kStage2Chunk = kStage2Threads * kStage2Per;
constexpr int kStage2Unroll = 4;

// Compacts entries [base, base + kStage2Chunk) of the segment table whose modulation row is m
// into hit_slot (partial slot of the hit's first piece) and hit_first (flat index of that
// piece among the hits'), in table order: H hits, NP pieces, hit_first[H] = NP. Every thread
// of a kStage2Threads-thread CTA calls it; it ends with a barrier.
__device__ __forceinline__ void compact_hits(const Segments& sg, int64_t m, int64_t base, int64_t R, int64_t G,
                                             uint32_t* hit_slot, int32_t* hit_first,
                                             int32_t (*warp_tot)[kStage2Threads / 32], int& H, int& NP) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // This thread's entries: segments s0 .. s0 + kStage2Per - 1 of the chunk.
    const int64_t s0 = base + (int64_t)tid * kStage2Per;
    int32_t np[kStage2Per];
    uint32_t sl[kStage2Per];
    int hc = 0, pc = 0;
#pragma unroll
    for (int i = 0; i < kStage2Per; ++i) {
        const int64_t s = s0 + i;
        np[i] = 0;
        sl[i] = 0;
        if (s < sg.nseg && ADALN_IN(kDbgSegments, s >= 0) && (int64_t)__ldg(sg.mod + s) == m) {
            // Clamp into [0, R] so a malformed table cannot index past the slots.
            const int64_t lo = max((int64_t)0, min(seg_start<true>(sg, s), R));
            const int64_t hi = max((int64_t)0, min(seg_start<true>(sg, s + 1), R));
            if (hi > lo) {
                const int64_t blo = tile_of_row(lo, R, G), bhi = tile_of_row(hi - 1, R, G);
                np[i] = (int32_t)(bhi - blo + 1);
                sl[i] = (uint32_t)(blo + s);
                ++hc;
                pc += np[i];
            }
        }
    }
    // Block-wide exclusive scan of (hits, pieces) in thread order = table order.
    int ih = hc, ip = pc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int th = __shfl_up_sync(0xFFFFFFFFu, ih, o);
        const int tp = __shfl_up_sync(0xFFFFFFFFu, ip, o);
        if (lane >= o) {
            ih += th;
            ip += tp;
        }
    }
    if (lane == 31) {
        warp_tot[0][warp] = ih;
        warp_tot[1][warp] = ip;
    }
    __syncthreads();
    int oh = ih - hc, op = ip - pc;
    H = 0;
    NP = 0;
#pragma unroll
    for (int w = 0; w < kStage2Threads / 32; ++w) {
        const int th = warp_tot[0][w], tp = warp_tot[1][w];
        if (w < warp) {
            oh += th;
            op += tp;
        }
        H += th;
        NP += tp;
    }
#pragma unroll
    for (int i = 0; i < kStage2Per; ++i) {
        if (np[i] > 0 && ADALN_IN(kDbgShared, oh >= 0 && oh < kStage2Chunk)) {
            hit_slot[oh] = sl[i];
            hit_first[oh] = op;
            ++oh;
            op += np[i];
        }
    }
    if (tid == 0 && ADALN_IN(kDbgShared, H >= 0 && H <= kStage2Chunk)) hit_first[H] = NP;
    __syncthreads();
}

// The hit holding piece q of a compacted list: the last h with hit_first[h] <= q; returns
// the piece's partial slot.
__device__ __forceinline__ int64_t hit_slot_of(int64_t q, int H, const uint32_t* hit_slot,
                                               const int32_t* hit_first) {
    int lo = 0, hi = H - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)hit_first[mid] <= q) lo = mid;
        else hi = mid - 1;
    }
    return (int64_t)hit_slot[lo] + (q - (int64_t)hit_first[lo]);
}

// Stage 2 over vector-major partials (modulation rows with many pieces). CTA (blockIdx.x, m)
// covers nvb = kStage2Threads / splits consecutive 16-byte vectors of columns; `splits`
// consecutive threads share one vector, piece j going to thread j mod splits, which adds its
// pieces in list order. A vector's pieces sit side by side, so the threads of a vector read
// consecutive 32-byte (bf16) or 16-byte (fp32) chunks. The threads' sums are then combined
// by a fixed tree: shuffles within a warp, then the vector's warps in warp order.
template <int VE, bool VARLEN>
__global__ void __launch_bounds__(kStage2Threads) stage2v_kernel(const Stage2Args a) {
    pdl_begin();
    constexpr int Q = VE / 4;  // float4 per vector
    constexpr int NW = kStage2Threads / 32;
    __shared__ float red[NW][2 * VE];
    __shared__ uint32_t hit_slot[kStage2Chunk];
    __shared__ int32_t hit_first[kStage2Chunk + 1];
    __shared__ int32_t warp_tot[2][NW];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int splits = a.splits, nvb = kStage2Threads / splits;
    const int k = tid % splits, vj = tid / splits;
    const int64_t V = a.D / VE, S = a.S;
    const int64_t v = (int64_t)blockIdx.x * nvb + vj;
    const bool vok = v < V;
    const int64_t R = a.seg.R, G = a.G;
    const float4* P0 = reinterpret_cast<const float4*>(a.partials) + (v * 2 + 0) * S * Q;
    const float4* P1 = reinterpret_cast<const float4*>(a.partials) + (v * 2 + 1) * S * Q;

    for (int64_t m = blockIdx.y; m < a.seg.nmod; m += gridDim.y) {
        float acc[2 * VE];
#pragma unroll
        for (int e = 0; e < 2 * VE; ++e) acc[e] = 0.0f;
        int64_t J = 0;  // pieces of row m before the current list

        auto sum_pieces = [&](int64_t n, auto slot_of) {
            if (vok) {
                int64_t q0 = ((int64_t)k - J) % splits;
                if (q0 < 0) q0 += splits;
                for (; q0 < n; q0 += (int64_t)kStage2Unroll * splits) {
                    float4 u[kStage2Unroll][Q], w[kStage2Unroll][Q];
#pragma unroll
                    for (int i = 0; i < kStage2Unroll; ++i) {
                        const int64_t q = q0 + (int64_t)i * splits;
                        if (q < n) {
                            const int64_t slot = slot_of(q);
                            if (ADALN_IN(kDbgPartials, slot >= 0 && slot < S)) {
#pragma unroll
                                for (int j = 0; j < Q; ++j) {
                                    u[i][j] = __ldg(P0 + slot * Q + j);
                                    w[i][j] = __ldg(P1 + slot * Q + j);
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < Q; ++j) u[i][j] = w[i][j] = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kStage2Unroll; ++i) {
                        if (q0 + (int64_t)i * splits < n) {
#pragma unroll
                            for (int j = 0; j < Q; ++j) {
                                acc[4 * j + 0] += u[i][j].x; acc[4 * j + 1] += u[i][j].y;
                                acc[4 * j + 2] += u[i][j].z; acc[4 * j + 3] += u[i][j].w;
                                acc[VE + 4 * j + 0] += w[i][j].x; acc[VE + 4 * j + 1] += w[i][j].y;
                                acc[VE + 4 * j + 2] += w[i][j].z; acc[VE + 4 * j + 3] += w[i][j].w;
                            }
                        }
                    }
                }
            }
            J += n;
        };

        if constexpr (!VARLEN) {
            const int64_t lo = min(m * a.seg.N, R), hi = min((m + 1) * a.seg.N, R);
            if (hi > lo) {
                const int64_t blo = tile_of_row(lo, R, G), bhi = tile_of_row(hi - 1, R, G);
                sum_pieces(bhi - blo + 1, [&](int64_t q) { return blo + q + m; });
            }
        } else {
            for (int64_t base = 0; base < a.seg.nseg; base += kStage2Chunk) {
                int H = 0, NP = 0;
                compact_hits(a.seg, m, base, R, G, hit_slot, hit_first, warp_tot, H, NP);
                if (H > 0) sum_pieces(NP, [&](int64_t q) { return hit_slot_of(q, H, hit_slot, hit_first); });
                __syncthreads();  // the next chunk reuses the hit lists and warp totals
            }
        }

        if (splits <= 32) {
            // The vector's threads are `splits` consecutive lanes of one warp.
            for (int o = 1; o < splits; o <<= 1) {
#pragma unroll
                for (int e = 0; e < 2 * VE; ++e) acc[e] += __shfl_xor_sync(0xFFFFFFFFu, acc[e], o);
            }
            if (k == 0 && vok && ADALN_IN(kDbgGrads, m >= 0 && m < a.seg.nmod && v >= 0 && v < V)) {
                float4* o0 = reinterpret_cast<float4*>(a.dshift + m * a.D + v * VE);
                float4* o1 = reinterpret_cast<float4*>(a.dscale + m * a.D + v * VE);
#pragma unroll
                for (int j = 0; j < Q; ++j) {
                    o0[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
                    o1[j] = make_float4(acc[VE + 4 * j], acc[VE + 4 * j + 1], acc[VE + 4 * j + 2],
                                        acc[VE + 4 * j + 3]);
                }
            }
        } else {
            // The vector's threads fill splits / 32 whole warps: a butterfly in each warp,
            // then the warps' sums in warp order.
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                for (int e = 0; e < 2 * VE; ++e) acc[e] += __shfl_xor_sync(0xFFFFFFFFu, acc[e], o);
            }
            if (lane == 0) {
#pragma unroll
                for (int e = 0; e < 2 * VE; ++e) red[warp][e] = acc[e];
            }
            __syncthreads();
            const int wpv = splits / 32;
            if (tid < nvb * 2 * VE) {
                const int vv = tid / (2 * VE), e = tid % (2 * VE);
                const int64_t vg = (int64_t)blockIdx.x * nvb + vv;
                if (vg < V && ADALN_IN(kDbgGrads, m >= 0 && m < a.seg.nmod && vg >= 0) &&
                    ADALN_IN(kDbgShared, vv * wpv + wpv <= NW)) {
                    float t = red[vv * wpv][e];
                    for (int w2 = 1; w2 < wpv; ++w2) t += red[vv * wpv + w2][e];
                    float* out = e < VE ? a.dshift : a.dscale;
                    out[m * a.D + vg * VE + (e % VE)] = t;
                }
            }
        }
        __syncthreads();  // the next row reuses the shared lists and sums
    }
}

template <bool VARLEN>
__global__ void __launch_bounds__(kStage2Threads, 4) stage2_kernel(const Stage2Args a) {
    pdl_begin();
    __shared__ float4 red[2][kStage2Threads];
    __shared__ uint32_t hit_slot[kStage2Chunk];       // partial slot of the hit's first piece
    __shared__ int32_t hit_first[kStage2Chunk + 1];   // flat index of the hit's first piece
    __shared__ int32_t warp_tot[2][kStage2Threads / 32];

    const int tid = threadIdx.x;
    const int cw = a.cw, splits = kStage2Threads / cw;
    const int ci = tid % cw, k = tid / cw;
    const int64_t D4 = a.D / 4;
    const int64_t c4 = (int64_t)blockIdx.x * cw + ci;
    const bool cok = c4 < D4;
    const int64_t R = a.seg.R, G = a.G;
    const float4* P = reinterpret_cast<const float4*>(a.partials) + c4;

    for (int64_t my = blockIdx.y; my < a.seg.nmod; my += gridDim.y) {
        // Modulation rows last to first: in a batch of ascending segment lengths the rows
        // with the most pieces come last, and this way their CTAs start in the first wave
        // (the packed D=3072 workload: 26.7 -> 19 us).
        const int64_t m = a.seg.nmod - 1 - my;
        float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
        int64_t J = 0;  // pieces of row m before the current list

        // Add this thread's share of pieces [0, n) of the current list (global index J + q),
        // piece q sitting in partial slot slot_of(q).
        auto sum_pieces = [&](int64_t n, auto slot_of) {
            if (cok) {
                for (int64_t q0 = (int64_t)((k - J) & (int64_t)(splits - 1)); q0 < n;
                     q0 += (int64_t)kStage2Unroll * splits) {
                    float4 u[kStage2Unroll], v[kStage2Unroll];
#pragma unroll
                    for (int i = 0; i < kStage2Unroll; ++i) {
                        const int64_t q = q0 + (int64_t)i * splits;
                        if (q < n) {
                            const int64_t slot = slot_of(q);
                            if (ADALN_IN(kDbgPartials, slot >= 0 && slot < a.S)) {
                                u[i] = __ldg(P + (slot * 2 + 0) * D4);
                                v[i] = __ldg(P + (slot * 2 + 1) * D4);
                            } else {
                                u[i] = v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kStage2Unroll; ++i) {
                        if (q0 + (int64_t)i * splits < n) {
                            acc0.x += u[i].x; acc0.y += u[i].y; acc0.z += u[i].z; acc0.w += u[i].w;
                            acc1.x += v[i].x; acc1.y += v[i].y; acc1.z += v[i].z; acc1.w += v[i].w;
                        }
                    }
                }
            }
            J += n;
        };

        if constexpr (!VARLEN) {
            const int64_t lo = min(m * a.seg.N, R), hi = min((m + 1) * a.seg.N, R);
            if (hi > lo) {
                const int64_t blo = tile_of_row(lo, R, G), bhi = tile_of_row(hi - 1, R, G);
                sum_pieces(bhi - blo + 1, [&](int64_t q) { return blo + q + m; });
            }
        } else {
            for (int64_t base = 0; base < a.seg.nseg; base += kStage2Chunk) {
                int H = 0, NP = 0;
                compact_hits(a.seg, m, base, R, G, hit_slot, hit_first, warp_tot, H, NP);
                if (H > 0) sum_pieces(NP, [&](int64_t q) { return hit_slot_of(q, H, hit_slot, hit_first); });
                __syncthreads();  // the next chunk reuses the hit lists and warp totals
            }
        }

        red[0][tid] = acc0;
        red[1][tid] = acc1;
        __syncthreads();
        for (int st = splits / 2; st >= 1; st >>= 1) {
            if (k < st && ADALN_IN(kDbgShared, tid + st * cw < kStage2Threads)) {
                const float4 u = red[0][tid + st * cw], v = red[1][tid + st * cw];
                float4& p = red[0][tid];
                float4& q = red[1][tid];
                p.x += u.x; p.y += u.y; p.z += u.z; p.w += u.w;
                q.x += v.x; q.y += v.y; q.z += v.z; q.w += v.w;
            }
            __syncthreads();
        }
        if (k == 0 && cok && ADALN_IN(kDbgGrads, m >= 0 && m < a.seg.nmod && c4 >= 0)) {
            reinterpret_cast<float4*>(a.dshift)[m * D4 + c4] = red[0][tid];
            reinterpret_cast<float4*>(a.dscale)[m * D4 + c4] = red[1][tid];
        }
        __syncthreads();
    }
}

template <typename T, int NV, bool VARLEN, bool RING, bool FULL, bool WIDE = false, bool SPLIT = false>
static const void* bwd_fn() {
    return reinterpret_cast<const void*>(&bwd_kernel<T, NV, VARLEN, RING, FULL, WIDE, SPLIT>);
}

// The split form: fp32, eight vectors a thread, a ring of half rows.
static const void* pick_split(bool varlen, bool full) {
    if (varlen)
        return full ? bwd_fn<float, 8, true, true, true, false, true>()
                    : bwd_fn<float, 8, true, true, false, false, true>();
    return full ? bwd_fn<float, 8, false, true, true, false, true>()
                : bwd_fn<float, 8, false, true, false, false, true>();
}

cudaError_t bwd_split_clusters(bool varlen, bool full, int tpb, size_t smem, int* out) {
    const void* fn = pick_split(varlen, full);
    cudaError_t e = allow_dynamic_smem(fn);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3((unsigned)tpb);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, fn, &cfg);
}

// Instantiated variants: ring + full row, ring + partial row, plain (partial row).
template <typename T, int NV, bool VARLEN>
static const void* pick_variant(bool ring, bool full) {
    if (ring) return full ? bwd_fn<T, NV, VARLEN, true, true>() : bwd_fn<T, NV, VARLEN, true, false>();
    return bwd_fn<T, NV, VARLEN, false, false>();
}

template <typename T, bool VARLEN>
static const void* pick_nv(int nv, bool ring, bool full) {
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

static const void* pick_bwd(int dtype, int nv, bool varlen, bool ring, bool full, int tpb) {
    if (dtype == 1 && nv == 4 && tpb > max_threads(4, 8)) {  // the wide form: ring, full rows
        if (!ring || !full || tpb > kWideThreads) return nullptr;
        return varlen ? bwd_fn<__nv_bfloat16, 4, true, true, true, true>()
                      : bwd_fn<__nv_bfloat16, 4, false, true, true, true>();
    }
    if (dtype == 0) return varlen ? pick_nv<float, true>(nv, ring, full) : pick_nv<float, false>(nv, ring, full);
    if (dtype == 1)
        return varlen ? pick_nv<__nv_bfloat16, true>(nv, ring, full)
                      : pick_nv<__nv_bfloat16, false>(nv, ring, full);
    return nullptr;
}

cudaError_t bwd_blocks_per_sm(int dtype, int nv, bool varlen, bool ring, bool full, int tpb,
                              size_t smem, int* out) {
    const void* fn = pick_bwd(dtype, nv, varlen, ring, full, tpb);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = allow_dynamic_smem(fn);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, fn, tpb, smem);
}

cudaError_t launch_bwd(const BwdArgs& args, int dtype, int nv, bool varlen, bool ring, bool full,
                       int64_t G, int tpb, size_t smem, bool split, cudaStream_t stream) {
    if (split && (dtype != 0 || nv != 8 || !ring || G % 2 != 0 || tpb > kSplitThreads))
        return cudaErrorInvalidValue;
    const void* fn = split ? pick_split(varlen, full) : pick_bwd(dtype, nv, varlen, ring, full, tpb);
    if (!fn) return cudaErrorInvalidValue;
    BwdArgs a = args;
    void* params[] = {&a};
    return launch_dependent(fn, dim3((unsigned)G), dim3((unsigned)tpb), params, smem, stream, split ? 2u : 1u);
}

cudaError_t debug_word_bwd(uint32_t* out, bool reset) { return debug_word(out, reset); }

cudaError_t launch_stage2(const Stage2Args& args, int dtype, bool varlen, int sms, cudaStream_t stream) {
    dim3 grid;
    const void* fn;
    const unsigned gy = (unsigned)(args.seg.nmod < 65535 ? args.seg.nmod : 65535);
    if (args.vec_major) {
        const int VE = dtype == 1 ? 8 : 4;
        const int64_t nvb = kStage2Threads / args.splits;
        grid = dim3((unsigned)((args.D / VE + nvb - 1) / nvb), gy);
        fn = dtype == 1 ? (varlen ? reinterpret_cast<const void*>(&stage2v_kernel<8, true>)
                                  : reinterpret_cast<const void*>(&stage2v_kernel<8, false>))
                        : (varlen ? reinterpret_cast<const void*>(&stage2v_kernel<4, true>)
                                  : reinterpret_cast<const void*>(&stage2v_kernel<4, false>));
    } else {
        grid = dim3((unsigned)((args.D / 4 + args.cw - 1) / args.cw), gy);
        fn = varlen ? reinterpret_cast<const void*>(&stage2_kernel<true>)
                    : reinterpret_cast<const void*>(&stage2_kernel<false>);
    }
    Stage2Args a = args;
    void* params[] = {&a};
    // A stage 2 of one wave starts as a dependent of the backward (its CTAs take the SMs the
    // backward's CTAs leave, then wait for it to complete): bf16 D=1536 on 32,760 rows with
    // vector-major partials, 97.6 -> 94.8 us a step. One of several waves measured slower that
    // way (the packed D=3072 workload: 2506 -> 2544 us a step), so it waits in the stream.
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kStage2Threads, 0);
    if (e != cudaSuccess) return e;
    if ((int64_t)grid.x * grid.y <= (int64_t)per_sm * sms)
        return launch_dependent(fn, grid, dim3(kStage2Threads), params, 0, stream);
    return cudaLaunchKernel(fn, grid, dim3(kStage2Threads), params, 0, stream);
}

}  // namespace adaln

namespace adaln {

// Sum over ranks of stacked per-rank gradients: out[i] = parts[0][i] + parts[1][i] + ...,
// always in rank order, so the result depends only on the inputs' bits, not on how they
// were gathered. 16-byte vectors where n allows, a grid-stride loop.
__global__ void __launch_bounds__(256) rank_sum_kernel(const float* __restrict__ parts, float* __restrict__ out,
                                                       int32_t world, int64_t n) {
    pdl_begin();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (n % 4 == 0) {
        const int64_t n4 = n / 4;
        const float4* p4 = reinterpret_cast<const float4*>(parts);
        float4* o4 = reinterpret_cast<float4*>(out);
        for (int64_t i = first; i < n4; i += stride) {
            if (!ADALN_IN(kDbgRanks, i >= 0 && world >= 1)) continue;
            float4 s = __ldg(p4 + i);
            for (int32_t r = 1; r < world; ++r) {
                const float4 v = __ldg(p4 + (int64_t)r * n4 + i);
                s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
            }
            o4[i] = s;
        }
    } else {
        for (int64_t i = first; i < n; i += stride) {
            if (!ADALN_IN(kDbgRanks, i >= 0 && world >= 1)) continue;
            float s = __ldg(parts + i);
            for (int32_t r = 1; r < world; ++r) s += __ldg(parts + (int64_t)r * n + i);
            out[i] = s;
        }
    }
}

cudaError_t launch_rank_sum(const float* parts, float* out, int32_t world, int64_t n, int sms,
                            cudaStream_t stream) {
    const int64_t units = n % 4 == 0 ? n / 4 : n;
    int64_t blocks = (units + 255) / 256;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    if (blocks < 1) blocks = 1;
    void* params[] = {&parts, &out, &world, &n};
    return launch_dependent(reinterpret_cast<const void*>(&rank_sum_kernel), dim3((unsigned)blocks), dim3(256),
                            params, 0, stream);
}

}  // namespace adaln
