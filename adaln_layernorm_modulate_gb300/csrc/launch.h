// Host-side entry points of the kernel translation units (internal to libadaln).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace adaln {

// Forward `ring`: kRingNone, kRingBulk or kRingCopy; backward `ring`: the bulk ring or
// none. `full`: the CTA covers the row exactly (ring variants only); `smem`: the ring's
// dynamic shared memory bytes.
cudaError_t fwd_blocks_per_sm(int dtype, int nv, bool varlen, int ring, bool full, int tpb,
                              size_t smem, int* out);
cudaError_t launch_fwd(const FwdArgs& args, int dtype, int nv, bool varlen, int ring, bool full,
                       int64_t G, int tpb, size_t smem, cudaStream_t stream);

// Row statistics alone (mean, rstd of R rows of x), with the forward's mapping (nv, tpb)
// and arithmetic; G CTAs, plain loads.
cudaError_t launch_stats(const void* x, float* mean, float* rstd, int64_t R, int64_t D, float eps,
                         int dtype, int nv, int tpb, int64_t G, cudaStream_t stream);

cudaError_t bwd_blocks_per_sm(int dtype, int nv, bool varlen, bool ring, bool full, int tpb,
                              size_t smem, int* out);
// split: the fp32 split form (G CTAs in clusters of two, G / 2 row tiles).
cudaError_t launch_bwd(const BwdArgs& args, int dtype, int nv, bool varlen, bool ring, bool full,
                       int64_t G, int tpb, size_t smem, bool split, cudaStream_t stream);
// Debug builds: the debug word of the forward's and the backward's module (0 in release
// builds), cleared after the read when `reset`.
cudaError_t debug_word_fwd(uint32_t* out, bool reset);
cudaError_t debug_word_bwd(uint32_t* out, bool reset);
// Resident two-CTA clusters of the split form on the current device.
cudaError_t bwd_split_clusters(bool varlen, bool full, int tpb, size_t smem, int* out);
// Stage 2 of a backward on a device of `sms` multiprocessors.
cudaError_t launch_stage2(const Stage2Args& args, int dtype, bool varlen, int sms, cudaStream_t stream);

// out[i] = sum over r in rank order of parts[r * n + i].
cudaError_t launch_rank_sum(const float* parts, float* out, int32_t world, int64_t n, int sms,
                            cudaStream_t stream);

}  // namespace adaln
