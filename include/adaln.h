/*
 * libadaln — fused AdaLN (LayerNorm-Modulate) forward and backward for GB300 (sm_103a).
 *
 * The operator is the fused normalisation + modulation node of video / MMDiT diffusion
 * transformers described in "AdaptiveLoad: Towards Efficient Video Diffusion Transformer
 * Training" (technical summary, section 2.B "Fused LayerNorm-Modulate CUDA kernels").
 * The pages name the operator without printing its formula; this library computes, for
 * every token row x of width D that is modulated by row m of the shift/scale tables:
 *
 *     mean = (1/D) sum_d x_d,   var = (1/D) sum_d (x_d - mean)^2   (biased)
 *     rstd = 1 / sqrt(var + eps),   xhat = (x - mean) * rstd       (no LayerNorm affine)
 *     y    = xhat * (1 + scale[m]) + shift[m]
 *
 * and the gradients of a loss L with dL/dy = dy:
 *
 *     dx        = rstd * (g - mean_d(g) - xhat * mean_d(g * xhat)),  g = dy * (1 + scale[m])
 *     dshift[m] = sum over tokens of m of dy,   dscale[m] = sum over tokens of m of dy * xhat
 *
 * The backward reduces dshift/dscale with threads pinned to a feature index d that
 * accumulate down the sequence (the section's "D-tile coalesced reduction"), into per-tile
 * fp32 partials that a second, fixed-order stage sums: results are bitwise reproducible
 * run to run on the same device with the same arguments. No float atomics are used.
 *
 * Layouts (all row-major, D contiguous):
 *   x, y, dy, dx      [R, D]   in `dtype`       R = Bt*N (dense) or total_tokens (packed)
 *   shift, scale      [nmod, D] in `dtype`      dense: nmod = Bt, token (b, n) uses row b
 *   mean, rstd        [R]      fp32
 *   dshift, dscale    [nmod, D] fp32            (always fp32, also for bf16 I/O)
 *   cu_seqlens        [nseg+1] int32 (device)   packed: cu_seqlens[0] = 0, non-decreasing,
 *                                               cu_seqlens[nseg] = total_tokens
 *   mod_idx           [nseg]   int32 (device)   segment s uses modulation row mod_idx[s]
 *
 * Ownership and execution. The caller owns every buffer. Every call is asynchronous and
 * ordered on the caller's `stream`; nothing synchronises except adaln_read_status. The
 * library allocates no device memory and keeps no state beyond cached device properties
 * (adaln_bwd_noalloc's fixed scratch array, below, is part of the loaded module).
 * Inputs and outputs must not alias.
 *
 * Preconditions (checked on the host; a violation returns a status and launches nothing):
 *   - x, y, dy, dx, shift, scale, dshift, dscale: 16-byte aligned; mean, rstd: 4-byte
 *     aligned; workspace: 256-byte aligned.
 *   - 8 <= D <= 16384 and D % 8 == 0; eps > 0 and finite.
 *   - Bt, N, total_tokens, nseg, nmod >= 0 (empty problems are valid: a backward with no
 *     tokens writes zero gradients).
 *
 * Data errors in device-resident tables (cu_seqlens not starting at 0, decreasing, or not
 * ending at total_tokens; mod_idx outside [0, nmod)) cannot be seen by the host. The
 * kernels detect them, skip the affected rows without any out-of-range access, and record
 * a code in the workspace; adaln_read_status returns it.
 *
 * Workspace. The packed forward and both backwards take a caller-allocated device
 * workspace of at least the size the matching *_workspace_size function returns for the
 * CURRENT device (the size depends on its SM count). It needs no initialisation.
 * Determinism holds for a fixed device model: the tile split follows its SM count.
 */
#ifndef ADALN_H_
#define ADALN_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ADALN_F32 = 0, ADALN_BF16 = 1 } adaln_dtype;

typedef enum {
    ADALN_OK = 0,
    ADALN_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad eps or dtype       */
    ADALN_ERR_UNSUPPORTED = 2,  /* D outside [8, 16384] or not a multiple of 8          */
    ADALN_ERR_ALIGNMENT = 3,    /* a pointer violates the alignment above               */
    ADALN_ERR_WORKSPACE = 4,    /* workspace null or smaller than required              */
    ADALN_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed          */
    ADALN_ERR_BAD_SEQLENS = 6,  /* device data: cu_seqlens malformed (adaln_read_status) */
    ADALN_ERR_BAD_MOD_IDX = 7,  /* device data: mod_idx out of range (adaln_read_status) */
    ADALN_ERR_TIMEOUT = 8       /* a kernel gave up waiting (1 s) for a bulk copy of its
                                   input rows, or for the row sums of the other CTA of its
                                   cluster (fp32 rows wider than 14336); its outputs from
                                   then on are not valid (adaln_read_status) */
} adaln_status;

/* Forward, dense batch x[Bt, N, D]; token (b, n) uses shift[b], scale[b].
 * Writes y, mean, rstd. Section 2.B, forward-pass bullet: statistics stay on chip, the
 * row is reduced by warp shuffles then a block reduction, and the modulation is applied
 * on a later pass over the row held in registers. One launch. */
int adaln_fwd(const void* x, const void* shift, const void* scale, void* y, float* mean,
              float* rstd, int64_t Bt, int64_t N, int64_t D, float eps, adaln_dtype dtype,
              cudaStream_t stream);

/* Workspace bytes adaln_bwd needs on the current device. */
size_t adaln_bwd_workspace_size(int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype);

/* Backward, dense batch. Reads dy, x, the forward's mean/rstd and scale; writes dx [Bt,N,D]
 * and dshift/dscale [Bt, D] (fp32, overwritten). Section 2.B, backward-pass bullet ("D-tile
 * coalesced reduction"): each row's dx is computed from the saved statistics while threads
 * pinned to feature indices accumulate dy and dy*xhat down their tile of rows; per-tile
 * partials are summed by a second, fixed-order stage. Two launches on `stream`; for fp32
 * rows wider than 14336 the first is a launch of two-CTA thread-block clusters (each CTA
 * half of every row), so such calls need a device and context that allow clusters. */
int adaln_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
              const void* scale, void* dx, float* dshift, float* dscale, void* workspace,
              size_t workspace_bytes, int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype,
              cudaStream_t stream);

/* The two stages of adaln_bwd as separate calls, taking adaln_bwd's exact arguments:
 * adaln_bwd_partials launches only the fused dx + per-tile partial kernel (writes dx and the
 * workspace partials; dshift/dscale untouched), adaln_bwd_reduce only the fixed-order
 * second stage (reads the workspace partials, writes dshift/dscale). Calling both in this
 * order on one stream is exactly adaln_bwd; they exist so each stage can be timed alone. */
int adaln_bwd_partials(const void* dy, const void* x, const float* mean, const float* rstd,
                       const void* scale, void* dx, float* dshift, float* dscale, void* workspace,
                       size_t workspace_bytes, int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype,
                       cudaStream_t stream);
int adaln_bwd_reduce(const void* dy, const void* x, const float* mean, const float* rstd,
                     const void* scale, void* dx, float* dshift, float* dscale, void* workspace,
                     size_t workspace_bytes, int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype,
                     cudaStream_t stream);

/* Workspace bytes adaln_fwd_varlen needs (a small status area). */
size_t adaln_fwd_varlen_workspace_size(int64_t total_tokens, int32_t nseg, int64_t D,
                                       adaln_dtype dtype);

/* Forward, packed mixed-length segments (x[total_tokens, D]); segment s uses modulation
 * row mod_idx[s] of shift/scale [nmod, D]. Same math as adaln_fwd. Section 2.A batches
 * sequences of very different lengths into buckets (B sequences of length S each); the pages
 * print no interface for feeding such a bucket to the operator. This call is the library's
 * reading: the bucket's sequences packed back to back, delimited by the prefix sums
 * cu_seqlens (segment s = rows [cu_seqlens[s], cu_seqlens[s+1])), each sequence with its
 * own modulation row (the timestep / condition embedding of its sample), as section 2.B's
 * per-sample modulation requires. The workspace receives the per-CTA status words. */
int adaln_fwd_varlen(const void* x, const void* shift, const void* scale, void* y, float* mean,
                     float* rstd, const int32_t* cu_seqlens, const int32_t* mod_idx, int32_t nseg,
                     int64_t total_tokens, int64_t nmod, int64_t D, float eps, void* workspace,
                     size_t workspace_bytes, adaln_dtype dtype, cudaStream_t stream);

/* Workspace bytes adaln_bwd_varlen needs on the current device. */
size_t adaln_bwd_varlen_workspace_size(int64_t total_tokens, int32_t nseg, int64_t nmod,
                                       int64_t D, adaln_dtype dtype);

/* Backward, packed segments (the layout of adaln_fwd_varlen, section 2.A buckets).
 * dshift/dscale [nmod, D]: row m sums every token of every segment with mod_idx == m, in a
 * fixed order; rows no segment uses are written as 0. Section 2.B, backward-pass bullet:
 * the D-tile reduction runs down each (row tile, segment) piece, and the pieces of every
 * modulation row are summed by the fixed-order second stage. */
int adaln_bwd_varlen(const void* dy, const void* x, const float* mean, const float* rstd,
                     const void* scale, void* dx, float* dshift, float* dscale,
                     const int32_t* cu_seqlens, const int32_t* mod_idx, int32_t nseg,
                     int64_t total_tokens, int64_t nmod, int64_t D, void* workspace,
                     size_t workspace_bytes, adaln_dtype dtype, cudaStream_t stream);

/* The two stages of adaln_bwd_varlen, with its exact arguments (see adaln_bwd_partials). */
int adaln_bwd_varlen_partials(const void* dy, const void* x, const float* mean, const float* rstd,
                              const void* scale, void* dx, float* dshift, float* dscale,
                              const int32_t* cu_seqlens, const int32_t* mod_idx, int32_t nseg,
                              int64_t total_tokens, int64_t nmod, int64_t D, void* workspace,
                              size_t workspace_bytes, adaln_dtype dtype, cudaStream_t stream);
int adaln_bwd_varlen_reduce(const void* dy, const void* x, const float* mean, const float* rstd,
                            const void* scale, void* dx, float* dshift, float* dscale,
                            const int32_t* cu_seqlens, const int32_t* mod_idx, int32_t nseg,
                            int64_t total_tokens, int64_t nmod, int64_t D, void* workspace,
                            size_t workspace_bytes, adaln_dtype dtype, cudaStream_t stream);

/* Backward without saved statistics, for callers that do not keep the forward's mean and
 * rstd (8 bytes a row of activation memory): they are first recomputed from x with the
 * forward's row mapping and arithmetic (bitwise the values the forward wrote, for the same
 * eps), into the end of the workspace, then the backward runs as adaln_bwd /
 * adaln_bwd_varlen. It costs one more read of x.
 * The workspace must hold the *_recompute_workspace_size bytes (which include the
 * backward's own); arguments and errors otherwise as adaln_bwd / adaln_bwd_varlen. */
size_t adaln_bwd_recompute_workspace_size(int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype);
int adaln_bwd_recompute(const void* dy, const void* x, const void* scale, void* dx, float* dshift,
                        float* dscale, void* workspace, size_t workspace_bytes, int64_t Bt, int64_t N,
                        int64_t D, float eps, adaln_dtype dtype, cudaStream_t stream);
size_t adaln_bwd_varlen_recompute_workspace_size(int64_t total_tokens, int32_t nseg, int64_t nmod,
                                                 int64_t D, adaln_dtype dtype);
int adaln_bwd_varlen_recompute(const void* dy, const void* x, const void* scale, void* dx,
                               float* dshift, float* dscale, const int32_t* cu_seqlens,
                               const int32_t* mod_idx, int32_t nseg, int64_t total_tokens, int64_t nmod,
                               int64_t D, float eps, void* workspace, size_t workspace_bytes,
                               adaln_dtype dtype, cudaStream_t stream);

/* Synchronises `stream`, then returns the device-side status recorded in `workspace` by
 * the last packed forward/backward (or backward) that used it: ADALN_OK,
 * ADALN_ERR_BAD_SEQLENS, ADALN_ERR_BAD_MOD_IDX or ADALN_ERR_TIMEOUT, in that order of
 * precedence (ADALN_ERR_CUDA if the copy fails, ADALN_ERR_WORKSPACE if the workspace holds
 * no status). Every wait a kernel makes on its own bulk copies is bounded (1 s); a kernel
 * that runs out of time stops, drains the copies it started and records the timeout. The
 * dense forward takes no workspace, so it has nowhere to record one. */
int adaln_read_status(const void* workspace, cudaStream_t stream);

/* Bytes of the fixed scratch array adaln_bwd_noalloc uses on every device that loads the
 * library (16 MiB). */
#define ADALN_NOALLOC_SCRATCH_BYTES (16u << 20)

/* adaln_bwd for callers that cannot allocate device memory (no caller workspace).
 * The paper has no counterpart to this call; it exists for callers such as a host framework
 * that only hands out the tensors it owns, code that runs under an allocator that must not
 * grow, or a plain C program without a device allocator. Same arguments and results as
 * adaln_bwd minus the workspace: the scratch is a fixed array of ADALN_NOALLOC_SCRATCH_BYTES
 * inside this library, held by every GPU that loads the library until the process exits.
 *   - Allocates nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *   - Problems whose scratch need, adaln_bwd_workspace_size(Bt, N, D, dtype), exceeds
 *     ADALN_NOALLOC_SCRATCH_BYTES are rejected with ADALN_ERR_WORKSPACE before any launch.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call before any
 *     stream capture.
 *   - Every call on a device shares the one array, which keeps the last call's contents;
 *     nothing in it needs to start at zero. Calls that overlap on the GPU (different
 *     streams, or different host threads, without ordering between them) race on it and
 *     give wrong gradients: order them on one stream.
 *   - The device address is cached per device index for the life of the process; it does
 *     not survive cudaDeviceReset (or any teardown of the device's primary context), after
 *     which this call must not be used in that process.
 *   - The kernels record device-side errors (a timed-out wait) in the array, where
 *     adaln_read_status cannot see them: read them with adaln_noalloc_read_status. */
int adaln_bwd_noalloc(const void* dy, const void* x, const float* mean, const float* rstd,
                      const void* scale, void* dx, float* dshift, float* dscale, int64_t Bt,
                      int64_t N, int64_t D, adaln_dtype dtype, cudaStream_t stream);

/* adaln_read_status for adaln_bwd_noalloc: synchronises `stream`, then returns the device-side
 * status the last adaln_bwd_noalloc on the current device recorded in the library's fixed
 * array (ADALN_OK or ADALN_ERR_TIMEOUT; ADALN_ERR_WORKSPACE before the first such call on the
 * device, ADALN_ERR_CUDA if the copy fails). It copies a few bytes to the host and allocates
 * nothing on the device. Like adaln_bwd_noalloc, this call has no counterpart in the paper. */
int adaln_noalloc_read_status(cudaStream_t stream);

/* ---- Row sharding across ranks ----------------------------------------------------------
 * A batch can be split into contiguous, segment-aligned row shards, one per rank (the pages
 * train on 8- and 16-GPU clusters, AdaptiveLoad technical summary sections 2.A and 4). The
 * forward needs no exchange; each rank's backward gives dshift/dscale over its own tokens,
 * and the batch's gradients are their sum over ranks. adaln_sum_ranks forms that sum from
 * the ranks' fp32 gradients stacked on one device, parts[world][n] (e.g. after an
 * all-gather), always adding in rank order 0, 1, ..., world - 1:
 *     out[i] = parts[0][i] + parts[1][i] + ... + parts[world - 1][i]
 * so every rank that runs it gets the same bits, whatever moved the data. parts and out are
 * device pointers, 16-byte aligned, not overlapping; n elements each. One launch on
 * `stream`. Returns ADALN_ERR_INVALID_ARG for world < 1 or n < 0. */
int adaln_sum_ranks(const float* parts, float* out, int32_t world, int64_t n, cudaStream_t stream);

/* ---- Debug build --------------------------------------------------------------------------
 * The library can be built a second time with -DADALN_DEBUG (libadaln_debug.so; the package's
 * build(debug=True)). In that build every kernel checks each computed index of a global or
 * shared-memory access against the extent of its buffer before the access; a failed check
 * skips the access (a load yields zeros) and sets the access's class bit in a device-side
 * debug word, without trapping. adaln_debug_read waits for the device (cudaDeviceSynchronize)
 * and stores in *word the OR of the bits set since the last reset (0: no check failed); with
 * reset != 0 it also clears them. Returns ADALN_ERR_INVALID_ARG for a null word, ADALN_ERR_CUDA
 * if the device reports an error, and ADALN_ERR_UNSUPPORTED from the release build, which
 * compiles the checks away. */
#define ADALN_DEBUG_ROWS     1u   /* x, dy, y, dx: row in [0, R), bytes within the row        */
#define ADALN_DEBUG_STATS    2u   /* mean, rstd: row in [0, R)                                */
#define ADALN_DEBUG_MOD      4u   /* shift, scale: modulation row in [0, nmod)                */
#define ADALN_DEBUG_PARTIALS 8u   /* backward partials: slot in [0, tiles + nseg), column < D */
#define ADALN_DEBUG_SEGMENTS 16u  /* cu_seqlens[0 .. nseg], mod_idx[0 .. nseg)                */
#define ADALN_DEBUG_SHARED   32u  /* shared memory: within the CTA's allocation               */
#define ADALN_DEBUG_GRADS    64u  /* dshift, dscale: [0, nmod) x [0, D)                       */
#define ADALN_DEBUG_RANKS    128u /* adaln_sum_ranks: [0, n) of each rank's row              */
#define ADALN_DEBUG_STATUS   256u /* workspace status words                                   */
int adaln_debug_read(uint32_t* word, int reset);

/* Dual-constraint bucket size, AdaptiveLoad technical summary section 2.A:
 *     B = max(1, min(floor(M_mem / S), floor(M_comp / S^p)))
 * with exact integer arithmetic (S^p is never formed past M_comp). Host only.
 * Returns B >= 1, or -ADALN_ERR_INVALID_ARG when S, M_mem or M_comp <= 0 or p < 1. */
int64_t adaln_bucket_batch(int64_t S, int64_t M_mem, int64_t M_comp, int32_t p);

/* ---- Host-side scheduling half of section 2.A (host only, no device work) ------------- */

/* adaln_bucket_batch with a real exponent p > 0, as a fitted exponent is. An integral p in
 * [1, 64] takes the exact integer path; otherwise S^p is evaluated in double precision and
 * floor(M_comp / S^p) can differ by one from the exact value when M_comp / S^p lies within
 * about 1e-13 (relative) of an integer. Returns B >= 1, or -ADALN_ERR_INVALID_ARG when S,
 * M_mem or M_comp <= 0 or p is not positive and finite. */
int64_t adaln_bucket_batch_real(int64_t S, int64_t M_mem, int64_t M_comp, double p);

/* Shape-Benchmarking cost fit, section 2.A: the least-squares fit of the step-time model
 *     t = a + b * B * S^p
 * to n measured (B[i], S[i], t[i]) samples, p searched in [p_lo, p_hi] (for each p the
 * model is linear in a and b, solved exactly; the residual is then minimised over p by a
 * grid bracket and golden-section refinement to 1e-12 in p). With a step-time budget
 * t_budget > a, the compute bound follows as M_comp = floor((t_budget - a) / b).
 * Writes out[0..4] = a, b, p, root-mean-square residual, M_comp (M_comp = 0 when
 * t_budget <= a or b <= 0). Returns ADALN_OK, or ADALN_ERR_INVALID_ARG for n < 3, a null
 * pointer, B or S <= 0, a non-finite t, or not 0 < p_lo < p_hi. */
int adaln_fit_step_cost(const int64_t* B, const int64_t* S, const double* t, int64_t n,
                        double p_lo, double p_hi, double t_budget, double* out);

/* Compute-load imbalance of a bucketing rule, the quantity section 2.A's scheduler lowers
 * (the results report its coefficient of variation across batches). Each of the n sample
 * lengths goes to the smallest of the nbuckets increasing bucket lengths that holds it; a
 * bucket's samples, in input order, fill batches of its batch size, the last one possibly
 * partial. Batch size: rule 0 = the equal-token rule max(1, floor(M_mem / S)); rule 1 =
 * the dual constraint adaln_bucket_batch_real(S, M_mem, M_comp, p). A batch of k samples of
 * bucket S costs k * S^p. Writes out[0..2] = coefficient of variation (population standard
 * deviation / mean) of the batch costs, number of batches, mean cost. Returns ADALN_OK, or
 * ADALN_ERR_INVALID_ARG for a null pointer, n < 1, nbuckets < 1, buckets not increasing and
 * positive, a length <= 0 or above the largest bucket, M_mem or M_comp <= 0, a bad p or rule. */
int adaln_bucket_load_cv(const int64_t* lengths, int64_t n, const int64_t* buckets,
                         int32_t nbuckets, int64_t M_mem, int64_t M_comp, double p, int32_t rule,
                         double* out);

/* Static, human-readable name of a status code. */
const char* adaln_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ADALN_H_ */
