// Device-side building blocks shared by the forward, backward and stage-2 kernels.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace adaln {

constexpr int kMaxCtas = 4096;      // upper bound on the row-tile count of one launch
constexpr int kStage2Threads = 256;
constexpr int kMaxStages = 8;       // deepest shared-memory ring, in rounds
enum : int { kRingNone = 0, kRingBulk = 1, kRingCopy = 2 };  // forward staging modes

// Largest CTA the host may pick for NV vectors a thread of VE-element vectors. It is the
// kernels' launch bound, which sets their register budget (65536 / bound a thread): bf16
// rows of 8 vectors a thread (64 elements; bf16 D <= 16384 needs at most 256 threads) get
// 255 registers, fp32 ones keep 512 threads for D = 16384.
__host__ __device__ constexpr int max_threads(int nv, int ve) {
    return nv == 1 ? 512 : nv >= 8 ? (ve == 8 ? 256 : 512) : 384;
}
// Launch bound of the backward's wide form (bf16, four vectors a thread, more threads than
// max_threads(4, 8)): the row's x and dy are read from the ring twice.
constexpr int kWideThreads = 512;
// Launch bound of the backward's split form (fp32 rows too wide for a two-round ring): the
// two CTAs of a cluster take half a row each, eight vectors a thread.
constexpr int kSplitThreads = 256;

// A CTA processes its rows in rounds of kRows rows, each thread owning NV 16-byte column
// vectors of every row. Wider per-thread slices hold fewer rows per round so the values
// stay in registers.
template <int NV>
struct RowShape {
    static constexpr int kRows = NV <= 2 ? 2 : 1;
    // The forward holds one row's values where the backward holds two (x and dy), so it
    // can take two rows a round up to NV = 3.
    static constexpr int kFwdRows = NV <= 3 ? 2 : 1;

};

// ---------------------------------------------------------------------------------------
// Debug builds (-DADALN_DEBUG, libadaln_debug.so): each computed index of a global or
// shared-memory access is checked against the extent of its buffer first. A failed check
// skips the access (a load yields zeros) and sets its class bit in the module's debug word,
// which adaln_debug_read returns; nothing traps. Release builds compile the checks away
// (ADALN_IN is the constant true and evaluates nothing).
// ---------------------------------------------------------------------------------------
enum : uint32_t {
    kDbgRows = 1u,       // x, dy, y, dx: row in [0, R), bytes within the row
    kDbgStats = 2u,      // mean, rstd: row in [0, R)
    kDbgMod = 4u,        // shift, scale: modulation row in [0, nmod), bytes within the row
    kDbgPartials = 8u,   // backward partials: slot in [0, S), column in [0, D)
    kDbgSegments = 16u,  // cu_seqlens[0 .. nseg], mod_idx[0 .. nseg)
    kDbgShared = 32u,    // shared-memory ring: within the launch's dynamic shared memory
    kDbgGrads = 64u,     // dshift, dscale: [0, nmod) x [0, D)
    kDbgRanks = 128u,    // rank sum: [0, n) of each rank's array and of the output
    kDbgStatus = 256u,   // status words: [0, kMaxCtas)
};
#ifdef ADALN_DEBUG
static __device__ unsigned int g_adaln_debug;  // one per translation unit (module)
static __device__ __noinline__ void debug_fail(uint32_t cls) { atomicOr(&g_adaln_debug, cls); }
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
    return r;
}
#define ADALN_IN(cls, cond) ((cond) || (::adaln::debug_fail(cls), false))
// [addr, addr + bytes) within the dynamic shared memory that starts at shared address base.
#define ADALN_IN_RING(base, addr, bytes) \
    ADALN_IN(::adaln::kDbgShared,        \
             (addr) >= (base) && (uint64_t)((addr) - (base)) + (uint64_t)(bytes) <= ::adaln::dynamic_smem_bytes())
// The module's debug word, optionally cleared (host side).
static inline cudaError_t debug_word(uint32_t* out, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_adaln_debug, sizeof(uint32_t));
    if (e == cudaSuccess && reset) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_adaln_debug, &zero, sizeof(uint32_t));
    }
    return e;
}
#else
#define ADALN_IN(cls, cond) true
#define ADALN_IN_RING(base, addr, bytes) true
static inline cudaError_t debug_word(uint32_t* out, bool) {
    *out = 0;
    return cudaSuccess;
}
#endif
// Row r of a tensor of R rows, bytes [off, off + n) of a row of rb bytes.
#define ADALN_IN_ROW(r, R, off, n, rb) \
    ADALN_IN(::adaln::kDbgRows, (r) >= 0 && (r) < (R) && (int64_t)(off) + (int64_t)(n) <= (int64_t)(rb))

// Workspace layout: [header | one status word per CTA | backward partials].
constexpr size_t kHeaderBytes = 256;
constexpr size_t kStatusWordsBytes = sizeof(uint32_t) * kMaxCtas;
constexpr size_t kPartialsOffset = kHeaderBytes + kStatusWordsBytes;
constexpr uint32_t kStatusMagic = 0x4E4C4441u;  // "ADLN"

enum : uint32_t { kErrSeqlens = 1u, kErrModIdx = 2u, kErrTimeout = 4u };

struct WsHeader {
    uint32_t magic;
    uint32_t nwords;
    uint32_t reserved[2];
};

// Row -> segment -> modulation row. Dense batches use segment s = [s*N, (s+1)*N) with
// modulation row s; packed batches read the device tables.
struct Segments {
    const int32_t* cu;   // packed: [nseg + 1]
    const int32_t* mod;  // packed: [nseg]
    int64_t nseg;
    int64_t N;           // dense: rows per sample
    int64_t nmod;
    int64_t R;           // total rows
};

struct FwdArgs {
    const void* x;
    const void* shift;
    const void* scale;
    void* y;
    float* mean;
    float* rstd;
    int64_t D;
    float eps;
    Segments seg;
    uint32_t* status;    // per-CTA status words (packed calls), or null
    WsHeader* header;
    int stages;          // shared-memory ring depth in rounds (ring kernels only)
};

struct BwdArgs {
    const void* dy;
    const void* x;
    const float* mean;
    const float* rstd;
    const void* scale;
    void* dx;
    // Per-piece fp32 column sums of dy (q = 0) and dy * xhat (q = 1) over piece slot b + s
    // (CTA b's rows of segment s), S = G + nseg slots, in one of two layouts:
    //   row-major     partials[(slot * 2 + q) * D + column]: a piece is one contiguous row,
    //                 for modulation rows with few pieces each (a row is read whole);
    //   vector-major  partials[((v * 2 + q) * S + slot) * VE + e], column = v * VE + e: one
    //                 16-byte vector's pieces sit side by side, for rows with many pieces
    //                 (their pieces are read down the slots).
    float* partials;
    int vec_major;
    int64_t D;
    Segments seg;
    uint32_t* status;
    WsHeader* header;
    int stages;
};

struct Stage2Args {
    const float* partials;  // the backward's, in the layout vec_major names
    float* dshift;
    float* dscale;
    int64_t D;
    int64_t G;           // row tiles of the backward launch
    int64_t S;           // partial slots: G + nseg
    int vec_major;
    int cw;              // row-major: float4 columns per CTA (power of two, <= kStage2Threads)
    int splits;          // vector-major: threads summing one vector (power of two, <= kStage2Threads)
    Segments seg;
};

// ---------------------------------------------------------------------------------------
// Row tiles: CTA b of G owns rows [b*R/G, (b+1)*R/G); with G <= R every tile is non-empty.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ int64_t tile_begin(int64_t b, int64_t R, int64_t G) { return b * R / G; }

// The tile that holds row r: the largest b with b*R/G <= r.
__device__ __forceinline__ int64_t tile_of_row(int64_t r, int64_t R, int64_t G) {
    return ((r + 1) * G - 1) / R;
}

template <bool VARLEN>
__device__ __forceinline__ int64_t seg_start(const Segments& sg, int64_t s) {
    if constexpr (VARLEN) return ADALN_IN(kDbgSegments, s >= 0 && s <= sg.nseg) ? (int64_t)__ldg(sg.cu + s) : 0;
    else return s * sg.N;
}

template <bool VARLEN>
__device__ __forceinline__ int64_t seg_mod(const Segments& sg, int64_t s) {
    if constexpr (VARLEN) return ADALN_IN(kDbgSegments, s >= 0 && s < sg.nseg) ? (int64_t)__ldg(sg.mod + s) : -1;
    else return s;
}

// Largest s in [0, nseg) with start(s) <= row. At most log2(nseg)+1 probes whatever the table
// holds, so a malformed table cannot stall it.
template <bool VARLEN>
__device__ int64_t seg_find(const Segments& sg, int64_t row) {
    if constexpr (!VARLEN) {
        return sg.N > 0 ? min(row / sg.N, sg.nseg - 1) : 0;
    } else {
        int64_t lo = 0, hi = sg.nseg - 1;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (seg_start<true>(sg, mid) <= row) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    }
}

// CTA b checks its share of the segment table; CTA 0 also checks both ends.
template <bool VARLEN>
__device__ uint32_t validate_segments(const Segments& sg, int64_t b, int64_t G) {
    if constexpr (!VARLEN) {
        return 0u;
    } else {
        uint32_t e = 0;
        const int64_t s0 = b * sg.nseg / G, s1 = (b + 1) * sg.nseg / G;
        for (int64_t s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
            if (!ADALN_IN(kDbgSegments, s >= 0 && s < sg.nseg)) continue;
            const int64_t a = __ldg(sg.cu + s), c = __ldg(sg.cu + s + 1);
            if (a > c || a < 0 || c > sg.R) e |= kErrSeqlens;
            const int64_t m = __ldg(sg.mod + s);
            if (m < 0 || m >= sg.nmod) e |= kErrModIdx;
        }
        if (b == 0 && threadIdx.x == 0 && ADALN_IN(kDbgSegments, sg.nseg >= 0)) {
            if (__ldg(sg.cu) != 0 || (int64_t)__ldg(sg.cu + sg.nseg) != sg.R) e |= kErrSeqlens;
        }
        return e;
    }
}

// Every CTA stores its status word (no zeroing, no atomics); CTA 0 stamps the header.
__device__ __forceinline__ void publish_status(uint32_t err, uint32_t* words, WsHeader* header) {
    // __syncthreads_or answers only "any thread non-zero?", so combine bit by bit.
    uint32_t all = 0;
    if (__syncthreads_or((int)(err & kErrSeqlens))) all |= kErrSeqlens;
    if (__syncthreads_or((int)(err & kErrModIdx))) all |= kErrModIdx;
    if (__syncthreads_or((int)(err & kErrTimeout))) all |= kErrTimeout;
    if (words == nullptr || threadIdx.x != 0 || !ADALN_IN(kDbgStatus, blockIdx.x < kMaxCtas)) return;
    words[blockIdx.x] = all;
    if (blockIdx.x == 0) {
        header->magic = kStatusMagic;
        header->nwords = gridDim.x;
    }
}

// ---------------------------------------------------------------------------------------
// Rounds: a CTA walks its tile in rounds of up to RB consecutive rows that never cross a
// segment boundary. Two walkers with the same start produce the same sequence, so a
// prefetching walker can run ahead of the consuming one.
// ---------------------------------------------------------------------------------------
template <bool VARLEN, int RB>
struct Walker {
    int64_t row;      // first row of the next round
    int64_t s;        // segment holding `row` once seg_end is valid
    int64_t seg_end;  // min(end of segment s, tile end); -1 before the first round
    bool bad;         // ran past the segment table

    __device__ __forceinline__ bool next(const Segments& sg, int64_t r1, int64_t& start, int& nr,
                                         int64_t& seg) {
        if (row >= r1) return false;
        if (row >= seg_end) {
            while (s < sg.nseg && seg_start<VARLEN>(sg, s + 1) <= row) ++s;
            if (s >= sg.nseg) {
                bad = true;
                row = r1;
                return false;
            }
            seg_end = min(seg_start<VARLEN>(sg, s + 1), r1);
        }
        start = row;
        nr = (int)min((int64_t)RB, seg_end - row);
        seg = s;
        row += nr;
        return true;
    }
};

// Asynchronous global -> shared copies issued per thread. Completion is tracked per thread
// with commit/wait groups and each thread reads back only what it copied itself, so no
// cross-thread synchronisation (and no waiting on anyone else) is involved.
// Copies are addressed by 32-bit shared-window addresses (cheaper index math).
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16_sa(uint32_t sa, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4_sa(uint32_t sa, const void* gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}
// Shared loads issued after a cp.async wait: volatile, so they stay behind the wait.
__device__ __forceinline__ uint4 lds128(uint32_t sa) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(sa));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t sa) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(sa));
    return v;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most n of this thread's groups are pending (n = ring depth - 1, 0..7).
__device__ __forceinline__ void cp_async_wait(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---------------------------------------------------------------------------------------
// Bulk (TMA) row copies into a shared-memory ring, completed on an mbarrier per slot.
// One thread issues a whole row with one instruction; every thread waits on the slot's
// mbarrier. Every wait is bounded: after kWaitLimitNs it sets the CTA's abort flag (so no
// later wait lingers), reports failure, and the kernel carries on with whatever is in the
// slot, so a stuck copy can cost at most one bounded wait, never a hang.
// ---------------------------------------------------------------------------------------
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Makes initialised mbarriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// One contiguous global -> shared copy of `bytes` (a multiple of 16, both ends 16-byte
// aligned) that completes `bytes` of the mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for phase `parity` of the mbarrier; false (and *abort set) if it did not complete
// within kWaitLimitNs, or immediately if another thread already gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*abort) return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------------------
// Two-CTA clusters (the backward's split form): the CTAs exchange each row's partial sums
// through distributed shared memory, announced on an mbarrier of the receiving CTA.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of both CTAs: all shared-memory writes before it are visible to the cluster
// after it. Used where both CTAs are known to arrive (after set-up, before exit).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this thread's prior writes.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// mbar_wait_bounded for a barrier another CTA of the cluster arrives on (acquire at cluster
// scope, so its writes into this CTA's shared memory are visible after it).
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*abort) return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------------------
// Programmatic dependent launch. Every kernel is launched so that it may be scheduled before
// the kernel ahead of it in the stream has finished: its CTAs take SMs as that kernel's CTAs
// retire. Each kernel first lets its own dependents be scheduled, then waits, before any
// global memory access, until the kernel ahead has completed and its writes are visible.
// Without such a kernel ahead (a copy, an event, a kernel launched without the attribute)
// the wait returns at once. This hides a launch's scheduling and set-up behind the end of
// the previous kernel; nothing is read or written early.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// cluster: CTAs a cluster along x (1: no clusters).
inline cudaError_t launch_dependent(const void* fn, dim3 grid, dim3 block, void** params, size_t smem,
                                    cudaStream_t stream, unsigned cluster = 1) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelExC(&cfg, fn, params);
}

// Lets `fn` use, with its static shared memory, up to the device's opt-in shared memory per
// block (host side).
inline cudaError_t allow_dynamic_smem(const void* fn) {
    int dev = 0, optin = 0;
    cudaFuncAttributes attr{};
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&attr, fn);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)attr.sharedSizeBytes);
    return e;
}

// ---------------------------------------------------------------------------------------
// Packed fp32 pairs: Blackwell's f32x2 ALU instructions. Each lane of a pair is rounded
// exactly as the scalar instruction would round it.
// ---------------------------------------------------------------------------------------
// A pair is held in one 64-bit register (low half = element 2p, high half = element 2p+1). Keeping pairs in this form end to end lets the compiler feed
// the f32x2 instructions without repacking 32-bit halves around every operation.
using f2r = unsigned long long;
__device__ __forceinline__ f2r p_add(f2r a, f2r b) {
    f2r d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2r p_sub(f2r a, f2r b) {
    f2r d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2r p_mul(f2r a, f2r b) {
    f2r d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2r p_fma(f2r a, f2r b, f2r c) {
    f2r d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2r p_splat(float v) {
    f2r d;
    asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(v));
    return d;
}
__device__ __forceinline__ float2 p_get(f2r a) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(a));
    return v;
}
__device__ __forceinline__ float p_hsum(f2r a) {
    const float2 v = p_get(a);
    return v.x + v.y;
}
constexpr f2r kPairZero = 0ull;  // (+0.0f, +0.0f)

// ---------------------------------------------------------------------------------------
// Reductions
// ---------------------------------------------------------------------------------------
// Butterfly sum over the warp: every lane ends with the same bits.
template <int NVAL>
__device__ __forceinline__ void warp_sum(float (&v)[NVAL]) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
        for (int i = 0; i < NVAL; ++i) v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], o);
    }
}

// CTA-wide sum of one value per warp, written by lane 0 of each warp to red[i][warp]; the
// slots of absent warps hold zeros. ng = the warp count rounded up to a power of two. Every
// group of ng lanes loads the ng slots and sums them with a butterfly over its own lanes,
// so each lane ends with the full sum, and all threads of the CTA get the same bits.
template <int NVAL>
__device__ __forceinline__ void cta_sum(const float (*red)[32], int ng, int lane,
                                        float (&out)[NVAL]) {
#pragma unroll
    for (int i = 0; i < NVAL; ++i) out[i] = red[i][lane & (ng - 1)];
    for (int o = ng >> 1; o >= 1; o >>= 1) {
#pragma unroll
        for (int i = 0; i < NVAL; ++i) out[i] += __shfl_xor_sync(0xFFFFFFFFu, out[i], o);
    }
}

// Zero the reduction slots no warp writes (called once, before the first barrier).
template <int NROWS>
__device__ __forceinline__ void zero_absent_warps(float (*red)[32], int nwarps) {
    for (int idx = threadIdx.x; idx < NROWS * 32; idx += blockDim.x)
        if ((idx & 31) >= nwarps) red[idx >> 5][idx & 31] = 0.0f;
}

// ---------------------------------------------------------------------------------------
// 16-byte vectors of the I/O type.
// ---------------------------------------------------------------------------------------
template <typename T>
struct Io;

template <>
struct Io<float> {
    static constexpr int VE = 4;  // elements per 16-byte vector
    __device__ static __forceinline__ float first(const void* p) {
        return __ldg(reinterpret_cast<const float*>(p));
    }
    // Element 0 of a row, from the row's first 32-bit word.
    __device__ static __forceinline__ float first_of_word(uint32_t w) { return __uint_as_float(w); }
    // As VE/2 pair registers.
    __device__ static __forceinline__ void unpackp(const uint4& v, f2r* f) {
        asm("mov.b64 %0, {%1, %2};" : "=l"(f[0]) : "r"(v.x), "r"(v.y));
        asm("mov.b64 %0, {%1, %2};" : "=l"(f[1]) : "r"(v.z), "r"(v.w));
    }
    __device__ static __forceinline__ uint4 packp(const f2r* f) {
        uint4 v;
        asm("mov.b64 {%0, %1}, %2;" : "=r"(v.x), "=r"(v.y) : "l"(f[0]));
        asm("mov.b64 {%0, %1}, %2;" : "=r"(v.z), "=r"(v.w) : "l"(f[1]));
        return v;
    }
};

template <>
struct Io<__nv_bfloat16> {
    static constexpr int VE = 8;
    // bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 pattern.
    __device__ static __forceinline__ float first(const void* p) {
        const uint32_t h = __ldg(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(h << 16);
    }
    __device__ static __forceinline__ float first_of_word(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ static __forceinline__ void unpackp(const uint4& v, f2r* f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            asm("{\n\t.reg .b32 lo, hi;\n\tshl.b32 lo, %1, 16;\n\tand.b32 hi, %1, 0xFFFF0000;\n\t"
                "mov.b64 %0, {lo, hi};\n\t}"
                : "=l"(f[j])
                : "r"(w[j]));
    }
    // Round each pair to bf16 (nearest, ties to even) and pack it into one 32-bit word.
    __device__ static __forceinline__ uint4 packp(const f2r* f) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            asm("{\n\t.reg .f32 lo, hi;\n\tmov.b64 {lo, hi}, %1;\n\tcvt.rn.bf16x2.f32 %0, hi, lo;\n\t}"
                : "=r"(w[j])
                : "l"(f[j]));
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Streamed (read-once) 16-byte load: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// 16-byte load of data reused across rows (modulation rows): read-only path, cached.
__device__ __forceinline__ uint4 ld_keep(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void st_vec(void* p, const uint4& v) {
    *reinterpret_cast<uint4*>(p) = v;
}

}  // namespace adaln
