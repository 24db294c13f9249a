// Device-side building blocks shared by the forward, backward and stage-2 kernels.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace adaln {

constexpr int kMaxCtas = 4096;      // upper bound on the row-tile count of one launch
constexpr int kStage2Threads = 256;

// A CTA processes one row at a time (or kRows rows per reduction round), each thread owning
// NV 16-byte column vectors of the row. Wider rows hold fewer rows per round so the
// accumulators stay in registers; kMaxThreads bounds the CTA size the host may pick.
template <int NV>
struct RowShape {
    static constexpr int kRows = NV >= 3 ? 1 : 2;
    static constexpr int kMaxThreads = NV >= 4 ? 1024 : 512;
};

// Workspace layout: [header | one status word per CTA | backward partials].
constexpr size_t kHeaderBytes = 256;
constexpr size_t kStatusWordsBytes = sizeof(uint32_t) * kMaxCtas;
constexpr size_t kPartialsOffset = kHeaderBytes + kStatusWordsBytes;
constexpr uint32_t kStatusMagic = 0x4E4C4441u;  // "ADLN"

enum : uint32_t { kErrSeqlens = 1u, kErrModIdx = 2u };

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
};

struct BwdArgs {
    const void* dy;
    const void* x;
    const float* mean;
    const float* rstd;
    const void* scale;
    void* dx;
    float* partials;     // [G + nseg][2][D]: slot b + s holds CTA b's sums over segment s
    int64_t D;
    Segments seg;
    uint32_t* status;
    WsHeader* header;
};

struct Stage2Args {
    const float* partials;
    float* dshift;
    float* dscale;
    int64_t D;
    int64_t G;           // row tiles of the backward launch
    int cw;              // float4 columns per CTA (power of two, <= kStage2Threads)
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
    if constexpr (VARLEN) return (int64_t)__ldg(sg.cu + s);
    else return s * sg.N;
}

template <bool VARLEN>
__device__ __forceinline__ int64_t seg_mod(const Segments& sg, int64_t s) {
    if constexpr (VARLEN) return (int64_t)__ldg(sg.mod + s);
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
            const int64_t a = __ldg(sg.cu + s), c = __ldg(sg.cu + s + 1);
            if (a > c || a < 0 || c > sg.R) e |= kErrSeqlens;
            const int64_t m = __ldg(sg.mod + s);
            if (m < 0 || m >= sg.nmod) e |= kErrModIdx;
        }
        if (b == 0 && threadIdx.x == 0) {
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
    if (words == nullptr || threadIdx.x != 0) return;
    words[blockIdx.x] = all;
    if (blockIdx.x == 0) {
        header->magic = kStatusMagic;
        header->nwords = gridDim.x;
    }
}

// ---------------------------------------------------------------------------------------
// 16-byte vectors of the I/O type.
// ---------------------------------------------------------------------------------------
template <typename T>
struct Io;

template <>
struct Io<float> {
    static constexpr int VE = 4;  // elements per 16-byte vector
    __device__ static __forceinline__ void unpack(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static __forceinline__ uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ static __forceinline__ float first(const void* p) {
        return __ldg(reinterpret_cast<const float*>(p));
    }
};

template <>
struct Io<__nv_bfloat16> {
    static constexpr int VE = 8;
    // bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 pattern.
    __device__ static __forceinline__ void unpack(const uint4& v, float* f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = __uint_as_float(w[j] << 16);
            f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
    __device__ static __forceinline__ uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static __forceinline__ uint4 pack(const float* f) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ static __forceinline__ float first(const void* p) {
        const uint32_t h = __ldg(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(h << 16);
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

template <int NVAL>
__device__ __forceinline__ void warp_sum(float (&v)[NVAL]) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
        for (int i = 0; i < NVAL; ++i) v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], o);
    }
}

}  // namespace adaln
