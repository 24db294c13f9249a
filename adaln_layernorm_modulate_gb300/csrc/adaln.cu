// libadaln C-ABI: argument checks, launch planning and launches. See include/adaln.h.
#include "adaln.h"

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "launch.h"

using namespace adaln;

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
int g_sms[kMaxDevices];  // 0 = not yet queried
std::map<std::tuple<int, int, int, int, int, int>, std::pair<int, int>> g_plans;  // launch plans

// Multiprocessor count of the current device (cached), or 0 on failure.
int current_sms(int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    *dev_out = dev;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_sms[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sms[dev] = sms;
    }
    return g_sms[dev];
}

// How a row of width D is spread over a CTA: each thread owns `nv` 16-byte vectors
// (v = tid + k * tpb), so a CTA holds one row in registers. The per-row reduction work is
// paid once per thread per row, so more elements per thread amortise it better, until
// registers run out (row_cfg below gives the measured preferences). Narrow rows shrink nv
// so a warp is not left idle; wide rows grow it so a row fits the CTA size the kernel is
// compiled for (max_threads(nv, elements per vector)).
struct RowCfg {
    int nv;
    int tpb;
    bool full;  // nv * tpb vectors == the row: no idle lanes
};


// The forward's per-thread copy ring is used with one mapping only, where it measured
// faster than the bulk ring: bf16 rows of 384 vectors, three a thread over four warps (two
// rows a round), i.e. D=3072 (992 us on the packed workload against 1035 us with the bulk
// ring, 134 us against 143 us on the MMDiT streams). With fp32 rows or any other mapping
// it measured slower (MMDiT fp32: 290 us against 263; bf16 D=6144, 3 x 256 threads at 143
// rows a CTA slot: 70% of the HBM peak against 90%).
bool copy_ring_cfg(int64_t D, adaln_dtype dtype, RowCfg* c) {
    if (dtype != ADALN_BF16 || D != 3 * 128 * 8) return false;
    *c = RowCfg{3, 128, true};
    return true;
}

// Row mapping of a launch (the bulk ring, plain loads, and the backward). The preferences
// were measured on GB300 (bf16 D=3072 forward: 6 x 64 threads, 67.9 us on a 32,760-token
// segment against 70.6 us for 4 x 96).
RowCfg row_cfg(int64_t D, adaln_dtype dtype, bool forward) {
    static const int kNv[] = {1, 2, 3, 4, 6, 8};
    const bool bf16 = dtype == ADALN_BF16;
    const int64_t VE = bf16 ? 8 : 4;
    const int64_t V = D / VE;
    // Forward rows of at most 6 vectors per lane: one warp per row. The CTA's reductions are
    // then warp shuffles and its barriers cover one warp, so the rows of different warps
    // never wait for each other (bf16 D=1536: 33 us against 36 us for 3 x 64 threads).
    if (forward && V % 32 == 0 && V / 32 <= 6 && V / 32 != 5) return RowCfg{(int)(V / 32), 32, true};
    // The same for backward rows of at most 3 vectors a lane (bf16 D=768: 221 us against 236 us
    // for 1 x 96 threads; 6 vectors a lane measured much slower: the backward keeps more).
    if (!forward && V % 32 == 0 && V / 32 <= 3) return RowCfg{(int)(V / 32), 32, true};
    // Elements a thread: the backward keeps x, dy and two column accumulators per element,
    // the forward one value (bf16 forwards take 48, the others 32).
    int64_t target = (forward ? (bf16 ? 48 : 32) : 16) / VE;
    if ((V + 31) / 32 < target) target = (V + 31) / 32;
    if (target < 1) target = 1;
    // Otherwise a mapping that covers the row exactly (whole warps, no idle lanes), with nv
    // as close to the target as possible (ties go to the smaller nv).
    int best = 0;
    for (int nv : kNv) {
        if (V % nv != 0 || (V / nv) % 32 != 0 || V / nv > max_threads(nv, (int)VE)) continue;
        if (nv > 2 * target) continue;
        if (best == 0 || std::llabs(nv - target) < std::llabs(best - target)) best = nv;
    }
    if (best != 0) return RowCfg{best, (int)(V / best), true};
    // bf16 backward rows too wide for four vectors a thread within max_threads(4, 8): the
    // wide form, four vectors a thread over up to kWideThreads threads, x and dy read from the
    // ring twice (D=14336: 448 threads; D=16384: 512).
    if (!forward && bf16 && V % 4 == 0 && (V / 4) % 32 == 0 && V / 4 > max_threads(4, (int)VE) &&
        V / 4 <= kWideThreads)
        return RowCfg{4, (int)(V / 4), true};
    for (int nv : kNv) {
        if (nv < target) continue;
        const int64_t tpb = ((V + nv - 1) / nv + 31) / 32 * 32;
        if (tpb <= max_threads(nv, (int)VE)) return RowCfg{nv, (int)tpb, V == nv * tpb};
    }
    const int64_t tpb = ((V + 7) / 8 + 31) / 32 * 32;
    return RowCfg{8, (int)tpb, V == 8 * tpb};
}

enum Kind { kFwd = 0, kBwd = 1 };

// Most shared memory a CTA gives its ring; less when registers let more CTAs share the
// SM. A CTA alone on its SM (wide rows in the backward) stops at 150 KB: deeper rings
// measured slower, the rest of the SM's shared memory serving as L1.
constexpr size_t kRingBudget = 150 * 1024;
// Rows whose two-round ring exceeds the budget still get one, up to this size, rather than
// plain loads into registers (fp32 D=12288 backward: two rounds of 96 KB; fp32 D=14336: two
// rounds of 112 KB, 1355 -> 868 us against plain loads). With the kernels' static shared
// memory (about 0.5 KB for such wide rows) it stays within the 227 KB a CTA may opt into.
constexpr size_t kRingLimit = 226 * 1024;
// Forwards with at least this many rows per resident CTA slot of the bulk-ring plan stage
// rows with the per-thread copy ring where copy_ring_cfg allows it, shorter ones with the
// bulk ring (which starts faster, see fwd.cu). bf16 D=3072 (912 bulk-ring slots on 152
// SMs): 36 rows a slot measured faster with the bulk ring, 73 with the copy ring.
constexpr int64_t kCopyRingRows = 64;

struct Plan {
    RowCfg c;
    int ring;       // kRingNone (plain loads into registers), kRingBulk or kRingCopy
    bool full;      // ring kernel specialised for rows the CTA covers exactly
    int stages;     // ring depth in rounds
    size_t smem;    // dynamic shared memory per CTA
    int64_t G;      // CTAs (= row tiles, or twice the row tiles in the split form)
    int sms;
    bool split;     // the backward's split form: two-CTA clusters, half a row each
};

// One ring round: RB rows of x (and of dy for the backward), each padded to the CTA's
// vector grid (nv * tpb * 16 bytes), plus for the copy ring one word per thread and row
// (its copy of the row's first element). The ring also holds one mbarrier per slot.
constexpr size_t kRingHeader = 128;
size_t ring_round_bytes(Kind kind, const RowCfg& c, int ring) {
    const size_t row = (size_t)c.tpb * c.nv * 16;
    if (kind == kFwd)  // RowShape<nv>::kFwdRows rows
        return (c.nv <= 3 ? 2 : 1) * (ring == kRingCopy ? row + (size_t)c.tpb * 4 : row);
    return (c.nv <= 2 ? 2 : 1) * 2 * row;  // RowShape<nv>::kRows, x and dy
}

// Ring depth and resident CTAs per SM of one kernel variant (cached per device).
bool ring_shape(Kind kind, adaln_dtype dtype, bool varlen, int dev, Plan* p) {
    const size_t round = p->ring ? ring_round_bytes(kind, p->c, p->ring) : 0;
    const auto key = std::make_tuple(dev, (int)kind, (int)dtype, p->c.nv,
                                     (int)varlen * 8 + p->ring * 2 + (int)p->full, p->c.tpb);
    std::pair<int, int> cached{0, 0};  // (stages, CTAs per SM)
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) cached = it->second;
    }
    if (cached.second == 0) {
        auto occupancy = [&](size_t smem, int* bps) {
            return kind == kFwd
                       ? fwd_blocks_per_sm((int)dtype, p->c.nv, varlen, p->ring, p->full, p->c.tpb, smem, bps)
                       : bwd_blocks_per_sm((int)dtype, p->c.nv, varlen, p->ring != kRingNone, p->full,
                                           p->c.tpb, smem, bps);
        };
        int stages = 0, bps = 0;
        if (p->ring) {
            // Size the ring so shared memory does not cut the residency registers allow:
            // the SM's shared memory is split among the CTAs the registers let in.
            int by_regs = 0, sm_bytes = 0;
            if (occupancy(0, &by_regs) != cudaSuccess || by_regs <= 0) return false;
            if (cudaDeviceGetAttribute(&sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
                cudaSuccess)
                return false;
            size_t allowance = ((size_t)sm_bytes - (size_t)by_regs * 2048) / (size_t)by_regs - kRingHeader;
            if (allowance > kRingBudget) allowance = kRingBudget;
            size_t st = allowance / round;
            if (st > (size_t)kMaxStages) st = kMaxStages;
            if (st < 2) st = 2;
            stages = (int)st;
        }
        if (occupancy(p->ring ? kRingHeader + (size_t)stages * round : 0, &bps) != cudaSuccess || bps <= 0)
            return false;
        cached = {stages, bps};
        std::lock_guard<std::mutex> lock(g_mu);
        g_plans[key] = cached;
    }
    p->stages = cached.first;
    p->smem = p->ring ? kRingHeader + (size_t)p->stages * round : 0;
    int64_t G = (int64_t)p->sms * cached.second;
    if (G > kMaxCtas) G = kMaxCtas;
    p->G = G;
    return true;
}

// The backward's split form for fp32 rows too wide for a two-round ring: a cluster of two
// CTAs per row tile, each staging half of every row (eight vectors a thread) in a ring of as
// many rounds as kRingLimit holds (three at D=16384: 3 x 64 KB), one cluster per resident
// cluster slot (cached per device).
bool split_plan(int64_t D, bool varlen, int dev, int64_t R, Plan* p) {
    const int64_t VC = D / 4 / 2;  // fp32 vectors of half a row
    const int tpb = (int)(((VC + 7) / 8 + 31) / 32 * 32);
    if (tpb > kSplitThreads) return false;
    p->c = RowCfg{8, tpb, VC == 8 * (int64_t)tpb};
    p->ring = kRingBulk;
    p->full = p->c.full;
    p->split = true;
    const size_t round = ring_round_bytes(kBwd, p->c, kRingBulk);
    const size_t st = std::min<size_t>(kMaxStages, (kRingLimit - kRingHeader) / round);
    if (st < 2) return false;
    p->stages = (int)st;
    p->smem = kRingHeader + st * round;
    const auto key = std::make_tuple(dev, (int)kBwd, (int)ADALN_F32, 8, 32 + (int)varlen * 2 + (int)p->full,
                                     tpb);
    int clusters = 0;  // resident clusters on the device
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) clusters = it->second.second;
    }
    if (clusters == 0) {
        if (bwd_split_clusters(varlen, p->full, tpb, p->smem, &clusters) != cudaSuccess || clusters <= 0)
            return false;
        std::lock_guard<std::mutex> lock(g_mu);
        g_plans[key] = {p->stages, clusters};
    }
    int64_t tiles = std::min<int64_t>(clusters, kMaxCtas / 2);
    if (tiles > R) tiles = R;
    if (tiles < 1) tiles = 1;
    p->G = 2 * tiles;
    return true;
}

// Launch plan: staging mode, ring depth, and row tiles = every resident CTA slot of the
// device (at most one per row).
bool make_plan(Kind kind, adaln_dtype dtype, int64_t D, bool varlen, int64_t R, Plan* p) {
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms <= 0) return false;
    p->sms = sms;
    p->split = false;
    p->c = row_cfg(D, dtype, kind == kFwd);
    // A ring needs two rounds; rows too wide for two rounds in kRingLimit load into registers,
    // except fp32 backward rows, which take the split form.
    p->ring = 2 * ring_round_bytes(kind, p->c, kRingBulk) + kRingHeader <= kRingLimit ? kRingBulk : kRingNone;
    if (kind == kBwd && p->ring == kRingNone && dtype == ADALN_F32 && split_plan(D, varlen, dev, R, p))
        return true;
    p->full = p->ring && p->c.full;
    if (!ring_shape(kind, dtype, varlen, dev, p)) return false;
    RowCfg copy;
    if (kind == kFwd && p->ring == kRingBulk && copy_ring_cfg(D, dtype, &copy) && R >= kCopyRingRows * p->G) {
        if (2 * ring_round_bytes(kind, copy, kRingCopy) + kRingHeader <= kRingLimit) {
            p->c = copy;
            p->ring = kRingCopy;
            p->full = copy.full;
            if (!ring_shape(kind, dtype, varlen, dev, p)) return false;
        }
    }
    // Bulk-ring forwards of more than one warp a CTA launch two tiles per resident CTA slot:
    // slots whose first tile finishes early take a second one, which evens out the uneven
    // finish of a single wave (bf16 D=5120: 116.3 -> 114.4 us; D=3072, 32,760 rows:
    // 68.1 -> 67.2 us). One-warp CTAs are faster in a single wave.
    if (kind == kFwd && p->ring == kRingBulk && p->c.tpb > 32) p->G = std::min<int64_t>(2 * p->G, kMaxCtas);
    if (p->G > R) p->G = R;
    if (p->G < 1) p->G = 1;
    return true;
}

// Layout of the backward's partials (see BwdArgs): vector-major where the modulation rows
// have at least kVecMajorPieces pieces each on average ((G + nseg) / nmod: every tile and
// every segment boundary inside a tile starts a piece), so that stage 2 reads each vector's
// pieces as one run; row-major where they have fewer, so that it reads each piece as one
// contiguous row (the packed D=3072 workload, ~1.5 pieces a row: 27 us for stage 2 against
// 46 us vector-major; bf16 D=1536 on 32,760 rows, 609 pieces: 94.8 us a step against 99.3).
constexpr int64_t kVecMajorPieces = 8;
int64_t pieces_per_row(int64_t G, int64_t nseg, int64_t nmod) {
    return (G + nseg + nmod - 1) / std::max<int64_t>(1, nmod);
}

// Vector-major stage 2: threads sharing one vector, the fewest powers of two that leave each
// at most 4 of a row's pieces, up to the whole CTA.
int stage2_splits(int64_t per_row) {
    int splits = 1;
    while (splits < kStage2Threads && (int64_t)splits * 4 < per_row) splits *= 2;
    return splits;
}

// float4 columns per stage-2 CTA: aim for ~2 CTAs per SM over all modulation rows.
int stage2_cw(int64_t D, int64_t nmod, int sms) {
    const int64_t D4 = D / 4;
    const int64_t target = 2 * (int64_t)sms;
    const int64_t ranges = (target + nmod - 1) / (nmod > 0 ? nmod : 1);
    const int64_t per = (D4 + ranges - 1) / ranges;
    int cw = 1;
    while ((int64_t)cw * 2 <= per && cw * 2 <= kStage2Threads) cw *= 2;
    return cw;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int64_t D, adaln_dtype dtype) {
    if (dtype != ADALN_F32 && dtype != ADALN_BF16) return ADALN_ERR_INVALID_ARG;
    if (D < 8 || D > 16384 || D % 8 != 0) return ADALN_ERR_UNSUPPORTED;
    return ADALN_OK;
}

bool rows_fit(int64_t R, int64_t D) { return R >= 0 && R <= (INT64_MAX / 16) / D; }

// Row tensors and modulation tables: present and 16-byte aligned.
int check_io(std::initializer_list<const void*> vecs, std::initializer_list<const void*> stats) {
    for (const void* p : vecs) {
        if (!p) return ADALN_ERR_INVALID_ARG;
        if (!aligned(p, 16)) return ADALN_ERR_ALIGNMENT;
    }
    for (const void* p : stats) {
        if (!p) return ADALN_ERR_INVALID_ARG;
        if (!aligned(p, 4)) return ADALN_ERR_ALIGNMENT;
    }
    return ADALN_OK;
}

int check_workspace(const void* ws, size_t bytes, size_t need) {
    if (!ws) return ADALN_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return ADALN_ERR_ALIGNMENT;
    if (bytes < need) return ADALN_ERR_WORKSPACE;
    return ADALN_OK;
}

size_t bwd_need(int64_t G, int64_t nseg, int64_t D) {
    return kPartialsOffset + (size_t)(G + nseg) * 2 * (size_t)D * sizeof(float);
}

int launched(cudaError_t e) { return e == cudaSuccess ? ADALN_OK : ADALN_ERR_CUDA; }

Segments dense_segments(int64_t Bt, int64_t N) {
    return Segments{nullptr, nullptr, Bt, N, Bt, Bt * N};
}

Segments packed_segments(const int32_t* cu, const int32_t* mod, int32_t nseg, int64_t total,
                         int64_t nmod) {
    return Segments{cu, mod, nseg, 0, nmod, total};
}

// Synchronises `stream`, then ORs the per-CTA status words a kernel left in `ws` (see
// adaln_read_status).
int read_status_words(const void* ws, cudaStream_t stream) {
    if (!ws) return ADALN_ERR_WORKSPACE;
    WsHeader h{};
    if (cudaMemcpyAsync(&h, ws, sizeof h, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return ADALN_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ADALN_ERR_CUDA;
    if (h.magic != kStatusMagic || h.nwords == 0 || h.nwords > (uint32_t)kMaxCtas)
        return ADALN_ERR_WORKSPACE;
    std::vector<uint32_t> words(h.nwords);
    if (cudaMemcpyAsync(words.data(), static_cast<const char*>(ws) + kHeaderBytes,
                        sizeof(uint32_t) * words.size(), cudaMemcpyDeviceToHost,
                        stream) != cudaSuccess)
        return ADALN_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ADALN_ERR_CUDA;
    uint32_t all = 0;
    for (uint32_t w : words) all |= w;
    if (all & kErrSeqlens) return ADALN_ERR_BAD_SEQLENS;
    if (all & kErrModIdx) return ADALN_ERR_BAD_MOD_IDX;
    if (all & kErrTimeout) return ADALN_ERR_TIMEOUT;
    return ADALN_OK;
}

// ---- shared bodies of the dense and packed calls -----------------------------------------

int run_fwd(const void* x, const void* shift, const void* scale, void* y, float* mean,
            float* rstd, const Segments& seg, int64_t D, float eps, void* ws, bool varlen,
            adaln_dtype dtype, cudaStream_t stream) {
    Plan p;
    if (!make_plan(kFwd, dtype, D, varlen, seg.R, &p)) return ADALN_ERR_CUDA;
    FwdArgs a{};
    a.x = x;
    a.shift = shift;
    a.scale = scale;
    a.y = y;
    a.mean = mean;
    a.rstd = rstd;
    a.D = D;
    a.eps = eps;
    a.seg = seg;
    a.status = ws ? reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + kHeaderBytes) : nullptr;
    a.header = static_cast<WsHeader*>(ws);
    a.stages = p.stages;
    return launched(
        launch_fwd(a, (int)dtype, p.c.nv, varlen, p.ring, p.full, p.G, p.c.tpb, p.smem, stream));
}

int64_t bwd_tiles(int64_t R, int64_t D, bool varlen, adaln_dtype dtype) {
    Plan p;
    if (!make_plan(kBwd, dtype, D, varlen, R, &p)) return -1;
    return p.G;
}

enum Stages { kPartials = 1, kReduce = 2, kBoth = 3 };

int run_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
            const void* scale, void* dx, float* dshift, float* dscale, const Segments& seg,
            int64_t D, void* ws, size_t ws_bytes, bool varlen, adaln_dtype dtype,
            cudaStream_t stream, int stages) {
    if (int rc = check_workspace(ws, ws_bytes, kPartialsOffset)) return rc;
    Plan p;
    if (!make_plan(kBwd, dtype, D, varlen, seg.R, &p)) return ADALN_ERR_CUDA;
    const int64_t G = p.G;
    const int64_t tiles = p.split ? G / 2 : G;
    if (int rc = check_workspace(ws, ws_bytes, bwd_need(G, seg.nseg, D))) return rc;
    char* base = static_cast<char*>(ws);
    BwdArgs a{};
    a.dy = dy;
    a.x = x;
    a.mean = mean;
    a.rstd = rstd;
    a.scale = scale;
    a.dx = dx;
    a.partials = reinterpret_cast<float*>(base + kPartialsOffset);
    const int64_t per_row = pieces_per_row(tiles, seg.nseg, seg.nmod);
    a.vec_major = per_row >= kVecMajorPieces ? 1 : 0;
    a.D = D;
    a.seg = seg;
    a.status = reinterpret_cast<uint32_t*>(base + kHeaderBytes);
    a.header = reinterpret_cast<WsHeader*>(base);
    a.stages = p.stages;
    if (stages & kPartials) {
        if (int rc = launched(launch_bwd(a, (int)dtype, p.c.nv, varlen, p.ring != kRingNone, p.full, G, p.c.tpb,
                                         p.smem, p.split, stream)))
            return rc;
    }
    if (!(stages & kReduce) || seg.nmod == 0) return ADALN_OK;
    Stage2Args s{};
    s.partials = a.partials;
    s.dshift = dshift;
    s.dscale = dscale;
    s.D = D;
    s.G = tiles;
    s.S = tiles + seg.nseg;
    s.vec_major = a.vec_major;
    s.cw = stage2_cw(D, seg.nmod, p.sms);
    s.splits = stage2_splits(per_row);
    s.seg = seg;
    return launched(launch_stage2(s, (int)dtype, varlen, p.sms, stream));
}

}  // namespace

extern "C" {

int adaln_fwd(const void* x, const void* shift, const void* scale, void* y, float* mean,
              float* rstd, int64_t Bt, int64_t N, int64_t D, float eps, adaln_dtype dtype,
              cudaStream_t stream) {
    if (int rc = check_shape(D, dtype)) return rc;
    if (Bt < 0 || N < 0 || !(eps > 0.0f) || !std::isfinite(eps)) return ADALN_ERR_INVALID_ARG;
    if (N > 0 && Bt > INT64_MAX / N) return ADALN_ERR_INVALID_ARG;
    const int64_t R = Bt * N;
    if (!rows_fit(R, D)) return ADALN_ERR_INVALID_ARG;
    if (R == 0) return ADALN_OK;
    if (int rc = check_io({x, shift, scale, y}, {mean, rstd})) return rc;
    return run_fwd(x, shift, scale, y, mean, rstd, dense_segments(Bt, N), D, eps, nullptr, false,
                   dtype, stream);
}

size_t adaln_bwd_workspace_size(int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype) {
    if (check_shape(D, dtype) || Bt < 0 || N < 0) return 0;
    if (N > 0 && Bt > INT64_MAX / N) return 0;
    const int64_t G = bwd_tiles(Bt * N, D, false, dtype);
    if (G < 0) return 0;
    return bwd_need(G, Bt, D);
}

}  // extern "C"

static int bwd_dense(const void* dy, const void* x, const float* mean, const float* rstd,
              const void* scale, void* dx, float* dshift, float* dscale, void* workspace,
              size_t workspace_bytes, int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype,
              cudaStream_t stream, int stages) {
    if (int rc = check_shape(D, dtype)) return rc;
    if (Bt < 0 || N < 0) return ADALN_ERR_INVALID_ARG;
    if (N > 0 && Bt > INT64_MAX / N) return ADALN_ERR_INVALID_ARG;
    const int64_t R = Bt * N;
    if (!rows_fit(R, D)) return ADALN_ERR_INVALID_ARG;
    if (Bt == 0) return ADALN_OK;
    if (int rc = check_io({dshift, dscale}, {})) return rc;
    if (R > 0) {
        if (int rc = check_io({dy, x, scale, dx}, {mean, rstd})) return rc;
    }
    return run_bwd(dy, x, mean, rstd, scale, dx, dshift, dscale, dense_segments(Bt, N), D,
                   workspace, workspace_bytes, false, dtype, stream, stages);
}

extern "C" {

int adaln_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
              const void* scale, void* dx, float* dshift, float* dscale, void* workspace,
              size_t workspace_bytes, int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype,
              cudaStream_t stream) {
    return bwd_dense(dy, x, mean, rstd, scale, dx, dshift, dscale, workspace, workspace_bytes, Bt, N,
                     D, dtype, stream, kBoth);
}

int adaln_bwd_partials(const void* dy, const void* x, const float* mean, const float* rstd,
                       const void* scale, void* dx, float* dshift, float* dscale, void* workspace,
                       size_t workspace_bytes, int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype,
                       cudaStream_t stream) {
    return bwd_dense(dy, x, mean, rstd, scale, dx, dshift, dscale, workspace, workspace_bytes, Bt, N,
                     D, dtype, stream, kPartials);
}

int adaln_bwd_reduce(const void* dy, const void* x, const float* mean, const float* rstd,
                     const void* scale, void* dx, float* dshift, float* dscale, void* workspace,
                     size_t workspace_bytes, int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype,
                     cudaStream_t stream) {
    return bwd_dense(dy, x, mean, rstd, scale, dx, dshift, dscale, workspace, workspace_bytes, Bt, N,
                     D, dtype, stream, kReduce);
}

size_t adaln_fwd_varlen_workspace_size(int64_t total_tokens, int32_t nseg, int64_t D,
                                       adaln_dtype dtype) {
    if (check_shape(D, dtype) || total_tokens < 0 || nseg < 0) return 0;
    return kPartialsOffset;
}

int adaln_fwd_varlen(const void* x, const void* shift, const void* scale, void* y, float* mean,
                     float* rstd, const int32_t* cu_seqlens, const int32_t* mod_idx, int32_t nseg,
                     int64_t total_tokens, int64_t nmod, int64_t D, float eps, void* workspace,
                     size_t workspace_bytes, adaln_dtype dtype, cudaStream_t stream) {
    if (int rc = check_shape(D, dtype)) return rc;
    if (nseg < 0 || total_tokens < 0 || total_tokens > INT32_MAX || nmod < 0)
        return ADALN_ERR_INVALID_ARG;
    if (!(eps > 0.0f) || !std::isfinite(eps)) return ADALN_ERR_INVALID_ARG;
    if (!rows_fit(total_tokens, D) || !rows_fit(nmod, D)) return ADALN_ERR_INVALID_ARG;
    if (!cu_seqlens || (nseg > 0 && !mod_idx)) return ADALN_ERR_INVALID_ARG;
    if (nseg == 0 && total_tokens > 0) return ADALN_ERR_INVALID_ARG;
    if (int rc = check_workspace(workspace, workspace_bytes, kPartialsOffset)) return rc;
    if (total_tokens > 0) {
        if (int rc = check_io({x, y}, {mean, rstd})) return rc;
        if (nmod > 0) {
            if (int rc = check_io({shift, scale}, {})) return rc;
        }
    }
    return run_fwd(x, shift, scale, y, mean, rstd,
                   packed_segments(cu_seqlens, mod_idx, nseg, total_tokens, nmod), D, eps,
                   workspace, true, dtype, stream);
}

size_t adaln_bwd_varlen_workspace_size(int64_t total_tokens, int32_t nseg, int64_t nmod,
                                       int64_t D, adaln_dtype dtype) {
    if (check_shape(D, dtype) || total_tokens < 0 || nseg < 0 || nmod < 0) return 0;
    const int64_t G = bwd_tiles(total_tokens, D, true, dtype);
    if (G < 0) return 0;
    return bwd_need(G, nseg, D);
}

}  // extern "C"

static int bwd_packed(const void* dy, const void* x, const float* mean, const float* rstd,
                     const void* scale, void* dx, float* dshift, float* dscale,
                     const int32_t* cu_seqlens, const int32_t* mod_idx, int32_t nseg,
                     int64_t total_tokens, int64_t nmod, int64_t D, void* workspace,
                     size_t workspace_bytes, adaln_dtype dtype, cudaStream_t stream, int stages) {
    if (int rc = check_shape(D, dtype)) return rc;
    if (nseg < 0 || total_tokens < 0 || total_tokens > INT32_MAX || nmod < 0)
        return ADALN_ERR_INVALID_ARG;
    if (!rows_fit(total_tokens, D) || !rows_fit(nmod, D)) return ADALN_ERR_INVALID_ARG;
    if (!cu_seqlens || (nseg > 0 && !mod_idx)) return ADALN_ERR_INVALID_ARG;
    if (nseg == 0 && total_tokens > 0) return ADALN_ERR_INVALID_ARG;
    if (nmod > 0) {
        if (int rc = check_io({dshift, dscale}, {})) return rc;
    }
    if (total_tokens > 0) {
        if (int rc = check_io({dy, x, dx}, {mean, rstd})) return rc;
        if (nmod > 0) {
            if (int rc = check_io({scale}, {})) return rc;
        }
    }
    return run_bwd(dy, x, mean, rstd, scale, dx, dshift, dscale,
                   packed_segments(cu_seqlens, mod_idx, nseg, total_tokens, nmod), D, workspace,
                   workspace_bytes, true, dtype, stream, stages);
}

extern "C" {

int adaln_bwd_varlen(const void* dy, const void* x, const float* mean, const float* rstd,
                     const void* scale, void* dx, float* dshift, float* dscale,
                     const int32_t* cu_seqlens, const int32_t* mod_idx, int32_t nseg,
                     int64_t total_tokens, int64_t nmod, int64_t D, void* workspace,
                     size_t workspace_bytes, adaln_dtype dtype, cudaStream_t stream) {
    return bwd_packed(dy, x, mean, rstd, scale, dx, dshift, dscale, cu_seqlens, mod_idx, nseg,
                      total_tokens, nmod, D, workspace, workspace_bytes, dtype, stream, kBoth);
}

int adaln_bwd_varlen_partials(const void* dy, const void* x, const float* mean, const float* rstd,
                     const void* scale, void* dx, float* dshift, float* dscale,
                     const int32_t* cu_seqlens, const int32_t* mod_idx, int32_t nseg,
                     int64_t total_tokens, int64_t nmod, int64_t D, void* workspace,
                     size_t workspace_bytes, adaln_dtype dtype, cudaStream_t stream) {
    return bwd_packed(dy, x, mean, rstd, scale, dx, dshift, dscale, cu_seqlens, mod_idx, nseg,
                      total_tokens, nmod, D, workspace, workspace_bytes, dtype, stream, kPartials);
}

int adaln_bwd_varlen_reduce(const void* dy, const void* x, const float* mean, const float* rstd,
                     const void* scale, void* dx, float* dshift, float* dscale,
                     const int32_t* cu_seqlens, const int32_t* mod_idx, int32_t nseg,
                     int64_t total_tokens, int64_t nmod, int64_t D, void* workspace,
                     size_t workspace_bytes, adaln_dtype dtype, cudaStream_t stream) {
    return bwd_packed(dy, x, mean, rstd, scale, dx, dshift, dscale, cu_seqlens, mod_idx, nseg,
                      total_tokens, nmod, D, workspace, workspace_bytes, dtype, stream, kReduce);
}

int adaln_read_status(const void* workspace, cudaStream_t stream) {
    return read_status_words(workspace, stream);
}

int64_t adaln_bucket_batch(int64_t S, int64_t M_mem, int64_t M_comp, int32_t p) {
    if (S <= 0 || M_mem <= 0 || M_comp <= 0 || p < 1) return -(int64_t)ADALN_ERR_INVALID_ARG;
    const int64_t by_memory = M_mem / S;
    // floor(M_comp / S^p) as p nested floor divisions: floor(floor(a/b)/c) == floor(a/(b*c))
    // for positive integers, so S^p is never formed and nothing can overflow.
    int64_t by_compute = M_comp;
    for (int32_t i = 0; i < p && by_compute > 0; ++i) by_compute /= S;
    const int64_t b = by_memory < by_compute ? by_memory : by_compute;
    return b > 1 ? b : 1;
}

const char* adaln_status_string(int status) {
    switch (status) {
        case ADALN_OK: return "ADALN_OK";
        case ADALN_ERR_INVALID_ARG: return "ADALN_ERR_INVALID_ARG: invalid argument";
        case ADALN_ERR_UNSUPPORTED: return "ADALN_ERR_UNSUPPORTED: D must be a multiple of 8 in [8, 16384]";
        case ADALN_ERR_ALIGNMENT: return "ADALN_ERR_ALIGNMENT: misaligned pointer";
        case ADALN_ERR_WORKSPACE: return "ADALN_ERR_WORKSPACE: workspace missing, too small or without status";
        case ADALN_ERR_CUDA: return "ADALN_ERR_CUDA: CUDA runtime error";
        case ADALN_ERR_BAD_SEQLENS: return "ADALN_ERR_BAD_SEQLENS: malformed cu_seqlens";
        case ADALN_ERR_BAD_MOD_IDX: return "ADALN_ERR_BAD_MOD_IDX: mod_idx out of range";
        case ADALN_ERR_TIMEOUT: return "ADALN_ERR_TIMEOUT: a kernel timed out waiting for its input copies";
        default: return "unknown adaln status";
    }
}

}  // extern "C"

// ---- Backward without saved statistics ---------------------------------------------------
// The statistics are recomputed by stats_kernel (csrc/fwd.cu) with the forward's row mapping
// and arithmetic, so bitwise the statistics the forward computed, into a region after the
// backward's own workspace; then the backward runs as usual.

namespace {

size_t recompute_stats_offset(int64_t G, int64_t nseg, int64_t D) {
    return (bwd_need(G, nseg, D) + 255) / 256 * 256;
}

size_t bwd_recompute_workspace(int64_t R, int64_t nseg, int64_t D, bool varlen, adaln_dtype dtype) {
    const int64_t G = bwd_tiles(R, D, varlen, dtype);
    if (G < 0) return 0;
    return recompute_stats_offset(G, nseg, D) + (size_t)R * 2 * sizeof(float);
}

int bwd_recompute(const void* dy, const void* x, const void* scale, void* dx, float* dshift,
                  float* dscale, const Segments& seg, int64_t D, float eps, void* ws, size_t ws_bytes,
                  bool varlen, adaln_dtype dtype, cudaStream_t stream) {
    if (!(eps > 0.0f) || !std::isfinite(eps)) return ADALN_ERR_INVALID_ARG;
    if (int rc = check_workspace(ws, ws_bytes, kPartialsOffset)) return rc;
    const int64_t G = bwd_tiles(seg.R, D, varlen, dtype);
    if (G < 0) return ADALN_ERR_CUDA;
    const size_t off = recompute_stats_offset(G, seg.nseg, D);
    if (int rc = check_workspace(ws, ws_bytes, off + (size_t)seg.R * 2 * sizeof(float))) return rc;
    float* mean = reinterpret_cast<float*>(static_cast<char*>(ws) + off);
    float* rstd = mean + seg.R;
    if (seg.R > 0) {
        Plan f;  // the forward's row mapping for these rows
        if (!make_plan(kFwd, dtype, D, varlen, seg.R, &f)) return ADALN_ERR_CUDA;
        if (int rc = launched(launch_stats(x, mean, rstd, seg.R, D, eps, (int)dtype, f.c.nv, f.c.tpb,
                                           std::min<int64_t>(f.G, seg.R), stream)))
            return rc;
    }
    return run_bwd(dy, x, mean, rstd, scale, dx, dshift, dscale, seg, D, ws, ws_bytes, varlen, dtype,
                   stream, kBoth);
}

}  // namespace

extern "C" {

size_t adaln_bwd_recompute_workspace_size(int64_t Bt, int64_t N, int64_t D, adaln_dtype dtype) {
    if (check_shape(D, dtype) || Bt < 0 || N < 0) return 0;
    if (N > 0 && Bt > INT64_MAX / N) return 0;
    return bwd_recompute_workspace(Bt * N, Bt, D, false, dtype);
}

int adaln_bwd_recompute(const void* dy, const void* x, const void* scale, void* dx, float* dshift,
                        float* dscale, void* workspace, size_t workspace_bytes, int64_t Bt, int64_t N,
                        int64_t D, float eps, adaln_dtype dtype, cudaStream_t stream) {
    if (int rc = check_shape(D, dtype)) return rc;
    if (Bt < 0 || N < 0) return ADALN_ERR_INVALID_ARG;
    if (N > 0 && Bt > INT64_MAX / N) return ADALN_ERR_INVALID_ARG;
    const int64_t R = Bt * N;
    if (!rows_fit(R, D)) return ADALN_ERR_INVALID_ARG;
    if (Bt == 0) return ADALN_OK;
    if (int rc = check_io({dshift, dscale}, {})) return rc;
    if (R > 0) {
        if (int rc = check_io({dy, x, scale, dx}, {})) return rc;
    }
    return bwd_recompute(dy, x, scale, dx, dshift, dscale, dense_segments(Bt, N), D, eps, workspace,
                         workspace_bytes, false, dtype, stream);
}

size_t adaln_bwd_varlen_recompute_workspace_size(int64_t total_tokens, int32_t nseg, int64_t nmod,
                                                 int64_t D, adaln_dtype dtype) {
    if (check_shape(D, dtype) || total_tokens < 0 || nseg < 0 || nmod < 0) return 0;
    return bwd_recompute_workspace(total_tokens, nseg, D, true, dtype);
}

int adaln_bwd_varlen_recompute(const void* dy, const void* x, const void* scale, void* dx,
                               float* dshift, float* dscale, const int32_t* cu_seqlens,
                               const int32_t* mod_idx, int32_t nseg, int64_t total_tokens, int64_t nmod,
                               int64_t D, float eps, void* workspace, size_t workspace_bytes,
                               adaln_dtype dtype, cudaStream_t stream) {
    if (int rc = check_shape(D, dtype)) return rc;
    if (nseg < 0 || total_tokens < 0 || total_tokens > INT32_MAX || nmod < 0)
        return ADALN_ERR_INVALID_ARG;
    if (!rows_fit(total_tokens, D) || !rows_fit(nmod, D)) return ADALN_ERR_INVALID_ARG;
    if (!cu_seqlens || (nseg > 0 && !mod_idx)) return ADALN_ERR_INVALID_ARG;
    if (nseg == 0 && total_tokens > 0) return ADALN_ERR_INVALID_ARG;
    if (nmod > 0) {
        if (int rc = check_io({dshift, dscale}, {})) return rc;
    }
    if (total_tokens > 0) {
        if (int rc = check_io({dy, x, dx}, {})) return rc;
        if (nmod > 0) {
            if (int rc = check_io({scale}, {})) return rc;
        }
    }
    return bwd_recompute(dy, x, scale, dx, dshift, dscale,
                         packed_segments(cu_seqlens, mod_idx, nseg, total_tokens, nmod), D, eps,
                         workspace, workspace_bytes, true, dtype, stream);
}

}  // extern "C"

// ---- dense backward without a caller workspace ---------------------------------------------
//
// Some callers cannot allocate device memory at the point where they run the backward: a
// host framework that hands out only the tensors it owns, code running under an allocator
// that must not grow, or a plain C caller with no allocator at all. For them the backward's
// scratch (status words and per-tile partials) lives in one fixed array that is part of
// this module: every GPU that loads the library holds ADALN_NOALLOC_SCRATCH_BYTES of it
// until the process exits.

static __device__ __align__(256) unsigned char g_noalloc_scratch[ADALN_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// The array's device address on the current device. In host code the array's name only
// stands in for the symbol, so the address must come from the runtime, once per device,
// with that device current.
int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ADALN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return ADALN_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return ADALN_OK;
}

}  // namespace

extern "C" int adaln_bwd_noalloc(const void* dy, const void* x, const float* mean,
                                 const float* rstd, const void* scale, void* dx, float* dshift,
                                 float* dscale, int64_t Bt, int64_t N, int64_t D,
                                 adaln_dtype dtype, cudaStream_t stream) {
    // The scratch needs no clearing: every call writes each status word and each partial it
    // later reads.
    if (int rc = check_shape(D, dtype)) return rc;
    if (Bt < 0 || N < 0) return ADALN_ERR_INVALID_ARG;
    if (Bt == 0) return ADALN_OK;
    void* scratch = nullptr;
    if (int rc = noalloc_scratch(&scratch)) return rc;
    // bwd_dense returns ADALN_ERR_WORKSPACE, before launching anything, when the problem
    // needs more scratch than the fixed array holds.
    return bwd_dense(dy, x, mean, rstd, scale, dx, dshift, dscale, scratch,
                     (size_t)ADALN_NOALLOC_SCRATCH_BYTES, Bt, N, D, dtype, stream, kBoth);
}

// The status words of the last adaln_bwd_noalloc on the current device sit at the head of
// the fixed array, exactly where a caller workspace holds them.
extern "C" int adaln_noalloc_read_status(cudaStream_t stream) {
    void* scratch = nullptr;
    if (int rc = noalloc_scratch(&scratch)) return rc;
    return read_status_words(scratch, stream);
}

// ---- row sharding across ranks: the fixed-order sum of the gradients --------------------

extern "C" int adaln_sum_ranks(const float* parts, float* out, int32_t world, int64_t n,
                               cudaStream_t stream) {
    if (world < 1 || n < 0) return ADALN_ERR_INVALID_ARG;
    if (n == 0) return ADALN_OK;
    if (n > INT64_MAX / world) return ADALN_ERR_INVALID_ARG;
    if (int rc = check_io({parts, out}, {})) return rc;
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms <= 0) return ADALN_ERR_CUDA;
    return launched(launch_rank_sum(parts, out, world, n, sms, stream));
}

extern "C" int adaln_debug_read(uint32_t* word, int reset) {
#ifdef ADALN_DEBUG
    if (word == nullptr) return ADALN_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return ADALN_ERR_CUDA;
    uint32_t f = 0, b = 0;
    if (debug_word_fwd(&f, reset != 0) != cudaSuccess || debug_word_bwd(&b, reset != 0) != cudaSuccess)
        return ADALN_ERR_CUDA;
    *word = f | b;
    return ADALN_OK;
#else
    (void)word;
    (void)reset;
    return ADALN_ERR_UNSUPPORTED;
#endif
}
