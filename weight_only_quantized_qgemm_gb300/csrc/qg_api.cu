// C ABI of libqgemm: argument validation, the per-shape dispatch table,
// tensor-map encoding, the device status word, the test-aid kernels (the
// FP8 activation split, the LUT3 dequantiser) and the offline LUT3 packer.
// See include/qgemm.h for the contract.
#include <atomic>
#include <cstring>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/qgemm.h"
#include "qg_gemm.cuh"
#include "qg_internal.h"
#include "qg_w8a8.h"

namespace qg {

__device__ uint32_t g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_timeout_ns{1000000000ull};
std::atomic<int> g_fault_unit{-1};
std::atomic<int> g_overlap{0};

struct DeviceInfo {
    std::once_flag once;
    int sms = 0;
    uint32_t* status = nullptr;
    cudaError_t err = cudaSuccess;
};
DeviceInfo g_dev[kMaxDevices];

// Per-device setup: SM count and the device address of the status word.
DeviceInfo* device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceInfo* d = &g_dev[dev];
    std::call_once(d->once, [d, dev]() {
        d->err = cudaDeviceGetAttribute(&d->sms, cudaDevAttrMultiProcessorCount, dev);
        if (d->err == cudaSuccess)
            d->err = cudaGetSymbolAddress(reinterpret_cast<void**>(&d->status), g_status_word);
    });
    return d->err == cudaSuccess ? d : nullptr;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D row-major tensor map: `rows` x `cols` elements, row stride `ld_bytes`,
// box `box_cols` x `box_rows`, 128-byte swizzle, out-of-range reads as zero.
bool make_tmap(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, uint64_t cols, uint64_t rows,
               uint64_t ld_bytes, uint32_t box_cols, uint32_t box_rows,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

LaunchCtl launch_ctl(const DeviceInfo* d) {
    LaunchCtl c;
    c.timeout_ns = g_timeout_ns.load();
    c.fault_unit = g_fault_unit.load();
    c.status = d->status;
    c.num_sms = d->sms;
    c.overlap = g_overlap.load() != 0;
    return c;
}

}  // namespace

bool overlap_enabled() { return g_overlap.load() != 0; }

namespace {

// ----------------------------------------------------------------- dispatch
// Per-(kind, M, N, K) choice of MMA width and grid.  The MMA N side is 16 for
// M <= 16 and 32 above (one weight pass for every M <= 32).  The grid comes
// from the dispatch table when it holds an entry for the shape (set by a
// caller, e.g. after measuring candidates), else from a cost rule.  When the
// tiles fit on the SMs it weighs two grids by the work units (128 rows x
// 128 K) of their busiest CTA:
//  - one CTA per 128-row tile: no tile is split, so no partial sums and no
//    reduction;
//  - k CTAs per tile, k the largest whole number with k x tiles <= SMs, at
//    most kMaxPiecesPerTile: the units split evenly, every tile into k
//    pieces of equal size.  (The tuner's picks on the attention and down
//    shapes were all such whole multiples: 3 per tile at 40 and 48 tiles, 8
//    at 8 tiles.)  A split tile costs the CTA that finishes it a partial-sum
//    store, an arrival atomic and the reduction, at the end of the kernel;
//    that tail measured about as long as kSplitCostUnits units of steady
//    streaming;
//  - where a unit's on-chip work rather than HBM sets the pace (the FP8
//    kernel at 17-32 rows, whose activation split doubles, and W8A8), also
//    one CTA per SM with the units split evenly, whose pieces straddle tile
//    boundaries: kStraddleCostUnits more (on down at 32 rows, 152 CTAs ran
//    25.5 us against 27.4 at 120; on the 5120 x 5120 shape 14.4 against 13.2).
// Ties go to the grid without splits, then to whole multiples.  More tiles
// than SMs: stream-K, one CTA per SM, unless whole tiles divide evenly over
// a grid (the largest divisor of the tile count up to the SM count) whose
// busiest CTA costs fewer units than stream-K's plus its split and straddle
// tails (W8A8 at 256 rows: 136 CTAs of two whole tiles ran 36.5 us against
// 41.1 us for stream-K over 152; the BF16 lm_head shape, 256 tiles, 50.2
// against 52.1 us on 128 CTAs).
constexpr int kMaxPiecesPerTile = 8;
constexpr long long kSplitCostUnits = 10;
constexpr long long kStraddleCostUnits = 5;

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

bool splits(long long U, int KU, int G) {
    for (int c = 0; c <= G; ++c) {
        const long long b = static_cast<long long>(c) * U / G;
        if (b % KU != 0) return true;
    }
    return false;
}

// The dispatch table: process-wide, shared by all devices and threads.  A
// generation counter tells the per-thread schedule caches to look again.
struct TableEntry {
    int kind, M, N, K, ctas;
};
std::mutex g_table_mu;
TableEntry g_table[256];
int g_table_n = 0;
std::atomic<uint64_t> g_table_gen{1};

int table_lookup(int kind, int M, int N, int K) {
    std::lock_guard<std::mutex> lk(g_table_mu);
    for (int i = 0; i < g_table_n; ++i) {
        const TableEntry& e = g_table[i];
        if (e.kind == kind && e.M == M && e.N == N && e.K == K) return e.ctas;
    }
    return 0;
}

// The schedule of a shape on `sms` SMs, with `forced` > 0 a dispatch-table grid.
Schedule schedule_for(int kind, int M, int N, int K, int sms, int forced) {
    Schedule s;
    s.nmma = kind == QG_KIND_W8A8 ? w8a8_tile_rows(M) : M <= 16 ? 16 : 32;
    // W8A8 tiles are 128 weight rows x nmma activation rows, weight-tile-major
    s.T = (N + 127) / 128 * (kind == QG_KIND_W8A8 ? (M + s.nmma - 1) / s.nmma : 1);
    // one unit = 128 rows x one 128-wide K block (W8A8: two blocks)
    s.KU = kind == QG_KIND_W8A8 ? (K + 255) / 256 : (K + 127) / 128;
    s.U = static_cast<long long>(s.T) * s.KU;
    const bool unit_bound = kind == QG_KIND_W8A8 || (kind == QG_KIND_FP8_BLOCK && M > 16);
    long long g = sms;
    if (forced > 0) {
        g = forced;
        if (g > s.U) g = s.U;
    } else if (s.T <= sms) {
        auto cost_of = [&](long long G, long long extra) {
            return ceil_div(s.U, G) + (splits(s.U, s.KU, static_cast<int>(G)) ? kSplitCostUnits + extra : 0);
        };
        long long k = sms / s.T;
        if (k > kMaxPiecesPerTile) k = kMaxPiecesPerTile;
        long long gb = k * s.T;
        if (gb > s.U) gb = s.U;
        long long best = s.KU;   // one CTA per tile
        g = s.T;
        if (cost_of(gb, 0) < best) {
            best = cost_of(gb, 0);
            g = gb;
        }
        const long long gc = sms < s.U ? sms : s.U;
        if (unit_bound && gc != g && cost_of(gc, kStraddleCostUnits) < best) g = gc;
    } else {
        if (g > s.U) g = s.U;
        // with more tiles than SMs every stream-K piece straddles tiles
        const long long stream_cost =
            ceil_div(s.U, g) + (splits(s.U, s.KU, static_cast<int>(g)) ? kSplitCostUnits + kStraddleCostUnits : 0);
        for (long long d = sms; d >= 1; --d) {
            if (s.T % d != 0) continue;
            if (s.T / d * s.KU < stream_cost) g = d;
            break;
        }
    }
    s.G = static_cast<int>(g);
    s.max_ctas = sms > s.G ? sms : s.G;
    return s;
}

Schedule choose_schedule(int kind, int M, int N, int K, int sms) {
    return schedule_for(kind, M, N, K, sms, table_lookup(kind, M, N, K));
}

// True when some tile's units are spread over more than one CTA.
bool schedule_splits(const Schedule& s) { return splits(s.U, s.KU, s.G); }

// Per-thread caches of the last few schedules (keyed by kind, shape, SM
// count and dispatch-table generation) and weight tensor maps (keyed by
// address and shape, which determine the map): the schedule search walks
// every CTA boundary and the map encoding is a driver call, both otherwise
// paid on every GEMM call.
constexpr int kCacheWays = 8;

struct SchedEntry {
    int kind = -1, M = 0, N = 0, K = 0, sms = 0;
    uint64_t gen = 0;
    Schedule s;
    size_t ws = 0;
};

size_t workspace_bytes_uncached(const Schedule& s);

const SchedEntry& cached_schedule(int kind, int M, int N, int K, int sms) {
    thread_local SchedEntry cache[kCacheWays];
    thread_local int next = 0;
    const uint64_t gen = g_table_gen.load(std::memory_order_acquire);
    for (const SchedEntry& e : cache)
        if (e.kind == kind && e.M == M && e.N == N && e.K == K && e.sms == sms && e.gen == gen) return e;
    SchedEntry& e = cache[next];
    next = (next + 1) % kCacheWays;
    e.kind = kind;
    e.M = M;
    e.N = N;
    e.K = K;
    e.sms = sms;
    e.gen = gen;
    e.s = choose_schedule(kind, M, N, K, sms);
    e.ws = kind == QG_KIND_W8A8 ? w8a8_workspace_bytes(e.s, schedule_splits(e.s)) : workspace_bytes_uncached(e.s);
    return e;
}

// Tensor maps of operands that stay put between calls, keyed by what the map
// encodes (address, shape and kind).
enum MapKind { kMapFp8Weights = 0, kMapLut3Scales = 1, kMapBf16Weights = 2 };

// The largest M a kind accepts: the decode kernels take M <= 32 in one MMA;
// the W8A8 kernel tiles M in 32-row blocks.
constexpr int kMaxMW8a8 = 1 << 16;
int k_multiple(int kind) { return kind == QG_KIND_LUT3 ? 128 : kind == QG_KIND_BF16 ? 8 : 16; }

int max_m(int kind) {
    switch (kind) {
        case QG_KIND_FP8_BLOCK:
        case QG_KIND_LUT3:
        case QG_KIND_BF16: return 32;
        case QG_KIND_W8A8: return kMaxMW8a8;
    }
    return 0;
}

struct MapEntry {
    const void* ptr = nullptr;
    uint64_t cols = 0, rows = 0;
    int kind = -1;
    CUtensorMap map;
};

// The cached map of a [rows, cols] operand, encoded on a miss; null if the
// driver refused it.
//   kMapFp8Weights: E4M3 weights, 128 x 128 boxes, 128-byte swizzle.
//   kMapLut3Scales: FP16 LUT3 scales [N, K/128], boxes of 8 groups x 128 rows.
//   kMapBf16Weights: BF16 weights [N, K], 64 x 128 boxes, 128-byte swizzle.
const CUtensorMap* cached_tmap(const void* ptr, uint64_t cols, uint64_t rows, MapKind kind) {
    thread_local MapEntry cache[kCacheWays];
    thread_local int next = 0;
    for (MapEntry& e : cache)
        if (e.ptr == ptr && e.cols == cols && e.rows == rows && e.kind == kind) return &e.map;
    MapEntry& e = cache[next];
    const bool ok = kind == kMapFp8Weights
                        ? make_tmap(&e.map, ptr, CU_TENSOR_MAP_DATA_TYPE_UINT8, cols, rows, cols, 128, 128)
                    : kind == kMapBf16Weights
                        ? make_tmap(&e.map, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cols, rows, cols * 2, 64, 128)
                        : make_tmap(&e.map, ptr, CU_TENSOR_MAP_DATA_TYPE_UINT16, cols, rows, cols * 2, 8, 128,
                                    CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) {
        e.ptr = nullptr;
        return nullptr;
    }
    next = (next + 1) % kCacheWays;
    e.ptr = ptr;
    e.cols = cols;
    e.rows = rows;
    e.kind = kind;
    return &e.map;
}

}  // namespace

size_t workspace_partial_bytes(const Schedule& s) {
    return static_cast<size_t>(s.max_ctas) * 2 * 32 * 128 * sizeof(float);
}

namespace {
size_t workspace_bytes_uncached(const Schedule& s) {
    if (!schedule_splits(s)) return 0;
    const size_t cnt = (static_cast<size_t>(s.T) * 4 * sizeof(uint32_t) + 255) & ~static_cast<size_t>(255);
    return workspace_partial_bytes(s) + cnt;
}
}  // namespace

size_t workspace_bytes(const Schedule& s) { return workspace_bytes_uncached(s); }

void workspace_counters(int kind, int M, int N, int K, size_t* offset, size_t* bytes) {
    *offset = 0;
    *bytes = 0;
    DeviceInfo* d = device_info();
    if (!d || M <= 0 || N <= 0 || K <= 0) return;
    const SchedEntry& e = cached_schedule(kind, M, N, K, d->sms);
    const Schedule& s = e.s;
    const size_t total = e.ws;
    if (total == 0) return;
    *offset = kind == QG_KIND_W8A8 ? w8a8_partial_bytes(s) : workspace_partial_bytes(s);
    *bytes = total - *offset;
}

uint32_t* device_status_ptr() {
    DeviceInfo* d = device_info();
    return d ? d->status : nullptr;
}

// ----------------------------------------------------------------- small kernels
namespace {

// One warp per 128-element block of BF16 activations: the FP8 GEMM's
// activation split (block exponent from the largest |x|, then the hi/lo E4M3
// codes of every x * 2^e), through the device functions the GEMM's split
// warps use.  Lane l handles elements 4l .. 4l+3.
__global__ void split_probe_kernel(const uint2* __restrict__ x, int64_t blocks, uint32_t* __restrict__ hi,
                                   uint32_t* __restrict__ lo, int* __restrict__ exponent) {
    const int lane = threadIdx.x & 31;
    const int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (blk >= blocks) return;
    const uint2 v = x[blk * 32 + lane];
    uint32_t m2 = bf16x2_absmax(v.x, v.y) & 0x7FFF7FFFu;
    uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int e = split_exponent(mx);
    const uint32_t pw2 = bf16x2_pow2(e);
    uint32_t h, l;
    split_e4m3x4(bf16x2_mul(v.x, pw2), bf16x2_mul(v.y, pw2), h, l);
    hi[blk * 32 + lane] = h;
    lo[blk * 32 + lane] = l;
    if (lane == 0) exponent[blk] = e;
}

// One thread per (row, 8-code word) of the packed LUT3 layout.
__global__ void dequant_lut3_kernel(const uint8_t* __restrict__ Wq, const uint4* __restrict__ qmap,
                                    const uint16_t* __restrict__ scales, uint16_t* __restrict__ D, int N, int K) {
    const int KT = (K + 255) / 256;
    const int words_per_row = KT * 32;
    const int64_t total = static_cast<int64_t>(N) * words_per_row;
    const uint4 qm = __ldg(qmap);
    const int G128 = K / 128;
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(t / words_per_row);
        const int wi = static_cast<int>(t % words_per_row);
        const int k0 = wi * 8;
        const int tk = k0 / 256, qq = (k0 % 256) / 32, w = (k0 % 32) / 8;
        const size_t off = (static_cast<size_t>(n / 128) * KT + tk) * 16384 +
                           (static_cast<size_t>(qq) * 128 + (n % 128)) * 16 + w * 4;
        const uint32_t word = *reinterpret_cast<const uint32_t*>(Wq + off);
        const int g = k0 / 128;
        const uint32_t sc = g < G128 ? scales[static_cast<int64_t>(n) * G128 + g] : 0u;
        const uint32_t sc2 = sc | (sc << 16);
        const LutPlanes tp = lut_planes(f16x2_mul(qm.x, sc2), f16x2_mul(qm.y, sc2), f16x2_mul(qm.z, sc2),
                                        f16x2_mul(qm.w, sc2));
        uint32_t o[4];
        lut3x8_to_f16(word, tp, o);
        for (int e = 0; e < 8; ++e) {
            if (k0 + e < K) {
                const uint32_t pair = o[e >> 1];
                D[static_cast<int64_t>(n) * K + k0 + e] = static_cast<uint16_t>((e & 1) ? (pair >> 16) : (pair & 0xFFFFu));
            }
        }
    }
}

__global__ void zero_rows_kernel(uint16_t* Y, int64_t ldy, int M, int N) {
    const int64_t total = static_cast<int64_t>(M) * N;
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x)
        Y[(t / N) * ldy + (t % N)] = 0;
}

// One warp per CTA of a schedule: the CTA's unit range and its split-K
// bookkeeping (first and last contributing CTA and slot of its first and last
// tile), through the device functions the GEMM kernels use.
__global__ void schedule_probe_kernel(long long U, int G, int KB, long long* __restrict__ ranges,
                                      int* __restrict__ info) {
    const int cta = blockIdx.x;
    const int lane = threadIdx.x;
    gemm::Params p{};
    p.U = U;
    p.G = G;
    p.KB = KB;
    const long long u0 = gemm::unit_begin(cta, U, G);
    const long long u1 = gemm::unit_begin(cta + 1, U, G);
    const int v = gemm::split_info_lane(p, u0, u1, lane);
    if (lane == 0) {
        ranges[2 * cta] = u0;
        ranges[2 * cta + 1] = u1;
    }
    if (lane < 6) info[6 * cta + lane] = v;
}

int grid_for(int64_t work, int threads) {
    int64_t g = (work + threads - 1) / threads;
    if (g > 4096) g = 4096;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_split_probe(const void* X, int64_t blocks, void* hi, void* lo, int* exponent, cudaStream_t st) {
    const int64_t threads = blocks * 32;
    const int64_t grid = (threads + 255) / 256;
    split_probe_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(static_cast<const uint2*>(X), blocks,
                                                                    static_cast<uint32_t*>(hi),
                                                                    static_cast<uint32_t*>(lo), exponent);
    return cudaGetLastError();
}

cudaError_t launch_dequant_lut3(const void* Wq, const void* qmap, const void* scales, void* D, int N, int K,
                                cudaStream_t st) {
    const int64_t work = static_cast<int64_t>(N) * ((K + 255) / 256) * 32;
    dequant_lut3_kernel<<<grid_for(work, 256), 256, 0, st>>>(static_cast<const uint8_t*>(Wq),
                                                             static_cast<const uint4*>(qmap),
                                                             static_cast<const uint16_t*>(scales),
                                                             static_cast<uint16_t*>(D), N, K);
    return cudaGetLastError();
}

cudaError_t launch_zero_rows(void* Y, int64_t ldy, int M, int N, cudaStream_t st) {
    zero_rows_kernel<<<grid_for(static_cast<int64_t>(M) * N, 256), 256, 0, st>>>(static_cast<uint16_t*>(Y), ldy,
                                                                               M, N);
    return cudaGetLastError();
}

// Argument checks of the FP8 entry points, in the order the header lists the
// errors; M == 0 or N == 0 is valid (a no-op).
qg_status check_fp8_args(const void* X, int64_t ldx, const void* W, const void* W_scale, const void* Y, int64_t ldy,
                         int M, int N, int K) {
    if (M < 0 || N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return QG_OK;
    if (!X || !W || !W_scale || !Y) return QG_ERR_INVALID_ARG;
    if (M > 32 || K % 16 != 0) return QG_ERR_UNSUPPORTED_SHAPE;
    if (ldx < K || ldy < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W) || (ldx % 8) != 0) return QG_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(W_scale) & 3u) != 0 || (reinterpret_cast<uintptr_t>(Y) & 1u) != 0)
        return QG_ERR_MISALIGNED;
    return QG_OK;
}

}  // namespace qg

// =================================================================== C ABI
using namespace qg;

extern "C" {

size_t qg_workspace_bytes(int kind, int M, int N, int K) {
    if (M < 1 || N < 1 || K < 1 || M > max_m(kind)) return 0;
    DeviceInfo* d = device_info();
    if (!d) return 0;
    return cached_schedule(kind, M, N, K, d->sms).ws;
}

size_t qg_workspace_bytes_max(int N) {
    if (N < 1) return 0;
    DeviceInfo* d = device_info();
    if (!d) return 0;
    Schedule s;
    s.T = (N + 127) / 128;
    s.max_ctas = d->sms;
    const size_t cnt = (static_cast<size_t>(s.T) * 4 * sizeof(uint32_t) + 255) & ~static_cast<size_t>(255);
    return workspace_partial_bytes(s) + cnt;
}

size_t qg_workspace_bytes_max_w8a8(int M, int N) {
    if (M < 1 || M > kMaxMW8a8 || N < 1) return 0;
    DeviceInfo* d = device_info();
    if (!d) return 0;
    Schedule s;
    s.nmma = w8a8_tile_rows(M);
    s.T = (N + 127) / 128 * ((M + s.nmma - 1) / s.nmma);
    s.max_ctas = d->sms;
    s.U = 1;
    s.KU = 1;
    s.G = 2;   // any split schedule: the size does not depend on K or the grid
    return w8a8_workspace_bytes(s, true);
}

qg_status qgemm_fp8_block(const void* X, int64_t ldx, const uint8_t* W, const float* W_scale, void* Y, int64_t ldy,
                          int M, int N, int K, void* workspace, size_t workspace_bytes_, cudaStream_t stream) {
    const qg_status v = check_fp8_args(X, ldx, W, W_scale, Y, ldy, M, N, K);
    if (v != QG_OK || M == 0 || N == 0) return v;
    DeviceInfo* d = device_info();
    if (!d) return QG_ERR_CUDA;
    if (K == 0) return launch_zero_rows(Y, ldy, M, N, stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
    const SchedEntry& se = cached_schedule(QG_KIND_FP8_BLOCK, M, N, K, d->sms);
    const Schedule s = se.s;
    const size_t need = se.ws;
    if (need > 0 && (!workspace || workspace_bytes_ < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return QG_ERR_WORKSPACE;
    Fp8Args a{};
    Fp8Maps maps{};
    const CUtensorMap* tmW = cached_tmap(W, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kMapFp8Weights);
    if (!tmW) return QG_ERR_CUDA;
    maps.m[0] = *tmW;
    a.X = X;
    a.ldx = ldx;
    a.nseg = 1;
    a.seg[0] = Fp8Seg{W, W_scale, Y, ldy, N};
    a.lds = (K + 127) / 128;
    a.M = M;
    a.K = K;
    a.ws = need > 0 ? workspace : nullptr;
    return launch_fp8(a, s, maps, launch_ctl(d), stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

qg_status qgemm_fp8_block_multi(const void* X, int64_t ldx, const qg_fp8_segment* segments, int nseg, int M, int K,
                                void* workspace, size_t workspace_bytes_, cudaStream_t stream) {
    if (nseg < 1 || nseg > QG_MAX_SEGMENTS || !segments) return QG_ERR_INVALID_ARG;
    int64_t rows = 0;   // the segments' tiles, concatenated
    for (int j = 0; j < nseg; ++j) {
        const qg_fp8_segment& g = segments[j];
        if (g.N < 1) return QG_ERR_INVALID_ARG;
        const qg_status v = check_fp8_args(X, ldx, g.W, g.W_scale, g.Y, g.ldy, M, g.N, K);
        if (v != QG_OK) return v;
        rows += (static_cast<int64_t>(g.N) + 127) / 128 * 128;
    }
    if (M == 0) return QG_OK;
    if (rows > INT32_MAX) return QG_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo* d = device_info();
    if (!d) return QG_ERR_CUDA;
    if (K == 0) {
        for (int j = 0; j < nseg; ++j)
            if (launch_zero_rows(segments[j].Y, segments[j].ldy, M, segments[j].N, stream) != cudaSuccess)
                return QG_ERR_CUDA;
        return QG_OK;
    }
    const int N = static_cast<int>(rows);
    const SchedEntry& se = cached_schedule(QG_KIND_FP8_BLOCK, M, N, K, d->sms);
    const Schedule s = se.s;
    const size_t need = se.ws;
    if (need > 0 && (!workspace || workspace_bytes_ < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return QG_ERR_WORKSPACE;
    Fp8Args a{};
    Fp8Maps maps{};
    for (int j = 0; j < nseg; ++j) {
        const qg_fp8_segment& g = segments[j];
        const CUtensorMap* tm = cached_tmap(g.W, static_cast<uint64_t>(K), static_cast<uint64_t>(g.N), kMapFp8Weights);
        if (!tm) return QG_ERR_CUDA;
        maps.m[j] = *tm;   // copied at once: a later lookup may reuse the cache entry
        a.seg[j] = Fp8Seg{g.W, g.W_scale, g.Y, g.ldy, g.N};
    }
    a.X = X;
    a.ldx = ldx;
    a.nseg = nseg;
    a.lds = (K + 127) / 128;
    a.M = M;
    a.K = K;
    a.ws = need > 0 ? workspace : nullptr;
    return launch_fp8(a, s, maps, launch_ctl(d), stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

qg_status qgemm_bf16(const void* X, int64_t ldx, const void* W, void* Y, int64_t ldy, int M, int N, int K,
                     void* workspace, size_t workspace_bytes_, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return QG_OK;
    if (!X || !W || !Y) return QG_ERR_INVALID_ARG;
    if (M > 32 || K % 8 != 0) return QG_ERR_UNSUPPORTED_SHAPE;
    if (ldx < K || ldy < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W) || (ldx % 8) != 0 || (reinterpret_cast<uintptr_t>(Y) & 1u) != 0)
        return QG_ERR_MISALIGNED;
    DeviceInfo* d = device_info();
    if (!d) return QG_ERR_CUDA;
    if (K == 0) return launch_zero_rows(Y, ldy, M, N, stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
    const SchedEntry& se = cached_schedule(QG_KIND_BF16, M, N, K, d->sms);
    const Schedule s = se.s;
    const size_t need = se.ws;
    if (need > 0 && (!workspace || workspace_bytes_ < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return QG_ERR_WORKSPACE;
    const CUtensorMap* tmW = cached_tmap(W, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kMapBf16Weights);
    if (!tmW) return QG_ERR_CUDA;
    CUtensorMap tmX;
    if (!make_tmap(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(ldx) * 2, 64, static_cast<uint32_t>(s.nmma)))
        return QG_ERR_CUDA;
    Bf16Args a;
    a.X = X;
    a.ldx = ldx;
    a.W = W;
    a.Y = Y;
    a.ldy = ldy;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ws = need > 0 ? workspace : nullptr;
    return launch_bf16(a, s, *tmW, tmX, launch_ctl(d), stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

qg_status qg_quantize_act_e4m3(const void* X, int64_t ldx, uint8_t* Xq, int64_t ldxq, float* X_scale, int64_t ldsx,
                               int M, int K, cudaStream_t stream) {
    if (M < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (M == 0 || K == 0) return QG_OK;
    if (!X || !Xq || !X_scale) return QG_ERR_INVALID_ARG;
    if (M > kMaxMW8a8 || K % 16 != 0) return QG_ERR_UNSUPPORTED_SHAPE;
    if (ldx < K || ldxq < K || ldsx < (static_cast<int64_t>(M) + 31) / 32 * 32) return QG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Xq) || !aligned16(X_scale) || ldx % 8 != 0 || ldxq % 16 != 0 || ldsx % 4 != 0)
        return QG_ERR_MISALIGNED;
    if ((K + 127) / 128 * ldsx > (int64_t(1) << 31) / 32) return QG_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo* d = device_info();
    if (!d) return QG_ERR_CUDA;
    return launch_quantize_act(X, ldx, Xq, ldxq, X_scale, ldsx, M, K, launch_ctl(d), stream) == cudaSuccess
               ? QG_OK
               : QG_ERR_CUDA;
}

qg_status qgemm_w8a8_block(const uint8_t* Xq, int64_t ldxq, const float* X_scale, int64_t ldsx, const uint8_t* W,
                           const float* W_scale, void* Y, int64_t ldy, int M, int N, int K, void* workspace,
                           size_t workspace_bytes_, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return QG_OK;
    if (!Xq || !X_scale || !W || !W_scale || !Y) return QG_ERR_INVALID_ARG;
    if (M > kMaxMW8a8 || K % 16 != 0) return QG_ERR_UNSUPPORTED_SHAPE;
    if (ldxq < K || ldy < N || ldsx < (static_cast<int64_t>(M) + 31) / 32 * 32) return QG_ERR_INVALID_ARG;
    if (!aligned16(Xq) || !aligned16(W) || !aligned16(X_scale) || ldxq % 16 != 0 || ldsx % 4 != 0)
        return QG_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(W_scale) & 3u) != 0 || (reinterpret_cast<uintptr_t>(Y) & 1u) != 0)
        return QG_ERR_MISALIGNED;
    // 4 arrival counters per tile, indexed by int
    if ((static_cast<int64_t>(N) + 127) / 128 * ((M + 31) / 32) > (int64_t(1) << 29)) return QG_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo* d = device_info();
    if (!d) return QG_ERR_CUDA;
    if (K == 0) return launch_zero_rows(Y, ldy, M, N, stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
    const SchedEntry& se = cached_schedule(QG_KIND_W8A8, M, N, K, d->sms);
    const Schedule s = se.s;
    const size_t need = se.ws;
    if (need > 0 && (!workspace || workspace_bytes_ < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return QG_ERR_WORKSPACE;
    const CUtensorMap* tmW = cached_tmap(W, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kMapFp8Weights);
    if (!tmW) return QG_ERR_CUDA;
    CUtensorMap tmX;
    if (!make_tmap(&tmX, Xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(ldxq), 128, static_cast<uint32_t>(s.nmma)))
        return QG_ERR_CUDA;
    W8a8Args a{};
    a.Sx = X_scale;
    a.ldsx = ldsx;
    a.S = W_scale;
    a.Y = Y;
    a.ldy = ldy;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ws = need > 0 ? workspace : nullptr;
    // Y by TMA stores where its alignment allows (see W8a8Args); N % 8 == 0
    // too, since the store writes the 16-byte granule that holds column N - 1
    // whole (measured: columns up to the next multiple of 8 were written)
    a.y_tma = aligned16(Y) && ldy % 8 == 0 && N % 8 == 0 &&
              make_tmap(&a.tmY, Y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<uint64_t>(N),
                        static_cast<uint64_t>(M), static_cast<uint64_t>(ldy) * 2, 32, 16, CU_TENSOR_MAP_SWIZZLE_NONE);
    return launch_w8a8(a, s, *tmW, tmX, launch_ctl(d), stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

qg_status qgemm_lut3(const void* X, int64_t ldx, const void* Wq, const void* qmap, const void* scales, void* Y,
                     int64_t ldy, int M, int N, int K, void* workspace, size_t workspace_bytes_,
                     cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return QG_OK;
    if (!X || !Wq || !qmap || !scales || !Y) return QG_ERR_INVALID_ARG;
    if (M > 32 || K % 128 != 0) return QG_ERR_UNSUPPORTED_SHAPE;
    if (ldx < K || ldy < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Wq) || !aligned16(qmap) || (ldx % 8) != 0) return QG_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(scales) & 1u) != 0 || (reinterpret_cast<uintptr_t>(Y) & 1u) != 0)
        return QG_ERR_MISALIGNED;
    DeviceInfo* d = device_info();
    if (!d) return QG_ERR_CUDA;
    if (K == 0) return launch_zero_rows(Y, ldy, M, N, stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
    const SchedEntry& se = cached_schedule(QG_KIND_LUT3, M, N, K, d->sms);
    const Schedule s = se.s;
    const size_t need = se.ws;
    if (need > 0 && (!workspace || workspace_bytes_ < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return QG_ERR_WORKSPACE;
    CUtensorMap tmX;
    if (!make_tmap(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(ldx) * 2, 64, static_cast<uint32_t>(s.nmma)))
        return QG_ERR_CUDA;
    // The scales go through the weight stage when their rows can be copied
    // by a tensor map (16-byte row pitch and base); otherwise the dequant
    // warps load them.
    const CUtensorMap* tmS = nullptr;
    if ((K / 128) % 8 == 0 && aligned16(scales)) {
        tmS = cached_tmap(scales, static_cast<uint64_t>(K / 128), static_cast<uint64_t>(N), kMapLut3Scales);
        if (!tmS) return QG_ERR_CUDA;
    }
    Lut3Args a;
    a.X = X;
    a.ldx = ldx;
    a.Wq = Wq;
    a.qmap = qmap;
    a.scales = scales;
    a.ldsc = K / 128;
    a.Y = Y;
    a.ldy = ldy;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ws = need > 0 ? workspace : nullptr;
    return launch_lut3(a, s, tmX, tmS, launch_ctl(d), stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

size_t qg_lut3_packed_bytes(int N, int K) {
    if (N < 0 || K < 0) return 0;
    return static_cast<size_t>((N + 127) / 128) * static_cast<size_t>((K + 255) / 256) * 16384u;
}

qg_status pack_lut3(const uint8_t* codes, void* packed, int N, int K) {
    if (N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return QG_OK;
    if (!codes || !packed) return QG_ERR_INVALID_ARG;
    const int KT = (K + 255) / 256;
    const size_t bytes = qg_lut3_packed_bytes(N, K);
    uint8_t* out = static_cast<uint8_t*>(packed);
    std::memset(out, 0, bytes);
    for (int n = 0; n < N; ++n) {
        const uint8_t* crow = codes + static_cast<size_t>(n) * K;
        const size_t tile_row = static_cast<size_t>(n / 128) * KT;
        const int r = n % 128;
        for (int k = 0; k < K; k += 8) {
            uint32_t word = 0;
            for (int i = 0; i < 8 && k + i < K; ++i) {
                const uint8_t c = crow[k + i];
                if (c > 7) return QG_ERR_INVALID_ARG;
                word |= static_cast<uint32_t>(c) << (4 * i);
            }
            const int tk = k / 256, q = (k % 256) / 32, w = (k % 32) / 8;
            const size_t off = (tile_row + tk) * 16384 + (static_cast<size_t>(q) * 128 + r) * 16 + w * 4;
            out[off + 0] = static_cast<uint8_t>(word);
            out[off + 1] = static_cast<uint8_t>(word >> 8);
            out[off + 2] = static_cast<uint8_t>(word >> 16);
            out[off + 3] = static_cast<uint8_t>(word >> 24);
        }
    }
    return QG_OK;
}

qg_status unpack_lut3(const void* packed, uint8_t* codes, int N, int K) {
    if (N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return QG_OK;
    if (!codes || !packed) return QG_ERR_INVALID_ARG;
    const int KT = (K + 255) / 256;
    const uint8_t* in = static_cast<const uint8_t*>(packed);
    for (int n = 0; n < N; ++n) {
        const size_t tile_row = static_cast<size_t>(n / 128) * KT;
        const int r = n % 128;
        for (int k = 0; k < K; ++k) {
            const int tk = k / 256, q = (k % 256) / 32, w = (k % 32) / 8, i = k % 8;
            const size_t off = (tile_row + tk) * 16384 + (static_cast<size_t>(q) * 128 + r) * 16 + w * 4 + i / 2;
            codes[static_cast<size_t>(n) * K + k] = static_cast<uint8_t>((in[off] >> (4 * (i % 2))) & 15u);
        }
    }
    return QG_OK;
}

qg_status qg_debug_fp8_split(const void* X, int64_t blocks, void* hi, void* lo, int* exponent,
                             cudaStream_t stream) {
    if (blocks < 0) return QG_ERR_INVALID_ARG;
    if (blocks == 0) return QG_OK;
    if (!X || !hi || !lo || !exponent) return QG_ERR_INVALID_ARG;
    if (blocks > (int64_t(1) << 31) / 32) return QG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(X) || !aligned16(hi) || !aligned16(lo) || (reinterpret_cast<uintptr_t>(exponent) & 3u))
        return QG_ERR_MISALIGNED;
    return launch_split_probe(X, blocks, hi, lo, exponent, stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

qg_status qg_dequant_lut3(const void* Wq, const void* qmap, const void* scales, void* D, int N, int K,
                          cudaStream_t stream) {
    if (N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return QG_OK;
    if (!Wq || !qmap || !scales || !D) return QG_ERR_INVALID_ARG;
    if (K % 128 != 0) return QG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(Wq) || !aligned16(qmap) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
        (reinterpret_cast<uintptr_t>(D) & 1u))
        return QG_ERR_MISALIGNED;
    return launch_dequant_lut3(Wq, qmap, scales, D, N, K, stream) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

qg_status qg_debug_schedule(int kind, int M, int N, int K, int* ctas, int64_t* ranges, int* info, int capacity,
                            cudaStream_t stream) {
    if (max_m(kind) == 0) return QG_ERR_INVALID_ARG;
    if (M < 1 || M > max_m(kind) || N < 1 || K < 1 || !ctas) return QG_ERR_INVALID_ARG;
    if (K % k_multiple(kind) != 0) return QG_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo* d = device_info();
    if (!d) return QG_ERR_CUDA;
    const Schedule s = cached_schedule(kind, M, N, K, d->sms).s;
    *ctas = s.G;
    if (!ranges || !info) return QG_OK;   // a query of the CTA count only
    if (capacity < s.G) return QG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ranges) & 7u) || (reinterpret_cast<uintptr_t>(info) & 3u)) return QG_ERR_MISALIGNED;
    schedule_probe_kernel<<<s.G, 32, 0, stream>>>(s.U, s.G, s.KU, reinterpret_cast<long long*>(ranges), info);
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

qg_status qg_dispatch_set(int kind, int M, int N, int K, int ctas) {
    if (max_m(kind) == 0) return QG_ERR_INVALID_ARG;
    if (M < 1 || M > max_m(kind) || N < 1 || K < 1 || ctas < 0) return QG_ERR_INVALID_ARG;
    DeviceInfo* d = device_info();
    if (!d) return QG_ERR_CUDA;
    if (ctas > d->sms) return QG_ERR_INVALID_ARG;
    {
        std::lock_guard<std::mutex> lk(g_table_mu);
        int at = -1;
        for (int i = 0; i < g_table_n; ++i) {
            const TableEntry& e = g_table[i];
            if (e.kind == kind && e.M == M && e.N == N && e.K == K) at = i;
        }
        if (ctas == 0) {
            if (at >= 0) g_table[at] = g_table[--g_table_n];
        } else if (at >= 0) {
            g_table[at].ctas = ctas;
        } else {
            if (g_table_n == static_cast<int>(sizeof(g_table) / sizeof(g_table[0]))) return QG_ERR_INVALID_ARG;
            g_table[g_table_n++] = TableEntry{kind, M, N, K, ctas};
        }
    }
    g_table_gen.fetch_add(1, std::memory_order_acq_rel);
    return QG_OK;
}

int qg_dispatch_get(int kind, int M, int N, int K) {
    if (M < 1 || M > max_m(kind) || N < 1 || K < 1) return 0;
    DeviceInfo* d = device_info();
    if (!d) return 0;
    return cached_schedule(kind, M, N, K, d->sms).s.G;
}

int qg_dispatch_rule(int kind, int M, int N, int K, int sms) {
    if (max_m(kind) == 0 || M < 1 || M > max_m(kind) || N < 1 || K < 1 || sms < 1) return 0;
    return schedule_for(kind, M, N, K, sms, 0).G;
}

void qg_dispatch_clear(void) {
    {
        std::lock_guard<std::mutex> lk(g_table_mu);
        g_table_n = 0;
    }
    g_table_gen.fetch_add(1, std::memory_order_acq_rel);
}

qg_status qg_last_device_status(cudaStream_t stream) {
    DeviceInfo* d = device_info();
    if (!d) return QG_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return QG_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, d->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return QG_ERR_CUDA;
    if (word != 0 && cudaMemset(d->status, 0, sizeof(word)) != cudaSuccess) return QG_ERR_CUDA;
    if (word & kDevTimeout) {
        // a call that timed out may have been a no-alloc call: its arrival
        // counters in the library's own scratch array are left set
        if (noalloc_clear_counters(stream) != cudaSuccess) return QG_ERR_CUDA;
        return QG_ERR_TIMEOUT;
    }
    return word ? QG_ERR_CUDA : QG_OK;
}

void qg_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns < 1000 ? 1000 : ns); }

void qg_set_fault_injection(int unit) { g_fault_unit.store(unit < 0 ? -1 : unit); }

void qg_set_weight_prefetch_overlap(int enable) { g_overlap.store(enable ? 1 : 0); }

const char* qg_status_string(qg_status s) {
    switch (s) {
        case QG_OK: return "ok";
        case QG_ERR_INVALID_ARG: return "invalid argument";
        case QG_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case QG_ERR_MISALIGNED: return "misaligned pointer or stride";
        case QG_ERR_CUDA: return "CUDA error";
        case QG_ERR_TIMEOUT: return "in-kernel wait timed out";
        case QG_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

const char* qg_version(void) { return "0.2.0"; }

}  // extern "C"
