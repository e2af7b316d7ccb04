// W3A16 learned-LUT decode GEMM for sm_103a (FLUTE "optimized_w3" page,
// sections Core contributions and Results, re-designed for tcgen05).
//
//   d[n, k] = fp16_rne(qmap[code[n, k]] * scale[n, k/128])
//   Y[m, n] = fp16( sum_k x[m, k] * d[n, k] )          (FP32 accumulation)
//
// Weights arrive pre-packed (pack_lut3): one 16 KB contiguous block per
// (128-row tile, 256-wide K step), one code per nibble, 16-byte chunks ordered
// so that the 32 lanes owning 32 consecutive rows read 512 contiguous bytes.
// The dequantiser keeps, per (row, 128-wide group), the scaled 8-entry table as
// two FP16 byte planes in registers and looks codes up with byte permutes
// whose selector is the code word itself (8 values = 1 shift + 8 permutes; no
// shared-memory table).  The scale is applied once per table entry, which
// gives the same FP16 values as scaling every weight.
//
// CTA roles as in the FP8 kernel (448 threads): warp 0 bulk-copies the packed
// block (evict-first) and TMA-loads four 64-wide FP16 X boxes per unit; warp 1
// issues 16 tcgen05.mma kind::f16 per unit into one TMEM accumulator per tile
// piece (no per-block fold: the scale is already inside d); warps 2-5 read the
// accumulator at the end of each piece and store FP16 or a split-K partial;
// warps 6-13 dequantise into a 3-deep A ring in TMEM.
#include <cuda_fp16.h>

#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr int kThreads = 448;
constexpr int kWarpMma = 1;
constexpr int kWarpDeq0 = 6;
constexpr int kStages = 6;
constexpr int kNA = 3;          // A buffers in TMEM, 128 columns each
constexpr int kND = 2;          // D buffers in TMEM, 32 columns each
constexpr int kTmemCols = 512;
constexpr int kDCol0 = kNA * 128;
constexpr int kWBytes = 16384;  // one packed (128 x 256) block

template <int NMMA>
struct Layout {
    static constexpr int kXBox = NMMA * 128;
    static constexpr int kStageBytes = kWBytes + 4 * kXBox;
    static constexpr int kBarOff = kStages * kStageBytes;
    static constexpr int kNumBars = 2 * kStages + 2 * kNA + 2 * kND;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 64 + 1024;
};

struct Lut3Params {
    const uint8_t* Wq;
    const uint4* qmap;
    const uint16_t* scales;
    int64_t ldsc;
    __half* Y;
    int64_t ldy;
    int M, N, K;
    int G128;             // K / 128 scale groups per row
    int KU;               // units (256-wide K steps) per tile
    long long U;
    int G;                // CTAs
    uint32_t* cnt;
    float* part;
    uint64_t timeout_ns;
    int fault_unit;
    uint32_t* status;
};

__device__ __forceinline__ int unit_owner(long long x, long long U, int G) {
    return static_cast<int>(((x + 1) * G - 1) / U);
}
__device__ __forceinline__ long long unit_begin(int c, long long U, int G) {
    return static_cast<long long>(c) * U / G;
}
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& c) {
    const bool ok = wait_bounded(bar, parity, c);
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if (globaltimer() - t0 > timeout_ns) return;
    }
}

template <int NMMA>
__global__ void __launch_bounds__(kThreads, 1)
    lut3_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const Lut3Params p) {
    using L = Layout<NMMA>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + L::kBarOff;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto afull = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto aempty = [&](int a) { return bar0 + 8u * (2 * kStages + kNA + a); };
    auto dfull = [&](int d) { return bar0 + 8u * (2 * kStages + 2 * kNA + d); };
    auto dempty = [&](int d) { return bar0 + 8u * (2 * kStages + 2 * kNA + kND + d); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = unit_begin(cta, p.U, p.G);
    const long long u1 = unit_begin(cta + 1, p.U, p.G);
    const int nunits = static_cast<int>(u1 - u0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 8 + 1);
        }
        for (int a = 0; a < kNA; ++a) {
            mbar_init(afull(a), 8);
            mbar_init(aempty(a), 1);
        }
        for (int d = 0; d < kND; ++d) {
            mbar_init(dfull(d), 1);
            mbar_init(dempty(d), 4);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncwarp();
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{p.timeout_ns, p.status, abort_flag};

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tmX);
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int issued = 0;
            for (int i = 0; i < nunits; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !wait_bounded(empty(s), ((i / kStages) - 1) & 1, wc)) break;
                if (cta == 0 && i == p.fault_unit) continue;   // failure-path test hook
                const long long u = u0 + i;
                const int ku = static_cast<int>(u % p.KU);
                const uint32_t st = base + s * L::kStageBytes;
                mbar_arrive_expect_tx(full(s), L::kStageBytes);
                bulk_load(st, p.Wq + static_cast<size_t>(u) * kWBytes, kWBytes, full(s), pol_w);
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    tma_load_2d(st + kWBytes + b * L::kXBox, &tmX, full(s), ku * 256 + b * 64, 0, pol_x);
                issued = i + 1;
            }
            for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i) {
                if (cta == 0 && i == p.fault_unit) continue;
                drain_wait(full(i % kStages), (i / kStages) & 1, p.timeout_ns);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(NMMA, false);
            int seg = -1;
            int last_i = -1;
            for (int i = 0; i < nunits; ++i) {
                const long long u = u0 + i;
                const int ku = static_cast<int>(u % p.KU);
                const bool seg_start = (i == 0) || (ku == 0);
                const bool seg_end = (ku == p.KU - 1) || (i == nunits - 1);
                if (seg_start) ++seg;
                const int s = i % kStages;
                const int a = i % kNA;
                const int d = seg % kND;
                if (!wait_bounded(full(s), (i / kStages) & 1, wc)) break;
                if (!wait_bounded(afull(a), (i / kNA) & 1, wc)) break;
                if (seg_start && seg >= kND && !wait_bounded(dempty(d), ((seg / kND) - 1) & 1, wc)) break;
                tc_fence_after();
                const uint32_t xs = base + s * L::kStageBytes + kWBytes;
                const uint32_t dt = tmem + kDCol0 + d * 32;
                const uint32_t at = tmem + a * 128;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t xa = xs + (j >> 2) * L::kXBox + (j & 3) * 32;
                    mma_ts_f16(dt, at + j * 8, smem_desc_sw128(xa), idesc, (seg_start && j == 0) ? 0u : 1u);
                }
                tc_commit(empty(s));
                tc_commit(aempty(a));
                if (seg_end) tc_commit(dfull(d));
                last_i = i;
            }
            // the A-buffer release of the last unit follows every MMA issued
            if (last_i >= 0) drain_wait(aempty(last_i % kNA), (last_i / kNA) & 1, p.timeout_ns);
        }
    } else if (warp < kWarpDeq0) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const int first_tile = static_cast<int>(u0 / p.KU);
        int seg = -1;
        for (int i = 0; i < nunits; ++i) {
            const long long u = u0 + i;
            const int ku = static_cast<int>(u % p.KU);
            if (i == 0 || ku == 0) ++seg;
            if (ku != p.KU - 1 && i != nunits - 1) continue;
            const int tile = static_cast<int>(u / p.KU);
            const int d = seg % kND;
            if (!warp_wait(dfull(d), (seg / kND) & 1, wc)) break;
            tc_fence_after();
            float v[NMMA];
            {
                uint32_t v0[16], v1[16];
                tmem_ld_x16(tl + kDCol0 + d * 32, v0);
                if constexpr (NMMA == 32) tmem_ld_x16(tl + kDCol0 + d * 32 + 16, v1);
                tmem_wait_ld();
#pragma unroll
                for (int m = 0; m < 16; ++m) v[m] = __uint_as_float(v0[m]);
                if constexpr (NMMA == 32) {
#pragma unroll
                    for (int m = 0; m < 16; ++m) v[16 + m] = __uint_as_float(v1[m]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty(d));
            const int n = tile * 128 + row;
            const bool whole = (ku == p.KU - 1) && (u - ku >= u0);
            if (whole) {
                if (n < p.N) {
#pragma unroll
                    for (int m = 0; m < NMMA; ++m)
                        if (m < p.M)
                            p.Y[static_cast<int64_t>(m) * p.ldy + n] = __float2half_rn(v[m]);
                }
                continue;
            }
            const int which = (tile == first_tile) ? 0 : 1;
            float* mine = p.part + (static_cast<size_t>(cta) * 2 + which) * NMMA * 128;
#pragma unroll
            for (int m = 0; m < NMMA; ++m)
                if (m < p.M) __stcg(mine + m * 128 + row, v[m]);
            __threadfence();
            __syncwarp();
            uint32_t prev = 0;
            if (lane == 0) prev = atomicAdd(p.cnt + tile * 4 + q, 1u);
            prev = __shfl_sync(0xffffffffu, prev, 0);
            const long long t0 = static_cast<long long>(tile) * p.KU;
            const int cf = unit_owner(t0, p.U, p.G);
            const int cl = unit_owner(t0 + p.KU - 1, p.U, p.G);
            if (static_cast<int>(prev) != cl - cf) continue;
            __threadfence();
#pragma unroll
            for (int m = 0; m < NMMA; ++m) {
                if (m >= p.M) break;
                float acc = 0.0f;
                for (int c2 = cf; c2 <= cl; ++c2) {
                    const int w2 = (tile == static_cast<int>(unit_begin(c2, p.U, p.G) / p.KU)) ? 0 : 1;
                    float* slot = p.part + ((static_cast<size_t>(c2) * 2 + w2) * NMMA + m) * 128 + row;
                    const float part = (c2 == cta) ? v[m] : __ldcg(slot);
                    __stcg(slot, 0.0f);   // every call leaves the workspace zero-filled
                    acc = __fadd_rn(acc, part);
                }
                if (n < p.N) p.Y[static_cast<int64_t>(m) * p.ldy + n] = __float2half_rn(acc);
            }
            if (lane == 0) p.cnt[tile * 4 + q] = 0u;
        }
    } else {
        // ------------------------------------------------------------ dequant
        const int q = warp & 3;
        const int h = (warp - kWarpDeq0) >> 2;     // which 128-wide group of the unit
        const int row = q * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 64;
        const uint4 qm = __ldg(p.qmap);
        for (int i = 0; i < nunits; ++i) {
            const long long u = u0 + i;
            const int tile = static_cast<int>(u / p.KU);
            const int g = static_cast<int>(u % p.KU) * 2 + h;
            const int n = tile * 128 + row;
            const uint32_t sc = (n < p.N && g < p.G128)
                                    ? static_cast<uint32_t>(__ldg(p.scales + static_cast<int64_t>(n) * p.ldsc + g))
                                    : 0u;
            const int s = i % kStages;
            const int a = i % kNA;
            if (!warp_wait(full(s), (i / kStages) & 1, wc)) break;
            const uint8_t* blk = gbase + s * L::kStageBytes;
            uint4 c[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                c[j] = *reinterpret_cast<const uint4*>(blk + (((4 * h + j) * 128 + row) << 4));
            const uint32_t sc2 = sc | (sc << 16);
            const LutPlanes t = lut_planes(f16x2_mul(qm.x, sc2), f16x2_mul(qm.y, sc2), f16x2_mul(qm.z, sc2),
                                           f16x2_mul(qm.w, sc2));
            uint32_t o0[32], o1[32];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t w4[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t r4[4];
                    lut3x8_to_f16(w4[w], t, r4);
#pragma unroll
                    for (int e = 0; e < 4; ++e) o0[16 * j + 4 * w + e] = r4[e];
                }
            }
#pragma unroll
            for (int j = 2; j < 4; ++j) {
                const uint32_t w4[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t r4[4];
                    lut3x8_to_f16(w4[w], t, r4);
#pragma unroll
                    for (int e = 0; e < 4; ++e) o1[16 * (j - 2) + 4 * w + e] = r4[e];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
            if (i >= kNA && !warp_wait(aempty(a), ((i / kNA) - 1) & 1, wc)) break;
            __syncwarp();
            tc_fence_after();
            tmem_st_x32(tl + a * 128, o0);
            tmem_st_x32(tl + a * 128 + 32, o1);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(a));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int NMMA>
cudaError_t launch_t(const Lut3Args& a, const Schedule& s, const CUtensorMap& tmX, const LaunchCtl& c,
                     cudaStream_t st) {
    using L = Layout<NMMA>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(lut3_gemm_kernel<NMMA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    Lut3Params p;
    p.Wq = static_cast<const uint8_t*>(a.Wq);
    p.qmap = static_cast<const uint4*>(a.qmap);
    p.scales = static_cast<const uint16_t*>(a.scales);
    p.ldsc = a.ldsc;
    p.Y = static_cast<__half*>(a.Y);
    p.ldy = a.ldy;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.G128 = a.K / 128;
    p.KU = s.KU;
    p.U = s.U;
    p.G = s.G;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    const size_t cnt_bytes = (static_cast<size_t>(s.T) * 4 * sizeof(uint32_t) + 255) & ~static_cast<size_t>(255);
    p.cnt = reinterpret_cast<uint32_t*>(ws);
    p.part = ws ? reinterpret_cast<float*>(ws + cnt_bytes) : nullptr;
    p.timeout_ns = c.timeout_ns;
    p.fault_unit = c.fault_unit;
    p.status = c.status;
    lut3_gemm_kernel<NMMA><<<s.G, kThreads, L::kSmemBytes, st>>>(tmX, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lut3(const Lut3Args& a, const Schedule& s, const CUtensorMap& tmX, const LaunchCtl& c,
                        cudaStream_t st) {
    if (s.nmma == 16) return launch_t<16>(a, s, tmX, c, st);
    return launch_t<32>(a, s, tmX, c, st);
}

}  // namespace qg
