// W8A16 FP8 block-scaled decode GEMM for sm_103a.
//
//   Y[m, n] = bf16( sum_kb  s[n/128, kb] * ( sum_{k in kb} x[m,k] * e4m3(W[n,k]) ) )
//
// The two-level fold ("atlas" m16_tc module page, section NUMERICS): each
// 128-wide K block is reduced on the tensor core into its own FP32
// accumulator, then multiplied by that block's FP32 scale once and added to an
// FP32 outer accumulator held in registers.
//
// Swap-AB: a 128-row slice of W is the MMA's M side (rows of TMEM), the M <= 32
// activation rows are the MMA's narrow N side (16 or 32), so no row of the
// tensor-core tile is padding except the N-side columns beyond M.
//
// One persistent CTA per SM (448 threads, 14 warps):
//   warp 0      TMA producer: 128x128 E4M3 weight tile (evict-first L2 hint)
//               and the 128-wide X slice (two 64-element boxes, 128-byte
//               swizzle) per work unit, into an 8-stage shared-memory ring.
//   warp 1      MMA issuer: 8 x tcgen05.mma kind::f16 (M=128, N=16|32, K=16)
//               per unit, A from TMEM, B (X) from shared memory, D in TMEM.
//   warps 2-5   fold / epilogue: tcgen05.ld of the block sum, outer += s*inner,
//               BF16 store or split-K partial + last-arriver reduction.
//   warps 6-13  dequant: shared -> registers -> E4M3 to BF16 (exact) ->
//               tcgen05.st into a 4-deep A ring in TMEM.
// Work units (tile of 128 rows, 128-wide K block) are split evenly over the
// CTAs in tile-major order (stream-K); a tile shared by several CTAs is
// summed, in ascending K order of its pieces, by whichever CTA finishes its
// piece last (an atomic arrival counter; nobody spins on another CTA).
#include <cuda_bf16.h>

#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr int kThreads = 448;
constexpr int kWarpMma = 1;
constexpr int kWarpDeq0 = 6;
constexpr int kStages = 8;
constexpr int kNA = 4;          // A buffers in TMEM, 64 columns each
constexpr int kND = 4;          // D buffers in TMEM, 32 columns each
constexpr int kTmemCols = 512;
constexpr int kDCol0 = kNA * 64;
constexpr int kWBytes = 128 * 128;

template <int NMMA>
struct Layout {
    static constexpr int kXBox = NMMA * 128;            // one 64-element X box, bytes
    static constexpr int kStageBytes = kWBytes + 2 * kXBox;
    static constexpr int kBarOff = kStages * kStageBytes;
    static constexpr int kNumBars = 2 * kStages + 2 * kNA + 2 * kND;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 64 + 1024;  // + alignment slack
};

struct Fp8Params {
    const float* S;
    int64_t lds;
    __nv_bfloat16* Y;
    int64_t ldy;
    int M, N, K;
    int KB;               // units (128-wide K blocks) per tile
    long long U;          // total units
    int G;                // CTAs
    uint32_t* cnt;        // per (tile, quadrant) arrival counters
    float* part;          // [G][2][NMMA][128] partial outer sums
    uint64_t timeout_ns;
    int fault_unit;
    uint32_t* status;
};

// CTA that owns unit x when U units are split evenly over G CTAs.
__device__ __forceinline__ int unit_owner(long long x, long long U, int G) {
    return static_cast<int>(((x + 1) * G - 1) / U);
}

__device__ __forceinline__ long long unit_begin(int c, long long U, int G) {
    return static_cast<long long>(c) * U / G;
}

// Warp-uniform bounded wait: every lane polls, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& c) {
    const bool ok = wait_bounded(bar, parity, c);
    return __all_sync(0xffffffffu, ok);
}

// Wait used only while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if (globaltimer() - t0 > timeout_ns) return;
    }
}

template <int NMMA>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_block_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                          const Fp8Params p) {
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
            mbar_init(empty(s), 8 + 1);   // 8 dequant warps + the MMA commit (X slice)
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
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmX);
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int issued = 0;
            for (int i = 0; i < nunits; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !wait_bounded(empty(s), ((i / kStages) - 1) & 1, wc)) break;
                if (cta == 0 && i == p.fault_unit) continue;   // failure-path test hook
                const long long u = u0 + i;
                const int tile = static_cast<int>(u / p.KB);
                const int kb = static_cast<int>(u % p.KB);
                const uint32_t st = base + s * L::kStageBytes;
                mbar_arrive_expect_tx(full(s), L::kStageBytes);
                tma_load_2d(st, &tmW, full(s), kb * 128, tile * 128, pol_w);
                tma_load_2d(st + kWBytes, &tmX, full(s), kb * 128, 0, pol_x);
                tma_load_2d(st + kWBytes + L::kXBox, &tmX, full(s), kb * 128 + 64, 0, pol_x);
                issued = i + 1;
            }
            // Every copy this thread started must land before the CTA can exit.
            for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i) {
                if (cta == 0 && i == p.fault_unit) continue;
                drain_wait(full(i % kStages), (i / kStages) & 1, p.timeout_ns);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(NMMA, true);
            int issued = 0;
            for (int i = 0; i < nunits; ++i) {
                const int s = i % kStages;
                const int a = i % kNA;
                const int d = i % kND;
                if (!wait_bounded(full(s), (i / kStages) & 1, wc)) break;
                if (!wait_bounded(afull(a), (i / kNA) & 1, wc)) break;
                if (i >= kND && !wait_bounded(dempty(d), ((i / kND) - 1) & 1, wc)) break;
                tc_fence_after();
                const uint32_t xs = base + s * L::kStageBytes + kWBytes;
                const uint32_t dt = tmem + kDCol0 + d * 32;
                const uint32_t at = tmem + a * 64;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t xa = xs + (j >> 2) * L::kXBox + (j & 3) * 32;
                    mma_ts_f16(dt, at + j * 8, smem_desc_sw128(xa), idesc, j > 0 ? 1u : 0u);
                }
                tc_commit(empty(s));
                tc_commit(aempty(a));
                tc_commit(dfull(d));
                issued = i + 1;
            }
            if (issued > 0) drain_wait(dfull((issued - 1) % kND), ((issued - 1) / kND) & 1, p.timeout_ns);
        }
    } else if (warp < kWarpDeq0) {
        // ------------------------------------------------------------ fold / epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const int first_tile = static_cast<int>(u0 / p.KB);
        float outer[NMMA];
#pragma unroll
        for (int m = 0; m < NMMA; ++m) outer[m] = 0.0f;
        for (int i = 0; i < nunits; ++i) {
            const long long u = u0 + i;
            const int tile = static_cast<int>(u / p.KB);
            const int kb = static_cast<int>(u % p.KB);
            const int d = i % kND;
            const float sc = __ldg(p.S + static_cast<int64_t>(tile) * p.lds + kb);
            if (!warp_wait(dfull(d), (i / kND) & 1, wc)) break;
            tc_fence_after();
            uint32_t v0[16], v1[16];
            tmem_ld_x16(tl + kDCol0 + d * 32, v0);
            if constexpr (NMMA == 32) tmem_ld_x16(tl + kDCol0 + d * 32 + 16, v1);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty(d));
#pragma unroll
            for (int m = 0; m < 16; ++m) outer[m] = __fadd_rn(outer[m], __fmul_rn(__uint_as_float(v0[m]), sc));
            if constexpr (NMMA == 32) {
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    outer[16 + m] = __fadd_rn(outer[16 + m], __fmul_rn(__uint_as_float(v1[m]), sc));
            }

            if (kb != p.KB - 1 && u != u1 - 1) continue;
            // ---- end of this CTA's piece of `tile`
            const int n = tile * 128 + row;
            const bool whole = (kb == p.KB - 1) && (u - kb >= u0);
            if (whole) {
                if (n < p.N) {
#pragma unroll
                    for (int m = 0; m < NMMA; ++m)
                        if (m < p.M) p.Y[static_cast<int64_t>(m) * p.ldy + n] = __float2bfloat16_rn(outer[m]);
                }
            } else {
                const int which = (tile == first_tile) ? 0 : 1;
                float* mine = p.part + (static_cast<size_t>(cta) * 2 + which) * NMMA * 128;
#pragma unroll
                for (int m = 0; m < NMMA; ++m)
                    if (m < p.M) __stcg(mine + m * 128 + row, outer[m]);
                __threadfence();
                __syncwarp();
                uint32_t prev = 0;
                if (lane == 0) prev = atomicAdd(p.cnt + tile * 4 + q, 1u);
                prev = __shfl_sync(0xffffffffu, prev, 0);
                const long long t0 = static_cast<long long>(tile) * p.KB;
                const int cf = unit_owner(t0, p.U, p.G);
                const int cl = unit_owner(t0 + p.KB - 1, p.U, p.G);
                if (static_cast<int>(prev) == cl - cf) {
                    // last piece to arrive: sum all pieces in ascending K order
                    __threadfence();
#pragma unroll
                    for (int m = 0; m < NMMA; ++m) {
                        if (m >= p.M) break;
                        float acc = 0.0f;
                        for (int c2 = cf; c2 <= cl; ++c2) {
                            const int w2 = (tile == static_cast<int>(unit_begin(c2, p.U, p.G) / p.KB)) ? 0 : 1;
                            float* slot = p.part + ((static_cast<size_t>(c2) * 2 + w2) * NMMA + m) * 128 + row;
                            const float part = (c2 == cta) ? outer[m] : __ldcg(slot);
                            __stcg(slot, 0.0f);   // every call leaves the workspace zero-filled
                            acc = __fadd_rn(acc, part);
                        }
                        if (n < p.N) p.Y[static_cast<int64_t>(m) * p.ldy + n] = __float2bfloat16_rn(acc);
                    }
                    if (lane == 0) p.cnt[tile * 4 + q] = 0u;   // leave the workspace clean
                }
            }
#pragma unroll
            for (int m = 0; m < NMMA; ++m) outer[m] = 0.0f;
        }
    } else {
        // ------------------------------------------------------------ dequant
        const int q = warp & 3;
        const int h = (warp - kWarpDeq0) >> 2;     // which 64-wide half of the K block
        const int row = q * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 32;
        for (int i = 0; i < nunits; ++i) {
            const int s = i % kStages;
            const int a = i % kNA;
            if (!warp_wait(full(s), (i / kStages) & 1, wc)) break;
            const uint8_t* wrow = gbase + s * L::kStageBytes + row * 128;
            uint4 c[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                c[j] = *reinterpret_cast<const uint4*>(wrow + (((4 * h + j) ^ (row & 7)) << 4));
            uint32_t o[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                e4m3x4_to_bf16(c[j].x, o[8 * j + 0], o[8 * j + 1]);
                e4m3x4_to_bf16(c[j].y, o[8 * j + 2], o[8 * j + 3]);
                e4m3x4_to_bf16(c[j].z, o[8 * j + 4], o[8 * j + 5]);
                e4m3x4_to_bf16(c[j].w, o[8 * j + 6], o[8 * j + 7]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
            if (i >= kNA && !warp_wait(aempty(a), ((i / kNA) - 1) & 1, wc)) break;
            __syncwarp();
            tc_fence_after();
            tmem_st_x32(tl + a * 64, o);
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
cudaError_t launch_t(const Fp8Args& a, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                     const LaunchCtl& c, cudaStream_t st) {
    using L = Layout<NMMA>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(fp8_block_gemm_kernel<NMMA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    Fp8Params p;
    p.S = a.S;
    p.lds = a.lds;
    p.Y = static_cast<__nv_bfloat16*>(a.Y);
    p.ldy = a.ldy;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.KB = s.KU;
    p.U = s.U;
    p.G = s.G;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    const size_t cnt_bytes = (static_cast<size_t>(s.T) * 4 * sizeof(uint32_t) + 255) & ~static_cast<size_t>(255);
    p.cnt = reinterpret_cast<uint32_t*>(ws);
    p.part = ws ? reinterpret_cast<float*>(ws + cnt_bytes) : nullptr;
    p.timeout_ns = c.timeout_ns;
    p.fault_unit = c.fault_unit;
    p.status = c.status;
    fp8_block_gemm_kernel<NMMA><<<s.G, kThreads, L::kSmemBytes, st>>>(tmW, tmX, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8(const Fp8Args& a, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                       const LaunchCtl& c, cudaStream_t st) {
    if (s.nmma == 16) return launch_t<16>(a, s, tmW, tmX, c, st);
    return launch_t<32>(a, s, tmW, tmX, c, st);
}

}  // namespace qg
