// W8A8 block-scaled GEMM for sm_103a: FP8 activations as well as FP8
// weights, for batches beyond the decode tier ("arc" PR page, the cuBLASLt
// block-scale section: block-scaled FP8 needs FP8 activations, hence an
// activation quantiser).
//
//   Xq, sx = quantise(X):  per (row m, 128-wide K block kb)
//            sx[kb, m] = amax / 448,  xq = e4m3_rne_satfinite(x / sx)
//   Y[m, n] = bf16( sum_kb (sx[kb, m] * s[n/128, kb]) * (sum_{k in kb} xq[m,k] * w[n,k]) )
//
// The GEMM tiles the output in 128 weight rows x 32 activation rows; a unit
// is one such tile x one 128-wide K block.  Both operands go to
// tcgen05.mma kind::f8f6f4 as stored (TMA, 128-byte swizzle); each unit's
// block sum lands in its own TMEM accumulator and the fold multiplies it by
// the unit's 32 block factors (activation scale x weight scale) once and adds
// it to an FP32 outer accumulator in registers: the same two-level fold as
// the W8A16 path.  Tiles are numbered weight-tile-major (the row blocks of a
// weight tile are neighbours, so its weights are read from HBM once and from
// L2 after); the stream-K split and the split-K partial sums are the shared
// ones of qg_gemm.cuh.
//
// One persistent CTA per SM, 256 threads:
//   warp 0      weight producer: one 16 KB TMA tile per unit (evict-first).
//   warp 1      activation producer, after the grid dependency wait: the
//               unit's 32 x 128 E4M3 slice (TMA) and its 32 activation scales
//               (one 128-byte bulk copy) into a ring.
//   warp 2      MMA issuer: 4 tcgen05.mma (M = 128, N = 32, K = 32) per unit.
//   warps 4-7   fold / epilogue, one per TMEM lane quadrant.
#include "qg_gemm.cuh"
#include "qg_w8a8.h"

namespace qg {
namespace {

using gemm::Cursor;
using gemm::Params;

constexpr int kNA = 32;          // activation rows per output tile (MMA N)
constexpr int kThreads = 256;
constexpr int kWarpWProd = 0, kWarpXProd = 1, kWarpMma = 2, kWarpFold0 = 4;

struct W8a8Layout {
    static constexpr int kWBytes = 128 * 128;      // one E4M3 weight unit
    static constexpr int kXBytes = kNA * 128;      // one E4M3 activation slice
    static constexpr int kXSlot = kXBytes + 1024;  // + 32 scales (128 B), padded to keep 1024-B alignment
    static constexpr int kXStages = 12;
    static constexpr int kAcc = 8;                 // TMEM accumulators of kNA columns
    static constexpr int kTmemCols = kAcc * kNA;   // 256
    static constexpr int kFixed = kXStages * kXSlot + 8 * (2 * 16 + 2 * kXStages + 2 * kAcc) + 64 + 1024;
    static constexpr int kWFit = (232448 - kFixed) / kWBytes;
    static constexpr int kWStages = kWFit < 12 ? kWFit : 12;
    static constexpr int kXOff = kWStages * kWBytes;
    static constexpr int kBarOff = kXOff + kXStages * kXSlot;
    static constexpr int kNumBars = 2 * kWStages + 2 * kXStages + 2 * kAcc;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 64 + 1024;
    static_assert(kWStages >= 8, "weight ring");
    static_assert(kXOff % 1024 == 0 && kXSlot % 1024 == 0, "keep the 1024-byte swizzle alignment");
    static_assert(kWStages * kWBytes >= 4 * gemm::scratch_quadrant<kNA>(), "reduction scratch in the weight ring");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// Output rows of tile t = (weight tile tn, activation row block tm), t = tn *
// tm_count + tm: weight row n = tn * 128 + row, activation rows tm * 32 ...
__device__ __forceinline__ void store_tile_rows(const Params& p, int tm_count, int tile, int row,
                                                const float (&v)[kNA]) {
    const int tn = tile / tm_count;
    const int m0 = (tile - tn * tm_count) * kNA;
    const int n = tn * 128 + row;
    if (n >= p.N) return;
    const gemm::Seg sg = p.seg[0];
#pragma unroll
    for (int m = 0; m < kNA; ++m)
        if (m0 + m < p.M)
            static_cast<__nv_bfloat16*>(sg.Y)[static_cast<int64_t>(m0 + m) * sg.ldy + n] = __float2bfloat16_rn(v[m]);
}

// Sum of a split tile's pieces (staged through idle shared memory) and its
// store; resets the tile's arrival counter.
__device__ __forceinline__ void finish_tile(const Params& p, int tm_count, int tile, int which, int split_info,
                                            int q, int lane, uint8_t* scratch) {
    const int row = q * 32 + lane;
    const int cf = __shfl_sync(0xffffffffu, split_info, 3 * which);
    const int cl = __shfl_sync(0xffffffffu, split_info, 3 * which + 1);
    const int w_first = __shfl_sync(0xffffffffu, split_info, 3 * which + 2);
    float acc[kNA];
    gemm::sum_pieces_staged<kNA>(p, row, lane, q, cf, cl, w_first, scratch, acc);
    store_tile_rows(p, tm_count, tile, row, acc);
    __syncwarp();
    if (lane == 0) p.cnt[tile * 4 + q] = 0u;
}

// End of a CTA's piece of `tile`, as gemm::end_piece with this kernel's
// tile-to-output mapping: a whole tile is stored; a split piece is stored to
// the workspace and counted; the last to arrive finishes the tile now when
// `scratch` is given, else returns true (finished at the end of the range).
__device__ __forceinline__ bool end_piece(const Params& p, int tm_count, const float (&outer)[kNA], int tile, int kb,
                                          long long u, long long u0, int first_tile, int split_info, int q, int lane,
                                          uint8_t* scratch) {
    const int row = q * 32 + lane;
    const bool whole = (kb == p.KB - 1) && (u - kb >= u0);
    if (whole) {
        store_tile_rows(p, tm_count, tile, row, outer);
        return false;
    }
    const int which = (tile == first_tile) ? 0 : 1;
    float4* mine = gemm::slot_base<kNA>(p, blockIdx.x, which) + row;
#pragma unroll
    for (int g = 0; g < kNA / 4; ++g)
        __stcg(mine + g * 128, make_float4(outer[4 * g], outer[4 * g + 1], outer[4 * g + 2], outer[4 * g + 3]));
    // every lane's partial visible GPU-wide before lane 0's arrival
    __threadfence();
    __syncwarp();
    uint32_t prev = 0;
    if (lane == 0) prev = atomicAdd(p.cnt + tile * 4 + q, 1u);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    const int cf = __shfl_sync(0xffffffffu, split_info, 3 * which);
    const int cl = __shfl_sync(0xffffffffu, split_info, 3 * which + 1);
    if (static_cast<int>(prev) != cl - cf) return false;
    __threadfence();
    if (scratch == nullptr) return true;
    finish_tile(p, tm_count, tile, which, split_info, q, lane, scratch);
    return false;
}

__global__ void __launch_bounds__(kThreads, 1)
    w8a8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const Params p,
                const float* __restrict__ sx, int64_t ldsx, int tm_count) {
    using L = W8a8Layout;
    constexpr int kWStages = L::kWStages;
    constexpr int kXStages = L::kXStages;
    constexpr int kAcc = L::kAcc;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + L::kBarOff;
    auto wfull = [&](int s) { return bar0 + 8u * s; };
    auto wempty = [&](int s) { return bar0 + 8u * (kWStages + s); };
    auto xfull = [&](int s) { return bar0 + 8u * (2 * kWStages + s); };
    auto xempty = [&](int s) { return bar0 + 8u * (2 * kWStages + kXStages + s); };
    constexpr int kBarD = 2 * kWStages + 2 * kXStages;
    auto dfull = [&](int a) { return bar0 + 8u * (kBarD + a); };
    auto dempty = [&](int a) { return bar0 + 8u * (kBarD + kAcc + a); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = gemm::unit_begin(cta, p.U, p.G);
    const long long u1 = gemm::unit_begin(cta + 1, p.U, p.G);
    const int nunits = static_cast<int>(u1 - u0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(wfull(s), 1);
            mbar_init(wempty(s), 1);   // commit: the unit's MMAs are complete
        }
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(xfull(s), 1);
            mbar_init(xempty(s), 1 + 4);   // the MMA commit and the four fold warps (scales read)
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(dfull(a), 1);
            mbar_init(dempty(a), 4);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncwarp();
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{p.timeout_ns, p.status, abort_flag};
    grid_dependents_launch();

    if (warp == kWarpWProd) {
        // ------------------------------------------------------------ weight producer
        if (lane == 0) {
            prefetch_tmap(&tmW);
            const uint64_t pol_w = policy_evict_first();
            int issued = 0;
            Cursor cur(u0, p.KB);
            for (int i = 0; i < nunits; ++i, cur.step(p.KB)) {
                const int s = i % kWStages;
                if (i >= kWStages && !wait_bounded(wempty(s), ((i / kWStages) - 1) & 1, wc)) break;
                if (cta == 0 && i == p.fault_unit) continue;   // failure-path test hook
                const int tn = cur.tile / tm_count;
                mbar_arrive_expect_tx(wfull(s), L::kWBytes);
                tma_load_2d(base + s * L::kWBytes, &tmW, wfull(s), cur.kr * 128, tn * 128, pol_w);
                issued = i + 1;
            }
            for (int i = issued - kWStages < 0 ? 0 : issued - kWStages; i < issued; ++i) {
                if (cta == 0 && i == p.fault_unit) continue;
                gemm::drain_wait(wfull(i % kWStages), (i / kWStages) & 1, p.timeout_ns);
            }
        }
    } else if (warp == kWarpXProd) {
        // ------------------------------------------------------------ activation producer
        if (lane == 0) {
            prefetch_tmap(&tmX);
            // Xq and its scales may be the output of the preceding grid
            grid_dependency_wait();
            const uint64_t pol_x = policy_evict_last();
            int issued = 0;
            Cursor cur(u0, p.KB);
            for (int i = 0; i < nunits; ++i, cur.step(p.KB)) {
                const int s = i % kXStages;
                if (i >= kXStages && !wait_bounded(xempty(s), ((i / kXStages) - 1) & 1, wc)) break;
                const int tm = cur.tile - (cur.tile / tm_count) * tm_count;
                const uint32_t dst = base + L::kXOff + s * L::kXSlot;
                mbar_arrive_expect_tx(xfull(s), L::kXBytes + kNA * 4);
                tma_load_2d(dst, &tmX, xfull(s), cur.kr * 128, tm * kNA, pol_x);
                bulk_load(dst + L::kXBytes, sx + static_cast<int64_t>(cur.kr) * ldsx + tm * kNA, kNA * 4, xfull(s),
                          pol_x);
                issued = i + 1;
            }
            for (int i = issued - kXStages < 0 ? 0 : issued - kXStages; i < issued; ++i)
                gemm::drain_wait(xfull(i % kXStages), (i / kXStages) & 1, p.timeout_ns);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        const bool elected = elect_one();
        constexpr uint32_t idesc = idesc_f8_e4m3(kNA);
        const uint64_t dw0 = smem_desc_sw128(base);
        const uint64_t dx0 = smem_desc_sw128(base + L::kXOff);
        int last = -1;
        for (int i = 0; i < nunits; ++i) {
            const int sw = i % kWStages;
            const int sx_ = i % kXStages;
            const int a = i % kAcc;
            if (!gemm::warp_wait(wfull(sw), (i / kWStages) & 1, wc)) break;
            if (!gemm::warp_wait(xfull(sx_), (i / kXStages) & 1, wc)) break;
            if (i >= kAcc && !gemm::warp_wait(dempty(a), ((i / kAcc) - 1) & 1, wc)) break;
            tc_fence_after();
            const uint64_t ad = dw0 + static_cast<uint64_t>((sw * L::kWBytes) >> 4);
            const uint64_t bd = dx0 + static_cast<uint64_t>((sx_ * L::kXSlot) >> 4);
            if (elected) {
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_ss_f8(tmem + a * kNA, ad + 2 * j, bd + 2 * j, idesc, j > 0 ? 1u : 0u);
                tc_commit(wempty(sw));
                tc_commit(xempty(sx_));
                tc_commit(dfull(a));
            }
            __syncwarp();
            last = i;
        }
        if (last >= 0 && elected) gemm::drain_wait(dfull(last % kAcc), (last / kAcc) & 1, p.timeout_ns);
    } else if (warp >= kWarpFold0) {
        // ------------------------------------------------------------ fold / epilogue
        const int q = warp & 3;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const int first_tile = static_cast<int>(u0 / p.KB);
        const int split_info = gemm::split_info_lane(p, u0, u1, lane);
        // Y and the workspace may still be in use by the preceding grid
        grid_dependency_wait();
        bool deferred = false;
        float outer[kNA];
#pragma unroll
        for (int m = 0; m < kNA; ++m) outer[m] = 0.0f;
        Cursor cur(u0, p.KB);
        for (int i = 0; i < nunits; ++i, cur.step(p.KB)) {
            const int a = i % kAcc;
            const int sx_ = i % kXStages;
            // the unit's weight block scale (one per 128 x 128 block)
            const int tn = cur.tile / tm_count;
            const float sw = __ldg(p.S + static_cast<int64_t>(tn) * p.lds + cur.kr);
            if (!gemm::warp_wait(dfull(a), (i / kAcc) & 1, wc)) break;
            // the scales came with the slice (async proxy): observe its barrier too
            if (!gemm::warp_wait(xfull(sx_), (i / kXStages) & 1, wc)) break;
            tc_fence_after();
            uint32_t v0[16], v1[16];
            tmem_ld_x16(tl + a * kNA, v0);
            tmem_ld_x16(tl + a * kNA + 16, v1);
            // the unit's activation scales, one per row of the block
            const float4* f4 = reinterpret_cast<const float4*>(gbase + L::kXOff + sx_ * L::kXSlot + L::kXBytes);
            float f[kNA];
#pragma unroll
            for (int j = 0; j < kNA / 4; ++j) {
                const float4 t = f4[j];
                f[4 * j] = t.x;
                f[4 * j + 1] = t.y;
                f[4 * j + 2] = t.z;
                f[4 * j + 3] = t.w;
            }
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(dempty(a));
                mbar_arrive(xempty(sx_));
            }
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                outer[m] = __fmaf_rn(__uint_as_float(v0[m]), __fmul_rn(f[m], sw), outer[m]);
                outer[m + 16] = __fmaf_rn(__uint_as_float(v1[m]), __fmul_rn(f[m + 16], sw), outer[m + 16]);
            }

            if (cur.kb != p.KB - 1 && i != nunits - 1) continue;
            // after the CTA's last unit the weight ring is idle: the reduction may use it
            const bool last = i == nunits - 1;
            if (end_piece(p, tm_count, outer, cur.tile, cur.kb, u0 + i, u0, first_tile, split_info, q, lane,
                          last ? gbase : nullptr))
                deferred = true;
            if (last && deferred) finish_tile(p, tm_count, first_tile, 0, split_info, q, lane, gbase);
#pragma unroll
            for (int m = 0; m < kNA; ++m) outer[m] = 0.0f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// One warp per (row m, 128-wide K block kb) of X: block maximum, scale
// amax / 448 (1 for an all-zero block), codes E4M3 RNE-satfinite of x / s.
// Lane l handles elements 4l .. 4l+3 of the block.  Rows [M, ldsx) of every
// scale column are written as 0.
__global__ void quantize_act_kernel(const uint16_t* __restrict__ X, int64_t ldx, uint8_t* __restrict__ Xq,
                                    int64_t ldxq, float* __restrict__ Sx, int64_t ldsx, int M, int K) {
    const int lane = threadIdx.x & 31;
    const int KB = (K + 127) / 128;
    // the GEMM that consumes Xq may be scheduled now; X may be the output of
    // the preceding grid
    grid_dependents_launch();
    grid_dependency_wait();
    const int64_t job = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t jobs = static_cast<int64_t>(KB) * ldsx;
    if (job >= jobs) return;
    const int kb = static_cast<int>(job / ldsx);
    const int m = static_cast<int>(job - static_cast<int64_t>(kb) * ldsx);
    if (m >= M) {
        if (lane == 0) Sx[static_cast<int64_t>(kb) * ldsx + m] = 0.0f;
        return;
    }
    // K is a multiple of 16, so a lane's four elements are all in range or all out
    const int k0 = kb * 128 + lane * 4;
    const bool in = k0 < K;
    uint2 raw = make_uint2(0u, 0u);
    if (in) raw = *reinterpret_cast<const uint2*>(X + static_cast<int64_t>(m) * ldx + k0);
    const float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                        __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(__fdiv_rn(x[1], s)), "f"(__fdiv_rn(x[0], s)));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(__fdiv_rn(x[3], s)), "f"(__fdiv_rn(x[2], s)));
    if (in)
        *reinterpret_cast<uint32_t*>(Xq + static_cast<int64_t>(m) * ldxq + k0) =
            static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    if (lane == 0) Sx[static_cast<int64_t>(kb) * ldsx + m] = s;
}

}  // namespace

cudaError_t launch_w8a8(const W8a8Args& a, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                        const LaunchCtl& c, cudaStream_t st) {
    using L = W8a8Layout;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(w8a8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    gemm::Params p = gemm::base_params(s, a.Y, a.ldy, a.M, a.N, a.K, a.ws, c);
    p.S = a.S;
    p.lds = (a.K + 127) / 128;
    const int tm_count = (a.M + kNA - 1) / kNA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s.G));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (c.overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, w8a8_kernel, tmW, tmX, p, a.Sx, a.ldsx, tm_count);
}

cudaError_t launch_quantize_act(const void* X, int64_t ldx, void* Xq, int64_t ldxq, float* Sx, int64_t ldsx, int M,
                                int K, const LaunchCtl& c, cudaStream_t st) {
    const int64_t jobs = static_cast<int64_t>((K + 127) / 128) * ldsx;
    const int64_t blocks = (jobs * 32 + 255) / 256;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (c.overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, quantize_act_kernel, static_cast<const uint16_t*>(X), ldx,
                              static_cast<uint8_t*>(Xq), ldxq, Sx, ldsx, M, K);
}

}  // namespace qg
