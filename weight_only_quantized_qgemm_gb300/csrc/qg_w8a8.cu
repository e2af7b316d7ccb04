// W8A8 block-scaled GEMM for sm_103a: FP8 activations as well as FP8
// weights, for batches beyond the decode tier ("arc" PR page, the cuBLASLt
// block-scale section: block-scaled FP8 takes FP8 activations, hence an
// activation quantiser).
//
//   Xq, sx = quantise(X):  per (row m, 128-wide K block kb)
//            sx[kb, m] = amax / 448,  xq = e4m3_rne_satfinite(x / sx)
//   Y[m, n] = bf16( sum_kb (sx[kb, m] * s[n/128, kb]) * (sum_{k in kb} xq[m,k] * w[n,k]) )
//
// The GEMM tiles the output in 128 weight rows x NA activation rows (NA = 64
// or 128: the MMA's N side); a unit is one tile x two 128-wide K blocks (two
// blocks per unit halve the barrier rounds per MMA).  Both operands go to
// tcgen05.mma kind::f8f6f4 as stored (TMA, 128-byte swizzle).  Each K
// block's sums land in their own TMEM accumulator; the fold multiplies them
// by the block's NA factors (activation scale x weight scale) once and adds
// them to FP32 outer sums held in registers: the two-level fold of the
// W8A16 path.  Tiles are numbered weight-tile-major, so
// the activation-row blocks of a weight tile are neighbours and its weights
// come from L2 after the first read.  Work units are split evenly over the
// CTAs (stream-K), a tile shared by several CTAs being summed by the last to
// arrive, as in the decode kernels, with partial sums kept per fold warp.
//
// One persistent CTA per SM, 4 + NA/16 warps:
//   warp 0      weight producer: two 128 x 128 TMA boxes per unit (a box
//               past K reads as zeros).
//   warp 1      activation producer, after the grid dependency wait: the
//               unit's two NA x 128 E4M3 boxes (TMA) and the NA activation
//               scales of each existing block (bulk copies) into a ring.
//   warp 2      MMA issuer: 8 tcgen05.mma (M = 128, N = NA, K = 32) per unit,
//               four per K block into that block's accumulator.
//   warp 3      factor warp: turns the unit's activation scales into block
//               factors (times the unit's weight scale, fetched 32 units
//               ahead, one unit per lane) in a ring of its own, so that an
//               activation slot is free again as soon as its MMAs complete.
//   warps 4-    fold / epilogue: NA/16 warps, warp w reading TMEM lane
//               quadrant w % 4 and 64 of the NA columns; a finished tile's
//               outputs go out through shared memory by TMA stores.
#include "qg_gemm.cuh"
#include "qg_w8a8.h"

namespace qg {
namespace {

using gemm::Cursor;
using gemm::Params;

constexpr int kWarpWProd = 0, kWarpXProd = 1, kWarpMma = 2, kWarpFactor = 3, kWarpFold0 = 4;
constexpr int kFoldCols = 64;   // activation rows (MMA columns) per fold warp
constexpr int kBlk = 2;         // 128-wide K blocks per unit

template <int NA>
struct W8a8Layout {
    static constexpr int kFold = NA / 16;                     // fold warps: 4 quadrants x NA/64 column halves
    static constexpr int kThreads = 32 * (kWarpFold0 + kFold);
    static constexpr int kWBox = 128 * 128;                   // one 128 x 128 E4M3 weight block
    static constexpr int kWBytes = kBlk * kWBox;              // one unit of weights
    static constexpr int kXBox = NA * 128;                    // one NA x 128 E4M3 activation block
    static constexpr int kXBytes = kBlk * kXBox;
    static constexpr int kXSlot = kXBytes + 1024;             // + kBlk x NA scales, padded to keep 1024-B alignment
    static constexpr int kXStages = NA == 128 ? 3 : 5;
    static constexpr int kAcc = 512 / (kBlk * NA);            // TMEM accumulator sets (kBlk x NA columns each)
    static constexpr int kGStages = 2 * kAcc;                 // factor ring (kBlk x NA floats a slot)
    static constexpr int kGSlot = kBlk * NA * 4;
    // per fold warp, two output staging buffers of 32 weight rows x 16
    // activation rows of BF16 (the boxes of the TMA stores of Y)
    static constexpr int kStageBuf = 32 * 16 * 2;
    static constexpr int kStageWarp = 2 * kStageBuf;
    static constexpr int kReserve = kGStages * kGSlot + kFold * kStageWarp + 8 * 96 + 64 + 1024;   // + barriers, misc, alignment
    static constexpr int kWFit = (232448 - kXStages * kXSlot - kReserve) / kWBytes;
    static constexpr int kWStages = kWFit < 12 ? kWFit : 12;
    static constexpr int kXOff = kWStages * kWBytes;
    static constexpr int kGOff = kXOff + kXStages * kXSlot;
    static constexpr int kStageOff = kGOff + kGStages * kGSlot;
    static constexpr int kBarOff = kStageOff + kFold * kStageWarp;
    static constexpr int kNumBars = 2 * kWStages + 2 * kXStages + 2 * kGStages + 2 * kAcc;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 64 + 1024;
    // the final split-K reduction stages pieces in both idle operand rings:
    // per fold warp, pieces of 32 rows x 64 columns of FP32
    static constexpr int kPieceBytes = 32 * kFoldCols * 4;
    static constexpr int kScratchWarp = kGOff / kFold / kPieceBytes * kPieceBytes;
    static_assert(kNumBars <= 96, "barrier area");
    static_assert(kWStages >= 3, "weight ring");
    static_assert(kBlk * NA * 4 <= 1024, "scales fit the slot's padding");
    static_assert(kXOff % 1024 == 0 && kXSlot % 1024 == 0, "keep the 1024-byte swizzle alignment");
    static_assert(kScratchWarp >= 2 * kPieceBytes, "reduction scratch");
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(NA <= kMaxTileRows, "workspace slots");
};

// Workspace: partial sums [G][2 slots][NA/4 column groups][128 rows] float4
// (slots sized for the widest tile, so that the counters behind them sit at
// one offset for every W8A8 shape), then one arrival counter per (tile, fold
// warp).
template <int NA>
__device__ __forceinline__ float4* part_slot(const Params& p, int cta, int which) {
    return reinterpret_cast<float4*>(p.part) + (static_cast<size_t>(cta) * 2 + which) * (NA / 4) * 128;
}

// Where a fold warp's outputs go: through its staging buffers and TMA
// stores of the Y map (Y 16-byte aligned, ldy and N multiples of 8), else by
// plain stores.
struct YOut {
    const CUtensorMap* map;
    int tma;
    uint8_t* stage;      // the warp's two staging buffers
};

// Output rows of tile t = (weight tile tn, activation row block tm), t = tn *
// tm_count + tm: weight row n = tn * 128 + row, activation rows tm * NA + h *
// 64 + j for the fold warp's column half h (row = q * 32 + lane).
//
// TMA path: four boxes of 32 weight rows x 16 activation rows, staged as
// [m][n] BF16 (64 bytes per activation row) in two alternating buffers; a
// buffer is rewritten once the store issued from it two boxes earlier has
// read it.  The store skips rows m >= M and columns n >= N.  The stores are
// asynchronous, so the fold goes on while they drain (scattered 2-byte
// stores held the fold warps for microseconds per tile, with the MMAs
// waiting behind them).
template <int NA>
__device__ __forceinline__ void store_cols(const Params& p, const YOut& yo, int tm_count, int tile, int row, int h,
                                           const float (&v)[kFoldCols]) {
    const int tn = tile / tm_count;
    const int m0 = (tile - tn * tm_count) * NA + h * kFoldCols;
    const int n = tn * 128 + row;
    if (yo.tma) {
        const int lane = row & 31;
#pragma unroll
        for (int r = 0; r < kFoldCols / 16; ++r) {
            uint8_t* buf = yo.stage + (r & 1) * (32 * 16 * 2);
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                *reinterpret_cast<__nv_bfloat16*>(buf + j * 64 + lane * 2) = __float2bfloat16_rn(v[16 * r + j]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // lane 0's n is the box's first column; a box wholly outside Y
                // is not issued, but its (empty) group keeps the alternation
                if (n < p.N && m0 + 16 * r < p.M) tma_store_2d(yo.map, smem_u32(buf), n, m0 + 16 * r);
                bulk_commit();
            }
        }
        return;
    }
    if (n >= p.N) return;
    const gemm::Seg sg = p.seg[0];
    __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(sg.Y);
#pragma unroll
    for (int j = 0; j < kFoldCols; ++j)
        if (m0 + j < p.M) Y[static_cast<int64_t>(m0 + j) * sg.ldy + n] = __float2bfloat16_rn(v[j]);
}

// Sum of a split tile's pieces for the fold warp's 32 rows x 64 columns, in
// ascending piece order, staged through idle shared memory (batches of
// pieces copied by 16-byte cp.async before any is read back), then stored;
// resets the warp's arrival counter.
template <int NA>
__device__ __forceinline__ void finish_tile(const Params& p, const YOut& yo, int tm_count, int tile, int which,
                                            int split_info, int q, int h, int fw, int lane, uint8_t* scratch) {
    using L = W8a8Layout<NA>;
    constexpr int kF4 = kFoldCols / 4;
    constexpr int kPieces = L::kScratchWarp / L::kPieceBytes;
    const int row = q * 32 + lane;
    const int cf = __shfl_sync(0xffffffffu, split_info, 3 * which);
    const int cl = __shfl_sync(0xffffffffu, split_info, 3 * which + 1);
    const int w_first = __shfl_sync(0xffffffffu, split_info, 3 * which + 2);
    const float4* mine = reinterpret_cast<const float4*>(scratch + fw * L::kScratchWarp) + lane;
    const uint32_t sq = smem_u32(mine);
    float acc[kFoldCols];
#pragma unroll
    for (int j = 0; j < kFoldCols; ++j) acc[j] = 0.0f;
    for (int c0 = cf; c0 <= cl; c0 += kPieces) {
        const int nb = cl - c0 + 1 < kPieces ? cl - c0 + 1 : kPieces;
#pragma unroll 1
        for (int b = 0; b < nb; ++b) {
            const int c2 = c0 + b;
            const float4* src = part_slot<NA>(p, c2, c2 == cf ? w_first : 0) + h * kF4 * 128 + row;
#pragma unroll
            for (int g = 0; g < kF4; ++g) cp_async_16(sq + (b * kF4 + g) * 512, src + g * 128, 16u);
        }
        cp_async_commit();
        cp_async_wait<0>();   // the lane reads back only what it copied
#pragma unroll 1
        for (int b = 0; b < nb; ++b) {
#pragma unroll
            for (int g = 0; g < kF4; ++g) {
                const float4 x = mine[(b * kF4 + g) * 32];
                acc[4 * g + 0] = __fadd_rn(acc[4 * g + 0], x.x);
                acc[4 * g + 1] = __fadd_rn(acc[4 * g + 1], x.y);
                acc[4 * g + 2] = __fadd_rn(acc[4 * g + 2], x.z);
                acc[4 * g + 3] = __fadd_rn(acc[4 * g + 3], x.w);
            }
        }
    }
    store_cols<NA>(p, yo, tm_count, tile, row, h, acc);
    __syncwarp();
    if (lane == 0) p.cnt[tile * L::kFold + fw] = 0u;   // ready for the next call
}

// End of a CTA's piece of `tile` for one fold warp.  A whole tile is stored;
// a split piece is stored to the workspace and counted; the last to arrive
// finishes the tile now when `scratch` is given, else returns true (finished
// at the end of the range, when shared memory is idle).
template <int NA>
__device__ __forceinline__ bool end_piece(const Params& p, const YOut& yo, int tm_count,
                                          const float (&outer)[kFoldCols], int tile, int kb, long long u,
                                          long long u0, int first_tile, int split_info, int q, int h, int fw,
                                          int lane, uint8_t* scratch) {
    using L = W8a8Layout<NA>;
    const int row = q * 32 + lane;
    const bool whole = (kb == p.KB - 1) && (u - kb >= u0);
    if (whole) {
        store_cols<NA>(p, yo, tm_count, tile, row, h, outer);
        return false;
    }
    const int which = (tile == first_tile) ? 0 : 1;
    float4* mine = part_slot<NA>(p, blockIdx.x, which) + h * (kFoldCols / 4) * 128 + row;
#pragma unroll
    for (int g = 0; g < kFoldCols / 4; ++g)
        __stcg(mine + g * 128, make_float4(outer[4 * g], outer[4 * g + 1], outer[4 * g + 2], outer[4 * g + 3]));
    // every lane's partial visible GPU-wide before lane 0's arrival
    __threadfence();
    __syncwarp();
    uint32_t prev = 0;
    if (lane == 0) prev = atomicAdd(p.cnt + tile * L::kFold + fw, 1u);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    const int cf = __shfl_sync(0xffffffffu, split_info, 3 * which);
    const int cl = __shfl_sync(0xffffffffu, split_info, 3 * which + 1);
    if (static_cast<int>(prev) != cl - cf) return false;
    __threadfence();
    if (scratch == nullptr) return true;
    finish_tile<NA>(p, yo, tm_count, tile, which, split_info, q, h, fw, lane, scratch);
    return false;
}

// Position of a running unit: its Cursor, its tile's (weight tile tn,
// activation row block tm) and the number of activation scales the block's
// copy takes (nsc), stepped without divisions.
template <int NA>
struct UnitPosT {
    Cursor c;
    int tn, tm, nsc;
    __device__ UnitPosT(long long u, int KB, int tm_count, int64_t ldsx) : c(u, KB) {
        tn = c.tile / tm_count;
        tm = c.tile - tn * tm_count;
        nsc = count(ldsx);
    }
    __device__ int count(int64_t ldsx) const {
        const int64_t left = ldsx - static_cast<int64_t>(tm) * NA;
        return left < NA ? static_cast<int>(left) : NA;
    }
    __device__ void next_tile(int tm_count, int64_t ldsx) {
        if (++tm == tm_count) {
            tm = 0;
            ++tn;
        }
        nsc = count(ldsx);
    }
    __device__ void step(int KB, int tm_count, int64_t ldsx) {
        c.step(KB);
        if (c.kb == 0) next_tile(tm_count, ldsx);
    }
    __device__ void advance(int n, int KB, int tm_count, int64_t ldsx) {
        const int t0 = c.tile;
        c.step(n, KB);
        for (int t = t0; t < c.tile; ++t) next_tile(tm_count, ldsx);
    }
};

template <int NA>
__global__ void __launch_bounds__(W8a8Layout<NA>::kThreads, 1)
    w8a8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmY, const Params p, const float* __restrict__ sx, int64_t ldsx,
                int tm_count, int y_tma) {
    using L = W8a8Layout<NA>;
    using UnitPos = UnitPosT<NA>;
    constexpr int kWStages = L::kWStages;
    constexpr int kXStages = L::kXStages;
    constexpr int kAcc = L::kAcc;
    constexpr int kFold = L::kFold;
    constexpr int kGStages = L::kGStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + L::kBarOff;
    auto wfull = [&](int s) { return bar0 + 8u * s; };
    auto wempty = [&](int s) { return bar0 + 8u * (kWStages + s); };
    auto xfull = [&](int s) { return bar0 + 8u * (2 * kWStages + s); };
    auto xempty = [&](int s) { return bar0 + 8u * (2 * kWStages + kXStages + s); };
    constexpr int kBarG = 2 * kWStages + 2 * kXStages;
    auto gready = [&](int j) { return bar0 + 8u * (kBarG + j); };
    auto gempty = [&](int j) { return bar0 + 8u * (kBarG + kGStages + j); };
    constexpr int kBarD = kBarG + 2 * kGStages;
    auto dfull = [&](int a) { return bar0 + 8u * (kBarD + a); };
    auto dempty = [&](int a) { return bar0 + 8u * (kBarD + kAcc + a); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMiscOff + 4);
    auto scales_at = [&](int s) {
        return reinterpret_cast<const float*>(gbase + L::kXOff + s * L::kXSlot + L::kXBytes);
    };
    auto factors_at = [&](int j) { return reinterpret_cast<float*>(gbase + L::kGOff + j * L::kGSlot); };

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
            mbar_init(xempty(s), 2);   // the MMA commit and the factor warp (scales read)
        }
        for (int j = 0; j < kGStages; ++j) {
            mbar_init(gready(j), 1);       // the factor warp
            mbar_init(gempty(j), kFold);   // every fold warp
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(dfull(a), 1);
            mbar_init(dempty(a), kFold);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncwarp();
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{p.timeout_ns, p.status, abort_flag};
    grid_dependents_launch();

    // Every role runs one iteration per unit, and a unit's MMAs take well
    // under a microsecond: the loops avoid divisions (rings and tile
    // coordinates are stepped incrementally).  The producers and the factor
    // and fold warps wait in one lane; the MMA warp waits as a whole and
    // issues from one elected lane (issuing from a lone diverged lane
    // measured about 15% slower).
    if (warp == kWarpWProd) {
        // ------------------------------------------------------------ weight producer
        if (lane == 0) {
            prefetch_tmap(&tmW);
            // a weight tile serves tm_count tiles in a row: keep it for their re-reads
            const uint64_t pol_w = tm_count > 1 ? policy_evict_last() : policy_evict_first();
            int issued = 0;
            UnitPos up(u0, p.KB, tm_count, ldsx);
            gemm::Ring<kWStages> rw(0);
            for (int i = 0; i < nunits; ++i, up.step(p.KB, tm_count, ldsx), rw.step(1)) {
                if (i >= kWStages && !wait_bounded(wempty(rw.slot), rw.phase ^ 1u, wc)) break;
                issued = i + 1;
                if (cta == 0 && i == p.fault_unit) continue;   // failure-path test hook
                // both 128 x 128 blocks of the unit (a block past K reads as zeros)
                mbar_arrive_expect_tx(wfull(rw.slot), L::kWBytes);
#pragma unroll
                for (int b = 0; b < kBlk; ++b)
                    tma_load_2d(base + rw.slot * L::kWBytes + b * L::kWBox, &tmW, wfull(rw.slot),
                                (up.c.kr * kBlk + b) * 128, up.tn * 128, pol_w);
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
            UnitPos up(u0, p.KB, tm_count, ldsx);
            gemm::Ring<kXStages> rx(0);
            for (int i = 0; i < nunits; ++i, up.step(p.KB, tm_count, ldsx), rx.step(1)) {
                if (i >= kXStages && !wait_bounded(xempty(rx.slot), rx.phase ^ 1u, wc)) break;
                const uint32_t dst = base + L::kXOff + rx.slot * L::kXSlot;
                // the unit's K blocks that exist (the last unit of a row may hold one)
                const int kb0 = up.c.kr * kBlk;
                const int nblk = p.lds - kb0 < kBlk ? p.lds - kb0 : kBlk;
                mbar_arrive_expect_tx(xfull(rx.slot), L::kXBytes + nblk * up.nsc * 4);
#pragma unroll
                for (int b = 0; b < kBlk; ++b)
                    tma_load_2d(dst + b * L::kXBox, &tmX, xfull(rx.slot), (kb0 + b) * 128, up.tm * NA, pol_x);
                for (int b = 0; b < nblk; ++b)
                    bulk_load(dst + L::kXBytes + b * NA * 4,
                              sx + static_cast<int64_t>(kb0 + b) * ldsx + static_cast<int64_t>(up.tm) * NA,
                              up.nsc * 4, xfull(rx.slot), pol_x);
                issued = i + 1;
            }
            for (int i = issued - kXStages < 0 ? 0 : issued - kXStages; i < issued; ++i)
                gemm::drain_wait(xfull(i % kXStages), (i / kXStages) & 1, p.timeout_ns);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        const bool elected = elect_one();
        constexpr uint32_t idesc = idesc_f8_e4m3(NA);
        const uint64_t dw0 = smem_desc_sw128(base);
        const uint64_t dx0 = smem_desc_sw128(base + L::kXOff);
        gemm::Ring<kWStages> rw(0);
        gemm::Ring<kXStages> rx(0);
        gemm::Ring<kAcc> ra(0);
        int last = -1;
        for (int i = 0; i < nunits; ++i, rw.step(1), rx.step(1), ra.step(1)) {
            if (!gemm::warp_wait(wfull(rw.slot), rw.phase, wc)) break;
            if (!gemm::warp_wait(xfull(rx.slot), rx.phase, wc)) break;
            if (i >= kAcc && !gemm::warp_wait(dempty(ra.slot), ra.phase ^ 1u, wc)) break;
            tc_fence_after();
            const uint64_t ad = dw0 + static_cast<uint64_t>((rw.slot * L::kWBytes) >> 4);
            const uint64_t bd = dx0 + static_cast<uint64_t>((rx.slot * L::kXSlot) >> 4);
            if (elected) {
#pragma unroll
                for (int b = 0; b < kBlk; ++b) {
                    // block b: its own accumulator of NA columns
                    const uint64_t adb = ad + static_cast<uint64_t>((b * L::kWBox) >> 4);
                    const uint64_t bdb = bd + static_cast<uint64_t>((b * L::kXBox) >> 4);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_ss_f8(tmem + (ra.slot * kBlk + b) * NA, adb + 2 * j, bdb + 2 * j, idesc, j > 0 ? 1u : 0u);
                }
                tc_commit(wempty(rw.slot));
                tc_commit(xempty(rx.slot));
                tc_commit(dfull(ra.slot));
            }
            __syncwarp();
            last = i;
        }
        if (last >= 0 && elected) gemm::drain_wait(dfull(last % kAcc), (last / kAcc) & 1, p.timeout_ns);
    } else if (warp == kWarpFactor) {
        // ------------------------------------------------------------ block factors
        // Lane l fetches the weight scales of unit i0 + l one batch of 32
        // units ahead of their use, so that no unit waits for a global load
        // (0 for a K block past the end).
        UnitPos bp(u0, p.KB, tm_count, ldsx);   // the first unit of the batch fetched next
        auto fetch = [&](int i0, float2& v) {
            v = make_float2(0.0f, 0.0f);
            if (i0 + lane < nunits) {
                UnitPos mine = bp;
                mine.advance(lane, p.KB, tm_count, ldsx);
                const int kb0 = mine.c.kr * kBlk;
                const float* srow = p.S + static_cast<int64_t>(mine.tn) * p.lds;
                v.x = __ldg(srow + kb0);
                if (kb0 + 1 < p.lds) v.y = __ldg(srow + kb0 + 1);
            }
            bp.advance(32, p.KB, tm_count, ldsx);
        };
        float2 sw_now, sw_next;
        fetch(0, sw_now);
        fetch(32, sw_next);
        UnitPos up(u0, p.KB, tm_count, ldsx);
        gemm::Ring<kXStages> rx(0);
        gemm::Ring<kGStages> rg(0);
        for (int i = 0; i < nunits; ++i, up.step(p.KB, tm_count, ldsx), rx.step(1), rg.step(1)) {
            if (i > 0 && (i & 31) == 0) {
                sw_now = sw_next;
                fetch(i + 32, sw_next);
            }
            bool ok = true;
            if (lane == 0) {
                ok = wait_bounded(xfull(rx.slot), rx.phase, wc);
                if (ok && i >= kGStages) ok = wait_bounded(gempty(rg.slot), rg.phase ^ 1u, wc);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            __syncwarp();   // orders the other lanes' reads after lane 0's wait
            const float sw0 = __shfl_sync(0xffffffffu, sw_now.x, i & 31);
            const float sw1 = __shfl_sync(0xffffffffu, sw_now.y, i & 31);
            const bool has1 = up.c.kr * kBlk + 1 < p.lds;
            const float* sc = scales_at(rx.slot);
            float* f = factors_at(rg.slot);
#pragma unroll
            for (int c = 0; c < NA / 32; ++c) {
                const int m = c * 32 + lane;
                f[m] = m < up.nsc ? __fmul_rn(sc[m], sw0) : 0.0f;
                f[NA + m] = (has1 && m < up.nsc) ? __fmul_rn(sc[NA + m], sw1) : 0.0f;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(xempty(rx.slot));
                mbar_arrive(gready(rg.slot));
            }
        }
    } else {
        // ------------------------------------------------------------ fold / epilogue
        const int fw = warp - kWarpFold0;   // 0 .. kFold-1
        const int q = warp & 3;             // TMEM lane quadrant of this warp
        const int h = fw >> 2;              // column half
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16) + h * kFoldCols;
        const int first_tile = static_cast<int>(u0 / p.KB);
        const int split_info = gemm::split_info_lane(p, u0, u1, lane);
        const YOut yo{&tmY, y_tma, gbase + L::kStageOff + fw * L::kStageWarp};
        if (y_tma && lane == 0) prefetch_tmap(&tmY);
        // Y and the workspace may still be in use by the preceding grid
        grid_dependency_wait();
        bool deferred = false;
        float outer[kFoldCols];
#pragma unroll
        for (int j = 0; j < kFoldCols; ++j) outer[j] = 0.0f;
        Cursor cur(u0, p.KB);
        gemm::Ring<kAcc> ra(0);
        gemm::Ring<kGStages> rg(0);
        for (int i = 0; i < nunits; ++i, cur.step(p.KB), ra.step(1), rg.step(1)) {
            bool ok = true;
            if (lane == 0) {
                ok = wait_bounded(dfull(ra.slot), ra.phase, wc);
                if (ok) ok = wait_bounded(gready(rg.slot), rg.phase, wc);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            __syncwarp();   // orders the other lanes' reads after lane 0's wait
            tc_fence_after();
#pragma unroll 1
            for (int b = 0; b < kBlk; ++b) {
                const float4* f4 = reinterpret_cast<const float4*>(factors_at(rg.slot) + b * NA + h * kFoldCols);
                const uint32_t tb = tl + (ra.slot * kBlk + b) * NA;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t v0[16], v1[16];
                    tmem_ld_x16(tb + 32 * c, v0);
                    tmem_ld_x16(tb + 32 * c + 16, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4 g0 = f4[8 * c + e];
                        const float4 g1 = f4[8 * c + 4 + e];
                        float* o = outer + 32 * c;
                        o[4 * e + 0] = __fmaf_rn(__uint_as_float(v0[4 * e + 0]), g0.x, o[4 * e + 0]);
                        o[4 * e + 1] = __fmaf_rn(__uint_as_float(v0[4 * e + 1]), g0.y, o[4 * e + 1]);
                        o[4 * e + 2] = __fmaf_rn(__uint_as_float(v0[4 * e + 2]), g0.z, o[4 * e + 2]);
                        o[4 * e + 3] = __fmaf_rn(__uint_as_float(v0[4 * e + 3]), g0.w, o[4 * e + 3]);
                        o[16 + 4 * e + 0] = __fmaf_rn(__uint_as_float(v1[4 * e + 0]), g1.x, o[16 + 4 * e + 0]);
                        o[16 + 4 * e + 1] = __fmaf_rn(__uint_as_float(v1[4 * e + 1]), g1.y, o[16 + 4 * e + 1]);
                        o[16 + 4 * e + 2] = __fmaf_rn(__uint_as_float(v1[4 * e + 2]), g1.z, o[16 + 4 * e + 2]);
                        o[16 + 4 * e + 3] = __fmaf_rn(__uint_as_float(v1[4 * e + 3]), g1.w, o[16 + 4 * e + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(dempty(ra.slot));
                mbar_arrive(gempty(rg.slot));
            }
            if (cur.kb != p.KB - 1 && i != nunits - 1) continue;
            // After the CTA's last unit both operand rings are idle once the
            // factor warp has read the last scales (the slot's release
            // completes; the MMAs are complete): the reduction may use them.
            const bool last = i == nunits - 1;
            if (last) {
                bool idle = true;
                if (lane == 0) idle = wait_bounded(xempty(i % kXStages), (i / kXStages) & 1, wc);
                if (!__shfl_sync(0xffffffffu, idle, 0)) break;
            }
            if (end_piece<NA>(p, yo, tm_count, outer, cur.tile, cur.kb, u0 + i, u0, first_tile, split_info, q, h,
                              fw, lane, last ? gbase : nullptr))
                deferred = true;
            if (last && deferred)
                finish_tile<NA>(p, yo, tm_count, first_tile, 0, split_info, q, h, fw, lane, gbase);
#pragma unroll
            for (int j = 0; j < kFoldCols; ++j) outer[j] = 0.0f;
        }
        // the staging buffers must have been read before the CTA's shared memory goes
        if (y_tma && lane == 0) bulk_wait_read<0>();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
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

size_t w8a8_partial_bytes(const Schedule& s) {
    return static_cast<size_t>(s.max_ctas) * 2 * 128 * kMaxTileRows * sizeof(float);
}

size_t w8a8_workspace_bytes(const Schedule& s, bool split) {
    if (!split) return 0;
    const size_t part = w8a8_partial_bytes(s);
    const size_t cnt = (static_cast<size_t>(s.T) * (s.nmma / 16) * sizeof(uint32_t) + 255) & ~static_cast<size_t>(255);
    return part + cnt;
}

template <int NA>
static cudaError_t launch_w8a8_na(const W8a8Args& a, const Schedule& s, const CUtensorMap& tmW,
                                  const CUtensorMap& tmX, const LaunchCtl& c, cudaStream_t st) {
    using L = W8a8Layout<NA>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(w8a8_kernel<NA>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    gemm::Params p = gemm::base_params(s, a.Y, a.ldy, a.M, a.N, a.K, a.ws, c);
    p.S = a.S;
    p.lds = (a.K + 127) / 128;
    uint8_t* w = static_cast<uint8_t*>(a.ws);
    p.part = reinterpret_cast<float*>(w);
    p.cnt = w ? reinterpret_cast<uint32_t*>(w + w8a8_partial_bytes(s)) : nullptr;
    const int tm_count = (a.M + NA - 1) / NA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s.G));
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (c.overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, w8a8_kernel<NA>, tmW, tmX, a.tmY, p, a.Sx, a.ldsx, tm_count, a.y_tma);
}

cudaError_t launch_w8a8(const W8a8Args& a, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                        const LaunchCtl& c, cudaStream_t st) {
    if (s.nmma == 64) return launch_w8a8_na<64>(a, s, tmW, tmX, c, st);
    if (s.nmma == 128) return launch_w8a8_na<128>(a, s, tmW, tmX, c, st);
    return cudaErrorInvalidValue;
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
