// The 3-bit learned-LUT decode GEMM pipeline for sm_103a (the FP8 format has
// its own kernel in qg_fp8.cu and shares only the parameter block, the work
// decomposition and the split-K epilogue defined here).
//
//   Y[m, n] = fp16( sum_k x[m,k] * deq(W)[n,k] )
//
// Swap-AB: a 128-row slice of W is the MMA's M side (TMEM lanes), the M <= 32
// activation rows are the MMA's narrow N side (16 or 32).  A work unit is one
// 128-row tile x one 128-wide K block.  The MMAs of a tile piece (the units of
// one tile in a CTA's range) accumulate in TMEM; the fold warps read each
// piece once.
//
// One persistent CTA per SM; warps by role (N = 16: 24 warps, 80 registers
// each; N = 32: 16 warps, 128 registers):
//   warp 0        code producer: 4 lanes in step, one bulk copy per unit
//                 (evict-first L2 hint) into a ring of up to 15 stages.  A
//                 stage is released when the dequant group has converted it.
//   last warp     X producer: 4 lanes in step, the unit's 128-wide X slice
//                 (two 64-element TMA boxes, 128-byte swizzle) into a ring held
//                 until the unit's MMAs complete.
//   warp 1 and the one before the X producer
//                 MMA issuers, unit i taken by issuer i % 2: 8 tcgen05.mma
//                 kind::f16 (M=128, N=16|32, K=16), A from TMEM, B (X) from
//                 shared memory, then the commits, from one elected lane.
//   warps 2-5     fold / epilogue, one per TMEM lane quadrant.
//   warps 6-      dequant: 4 groups (2 at N = 32) of four warps, group g
//                 taking units i with i % groups == g: shared memory ->
//                 registers -> FP16 by byte-permute lookups -> tcgen05.st into
//                 a ring of A buffers in TMEM (one per group at N = 16, three
//                 per group at N = 32).
//
// Work units are split evenly over the CTAs in tile-major order (stream-K);
// a tile shared by several CTAs is summed, in ascending K order of its
// pieces, by whichever CTA finishes its piece last (an atomic arrival
// counter; nobody spins on another CTA).  Every wait is bounded: a wait that
// runs out records a timeout in the status word, the CTA drains its own
// copies and MMAs, frees its TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {
namespace gemm {

constexpr int kWarpFold0 = 2;
constexpr int kWarpDeq0 = 6;

// Warp roles for an MMA width: dequant groups of four warps (one per TMEM lane
// quadrant) taking every kDeqGroups-th unit, then the second MMA issuer and the
// X producer.  Four groups at N = 16 (24 warps): the byte permutes of the
// dequant keep the ALU pipe busy only if enough warps convert at once (three
// groups measured 31.7 us, four 30.4 us on 28672 x 8192 at M = 16, same box).
// Two at N = 32, whose wider fold needs the registers of a 16-warp CTA.
template <int NMMA>
struct Roles {
    static constexpr int kDeqGroups = NMMA == 16 ? 4 : 2;
    static constexpr int kWarpMma2 = kWarpDeq0 + 4 * kDeqGroups;
    static constexpr int kWarpXProd = kWarpMma2 + 1;
    static constexpr int kThreads = 32 * (kWarpXProd + 1);
};
constexpr int kIssuers = 2;
constexpr int kProdLanes = 4;   // lanes of a producer warp that issue copies
constexpr unsigned kProdMask = (1u << kProdLanes) - 1u;
constexpr int kTmemCols = 512;
// Shared memory per TMEM lane quadrant that the final split-K reduction of a
// CTA may use (see sum_pieces): five pieces of 32 rows x NOUT FP32 values.
template <int NOUT>
__host__ __device__ constexpr int scratch_quadrant() { return 5 * 32 * NOUT * 4; }

// Output segments: up to kMaxSegs weight matrices that share X run as one
// grid over their concatenated 128-row tiles (e.g. the Q, K and V
// projections); a plain call is one segment.  Segment j owns tiles
// [tile0, next segment's tile0) and writes rows [0, n) of its own Y.
constexpr int kMaxSegs = 4;
struct Seg {
    int tile0;         // first tile of the segment in the grid's tile order
    int n;             // output rows (weight rows) of the segment
    const float* S;    // FP8: the segment's block scales [ceil(n/128), lds]
    void* Y;
    int64_t ldy;
};

struct Params {
    // weights
    const uint8_t* Wq;            // packed LUT3 weights (bulk copies)
    const uint4* qmap;            // LUT3 map
    const uint16_t* lut_scales;   // LUT3 per-(row, group) FP16 scales
    int64_t ld_lut_scales;
    int KT;                       // LUT3: 256-wide packed blocks per tile row
    const float* S;               // FP8 block scales
    int64_t lds;
    const void* X;                // activations (FP8 path: read by the split warps)
    int64_t ldx;
    // output and shape
    int nseg;
    Seg seg[kMaxSegs];
    int M, N, K;                  // N: rows of all segments' tiles (LUT3: its rows)
    int KB;                       // units (128-wide K blocks) per tile
    long long U;                  // total units
    int G;                        // CTAs
    float* part;                  // [G][2][128][NMMA] partial sums (scratch)
    uint32_t* cnt;                // per (tile, quadrant) arrival counters, zero between calls
    uint64_t timeout_ns;
    int fault_unit;
    uint32_t* status;
};

template <int NMMA, int WBYTES>
struct Layout {
    // TMEM: kNA A buffers (64 columns, 128 rows x 128 K of 16-bit weights),
    // then four accumulators of NMMA columns: one per MMA issuer for each of
    // two tile pieces in flight (a piece = the units of one tile in this CTA's
    // range).  The format has no per-block fold scale, so a piece's MMAs
    // accumulate in TMEM across its K blocks and the fold reads each piece
    // once instead of once per unit.  Every A buffer belongs to one dequant
    // group; four groups get one each (two each would need 512 columns before
    // the accumulators), so a group converting its next unit first waits for
    // the MMAs of its previous one.
    static constexpr int kNA = Roles<NMMA>::kDeqGroups == 4 ? 4 : 6;
    static constexpr int kDCol0 = kNA * 64;               // accumulator (b, j) at kDCol0 + NMMA (2 b + j)
    static_assert(kDCol0 + 4 * NMMA <= kTmemCols, "TMEM columns");
    static constexpr int kXSlot = NMMA * 256;             // two 64-element X boxes
    static constexpr int kXBox = NMMA * 128;
    // X slots: enough for the X copies (L2 hits) to run ahead of the MMAs
    // (and for the final split-K reduction's staging); the rest of the budget
    // goes to the weight ring.
    static constexpr int kXStages = 12;
    static constexpr int kWBudget = 212992 - kXStages * kXSlot;   // 208 KB in all
    // A multiple of the dequant group count, so that every use of a weight stage
    // falls to the same dequant group (units i and i + kWStages are taken by
    // the same group).  A group's parity wait on a stage is then always for the
    // phase right after one it has already seen; otherwise it could be for a
    // phase after another group's still-pending one, and a parity wait cannot
    // tell those two apart.
    static constexpr int kG = Roles<NMMA>::kDeqGroups;
    // At most 15 stages.  Measured on the 28672 x 8192 shape at M = 16 (code
    // stages x X slots): 15 x 12 32.7 us, 12 x 12 32.9, 18 x 12 32.9, 15 x 6
    // 33.0, 18 x 6 33.1, 21 x 6 33.1, 9 x 18 34.8.
    static constexpr int kWFit = (kWBudget / WBYTES) < 15 ? (kWBudget / WBYTES) : 15;
    static constexpr int kWStages = kWFit / kG * kG;
    static constexpr int kXOff = kWStages * WBYTES;
    static constexpr int kBarOff = kXOff + kXStages * kXSlot;
    static constexpr int kNumBars = 2 * kWStages + 2 * kXStages + 2 * kNA + 6;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 64 + 1024;  // + alignment slack
    static_assert(WBYTES % 1024 == 0 && kXSlot % 1024 == 0, "keep the 1024-byte swizzle alignment");
    static_assert(kXStages >= kNA, "X copies run at least as far ahead as the dequant");
    // the same ownership rule for the other rings: an X stage and an A buffer
    // are always used by the same MMA issuer and the same dequant group
    static_assert(kXStages % kIssuers == 0 && kNA % kIssuers == 0 && kNA % kG == 0, "ring ownership");
    static_assert(kWStages >= 8, "the weight ring must cover HBM latency");
    static_assert(kWStages % kG == 0, "a weight stage must belong to one dequant group");
    static_assert(kWStages > kProdLanes && kXStages > kProdLanes, "a stage's previous unit is issued in an earlier pass");
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(kXStages * kXSlot >= 4 * scratch_quadrant<NMMA>(), "reduction scratch in the X ring");
};

__device__ __forceinline__ int unit_owner(long long x, long long U, int G) {
    return static_cast<int>(((x + 1) * G - 1) / U);
}

__device__ __forceinline__ long long unit_begin(int c, long long U, int G) {
    return static_cast<long long>(c) * U / G;
}

// (tile, K block) of a running unit index, advanced without divisions (a 64-bit
// division costs hundreds of cycles and used to dominate the per-unit loops).
// kb is the unit's place in its tile's K order (which decides where pieces
// end); kr is the K block it actually covers: tile t takes its blocks in the
// order t mod KB, t mod KB + 1, ..., wrapping around, so that at any moment
// the CTAs streaming different tiles read different slices of X instead of
// all hitting the same few L2 lines.
struct Cursor {
    int tile, kb, kr;
    __device__ static int first_block(int tile, int KB) { return tile % KB; }
    __device__ Cursor(long long u, int KB) : tile(static_cast<int>(u / KB)), kb(static_cast<int>(u % KB)) {
        kr = kb + first_block(tile, KB);
        if (kr >= KB) kr -= KB;
    }
    __device__ void step(int KB) {
        if (++kr == KB) kr = 0;
        if (++kb == KB) {
            kb = 0;
            ++tile;
            kr = first_block(tile, KB);
        }
    }
    __device__ void step(int n, int KB) {
        kb += n;
        if (kb < KB) {
            kr += n;
            while (kr >= KB) kr -= KB;
            return;
        }
        while (kb >= KB) {
            kb -= KB;
            ++tile;
        }
        kr = kb + first_block(tile, KB);
        if (kr >= KB) kr -= KB;
    }
};

// Slot of a ring of N slots and the parity of that slot's current use, for a
// running unit index advanced by a fixed stride: i % N and (i / N) & 1 kept
// incrementally (divisions by ring sizes that are not powers of two cost a
// handful of integer instructions per use, on the pipe the dequantiser needs).
template <int N>
struct Ring {
    int slot;
    uint32_t phase;
    __device__ explicit Ring(int i) : slot(i % N), phase(static_cast<uint32_t>((i / N) & 1)) {}
    __device__ __forceinline__ void step(int d) {   // d <= N
        slot += d;
        if (slot >= N) {
            slot -= N;
            phase ^= 1u;
        }
    }
};

// Warp-uniform bounded wait: every lane polls, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& c) {
    const bool ok = wait_bounded(bar, parity, c);
    return __all_sync(0xffffffffu, ok);
}

// Wait used only while draining before exit: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if (globaltimer() - t0 > timeout_ns) return;
    }
}

// The (cf, cl, slot) lanes of a CTA's first and last tile (see end_piece).
__device__ __forceinline__ int split_info_lane(const Params& p, long long u0, long long u1, int lane) {
    int v = 0;
    if (lane < 6) {
        const long long t = lane < 3 ? u0 / p.KB : (u1 - 1) / p.KB;
        const long long t0 = t * p.KB;
        const int cf = unit_owner(t0, p.U, p.G);
        if (lane % 3 == 0) v = cf;
        if (lane % 3 == 1) v = unit_owner(t0 + p.KB - 1, p.U, p.G);
        if (lane % 3 == 2) v = unit_begin(cf, p.U, p.G) == t0 ? 0 : 1;
    }
    return v;
}

// The segment holding `tile` (constant-index selects: a dynamic index into
// the kernel parameters would go through local memory).
__device__ __forceinline__ Seg seg_of(const Params& p, int tile) {
    Seg r = p.seg[0];
#pragma unroll
    for (int j = 1; j < kMaxSegs; ++j)
        if (j < p.nseg && tile >= p.seg[j].tile0) r = p.seg[j];
    return r;
}

// Rows [m < M] of output row `row` of `tile` (its segment's Y and row index).
template <int NOUT, class Store>
__device__ __forceinline__ void store_rows(const Params& p, int tile, int row, const float (&v)[NOUT]) {
    const Seg sg = seg_of(p, tile);
    const int n = (tile - sg.tile0) * 128 + row;
    if (n < sg.n) {
#pragma unroll
        for (int m = 0; m < NOUT; ++m)
            if (m < p.M) Store::store(sg.Y, static_cast<int64_t>(m) * sg.ldy + n, v[m]);
    }
}

// Slot of CTA c2's piece of the tile: cf's piece may be in its second slot
// (w_first), every later contributor's is in its first.
template <int NOUT>
__device__ __forceinline__ const float4* piece_slot(const Params& p, int row, int c2, int cf, int w_first) {
    return reinterpret_cast<const float4*>(p.part) +
           ((static_cast<size_t>(c2) * 2 + (c2 == cf ? w_first : 0)) * 128 + row) * (NOUT / 4);
}

// Split-K partial sums live in the workspace as [slot][column group g][row]
// float4s (g = 4 columns): for each column group the 32 lanes of a TMEM lane
// quadrant, one output row per lane, touch 512 contiguous bytes.  (Row-major
// partials made every 16-byte access of a warp hit 32 different L2 lines.)
template <int NOUT>
__device__ __forceinline__ float4* slot_base(const Params& p, int cta, int which) {
    return reinterpret_cast<float4*>(p.part) + (static_cast<size_t>(cta) * 2 + which) * (NOUT / 4) * 128;
}

// Slot of CTA c2's piece of the tile: cf's piece may be in its second slot
// (w_first), every later contributor's is in its first.
template <int NOUT>
__device__ __forceinline__ const float4* piece_slot(const Params& p, int c2, int cf, int w_first) {
    return slot_base<NOUT>(p, c2, c2 == cf ? w_first : 0);
}

// Sum of the pieces [cf, cl] of a split tile for the lane's output row, in
// ascending piece order, into acc.  The pieces are staged through shared
// memory that is idle by the end of the CTA's range (scratch_quadrant<NOUT>()
// bytes per TMEM lane quadrant, laid out [piece][column group][lane] so that
// a warp's accesses are conflict-free): every lane copies a batch of pieces
// (up to five) with 16-byte cp.async copies before reading any back, so that
// a batch costs one L2 round trip.
template <int NOUT>
__device__ __forceinline__ void sum_pieces_staged(const Params& p, int row, int lane, int q, int cf, int cl,
                                                  int w_first, uint8_t* scratch, float (&acc)[NOUT]) {
    constexpr int kF4 = NOUT / 4;
    constexpr int kPieces = scratch_quadrant<NOUT>() / (32 * NOUT * 4);
    const float4* mine = reinterpret_cast<const float4*>(scratch + q * scratch_quadrant<NOUT>()) + lane;
    const uint32_t sq = smem_u32(mine);
#pragma unroll
    for (int m = 0; m < NOUT; ++m) acc[m] = 0.0f;
    for (int c0 = cf; c0 <= cl; c0 += kPieces) {
        const int nb = cl - c0 + 1 < kPieces ? cl - c0 + 1 : kPieces;
#pragma unroll 1
        for (int b = 0; b < nb; ++b) {
            const float4* src = piece_slot<NOUT>(p, c0 + b, cf, w_first) + row;
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
}

// A CTA ends a split piece only in its first and its last tile.  For both,
// the first and last contributing CTAs (cf, cl) and the slot holding cf's
// piece (slot 0 when the tile is cf's first tile, i.e. when cf's range starts
// exactly at the tile; every later contributor's range starts inside the
// tile, so their pieces are all in slot 0) are worked out once per CTA,
// before any unit is ready, so that the 64-bit divisions stay out of the
// reduction.  Lane 3w + k holds value k (cf, cl, slot) of the first (w = 0) or
// last (w = 1) tile; the reduction fetches them by shuffle.
//
// The last of a tile's CTAs to arrive sums every piece in ascending K order
// and stores the tile (finish_tile).  The sum is staged through shared memory
// that is idle only after the CTA's last unit, so a CTA that arrives last at
// its first tile in the middle of its range defers that reduction to the end
// of its range (the tile's pieces and counter stay as they are until then).

// Sum and store of split tile `tile` (`which`: 0 = the CTA's first tile, 1 =
// its last) by its last-arriving CTA; resets the tile's arrival counter.
template <int NOUT, class Store>
__device__ __forceinline__ void finish_tile(const Params& p, int tile, int which, int split_info, int q, int lane,
                                            uint8_t* scratch) {
    const int row = q * 32 + lane;
    const int cf = __shfl_sync(0xffffffffu, split_info, 3 * which);
    const int cl = __shfl_sync(0xffffffffu, split_info, 3 * which + 1);
    const int w_first = __shfl_sync(0xffffffffu, split_info, 3 * which + 2);
    float acc[NOUT];
    sum_pieces_staged<NOUT>(p, row, lane, q, cf, cl, w_first, scratch, acc);
    store_rows<NOUT, Store>(p, tile, row, acc);
    __syncwarp();
    if (lane == 0) p.cnt[tile * 4 + q] = 0u;   // ready for the next call
}

// End of a CTA's piece of `tile` (one warp, TMEM lane quadrant q, one output
// row per lane).  A whole tile is stored directly.  A split piece goes to the
// workspace and counts its arrival; the last to arrive finishes the tile now
// when `scratch` (shared memory no longer in use) is given, and otherwise
// returns true: the caller finishes the tile at the end of its range.
// Store::store(Y, index, value) writes one output element.
template <int NOUT, class Store>
__device__ __forceinline__ bool end_piece(const Params& p, const float (&outer)[NOUT], int tile, int kb,
                                          long long u, long long u0, int first_tile, int split_info, int q,
                                          int lane, uint8_t* scratch) {
    const int row = q * 32 + lane;
    const int cta = blockIdx.x;
    const bool whole = (kb == p.KB - 1) && (u - kb >= u0);
    if (whole) {
        store_rows<NOUT, Store>(p, tile, row, outer);
        return false;
    }
    const int which = (tile == first_tile) ? 0 : 1;
    float4* mine = slot_base<NOUT>(p, cta, which) + row;
#pragma unroll
    for (int g = 0; g < NOUT / 4; ++g)
        __stcg(mine + g * 128, make_float4(outer[4 * g], outer[4 * g + 1], outer[4 * g + 2], outer[4 * g + 3]));
    // Every lane's partial must be visible GPU-wide before lane 0's arrival: a
    // sequentially consistent fence per writing lane (an acquire-release fence
    // is not enough, since the lanes that wrote are not the lane that performs
    // the atomic).
    __threadfence();
    __syncwarp();
    uint32_t prev = 0;
    if (lane == 0) prev = atomicAdd(p.cnt + tile * 4 + q, 1u);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    const int cf = __shfl_sync(0xffffffffu, split_info, 3 * which);
    const int cl = __shfl_sync(0xffffffffu, split_info, 3 * which + 1);
    if (static_cast<int>(prev) != cl - cf) return false;
    // last piece to arrive: every other piece is visible
    __threadfence();
    if (scratch == nullptr) return true;
    finish_tile<NOUT, Store>(p, tile, which, split_info, q, lane, scratch);
    return false;
}

template <int NMMA, class F>
__global__ void __launch_bounds__(Roles<NMMA>::kThreads, 1)
    qgemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 const Params p) {
    using L = Layout<NMMA, F::kStageBytes>;
    constexpr int kDeqGroups = Roles<NMMA>::kDeqGroups;
    constexpr int kWarpMma2 = Roles<NMMA>::kWarpMma2;
    constexpr int kWarpXProd = Roles<NMMA>::kWarpXProd;
    constexpr int kWStages = L::kWStages;
    constexpr int kXStages = L::kXStages;
    constexpr int kNA = L::kNA;
    constexpr int kDCol0 = L::kDCol0;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + L::kBarOff;
    auto wfull = [&](int s) { return bar0 + 8u * s; };
    auto wempty = [&](int s) { return bar0 + 8u * (kWStages + s); };
    auto xfull = [&](int s) { return bar0 + 8u * (2 * kWStages + s); };
    auto xempty = [&](int s) { return bar0 + 8u * (2 * kWStages + kXStages + s); };
    constexpr int kBarA = 2 * kWStages + 2 * kXStages;
    auto afull = [&](int a) { return bar0 + 8u * (kBarA + a); };
    auto afree = [&](int a) { return bar0 + 8u * (kBarA + kNA + a); };
    // accumulator (b, j) of piece buffer b, issuer j: complete / drained
    auto dfull = [&](int b, int j) { return bar0 + 8u * (kBarA + 2 * kNA + 2 * b + j); };
    auto dempty = [&](int b) { return bar0 + 8u * (kBarA + 2 * kNA + 4 + b); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = unit_begin(cta, p.U, p.G);
    const long long u1 = unit_begin(cta + 1, p.U, p.G);
    const int nunits = static_cast<int>(u1 - u0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(wfull(s), 1);
            mbar_init(wempty(s), 4);   // the four warps of the dequant group that read it
        }
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(xfull(s), 1);
            mbar_init(xempty(s), 1);   // commit: the unit's MMAs are complete
        }
        for (int a = 0; a < kNA; ++a) {
            mbar_init(afull(a), 4);   // the four warps of the dequant group
            mbar_init(afree(a), 1);   // commit: the unit's MMAs are complete
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(dfull(b, 0), 1);   // commit: the issuer's last MMAs of the piece are complete
            mbar_init(dfull(b, 1), 1);
            mbar_init(dempty(b), 4);     // the four fold warps
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
    // The next grid on the stream may be scheduled now; its CTAs start as ours
    // exit, and only its weight stream runs before it waits for this grid.
    grid_dependents_launch();

    if (warp == 0) {
        // ------------------------------------------------------------ weight producer
        // kProdLanes lanes issue kProdLanes consecutive units per pass of the
        // loop, so one pass of its bookkeeping starts kProdLanes copies: a
        // single producing thread, sharing its scheduler with three dequant
        // warps, could not issue a copy as often as the dequant consumes one.
        // The lanes move in step.  A lane waiting for the release of unit
        // i - kWStages then knows that unit i - 2 kWStages was released (unit
        // i - kWStages was issued in an earlier pass, after that release), so
        // the parity of its wait cannot match an older phase of the stage.
        if (lane < kProdLanes) {
            if (F::kUsesTensorMapW && lane == 0) prefetch_tmap(&tmW);
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_s = policy_evict_last();   // a scale box serves 8 units
            int last = -1;   // the last unit this lane issued
            Cursor cur(u0 + lane, p.KB);
            Ring<kWStages> rw(lane);
            for (int i0 = 0; i0 < nunits; i0 += kProdLanes, cur.step(kProdLanes, p.KB), rw.step(kProdLanes)) {
                const int i = i0 + lane;
                const int s = rw.slot;
                const bool mine = i < nunits;
                const bool ok = !mine || i < kWStages || wait_bounded(wempty(s), rw.phase ^ 1u, wc);
                if (!__all_sync(kProdMask, ok)) break;
                if (mine && !(cta == 0 && i == p.fault_unit)) {   // failure-path test hook
                    mbar_arrive_expect_tx(wfull(s), F::kStageBytes);
                    F::load_w(base + s * F::kStageBytes, &tmW, p, wfull(s), cur.tile, cur.kr, pol_w, pol_s);
                    last = i;
                }
            }
            // Every copy started must land before the CTA can exit.  Only the
            // last kWStages units issued can be in flight: each older unit's
            // stage was consumed before it was filled again.  Those units sit in
            // distinct stages with nothing issued after them, so the parity of
            // each one's wait is unambiguous.
            const int newest = __reduce_max_sync(kProdMask, last);
            for (int i = last; i >= 0 && i > newest - kWStages; i -= kProdLanes)
                if (!(cta == 0 && i == p.fault_unit)) drain_wait(wfull(i % kWStages), (i / kWStages) & 1, p.timeout_ns);
        }
    } else if (warp == kWarpXProd) {
        // ------------------------------------------------------------ X producer
        // kProdLanes lanes in step, as for the weights.
        if (lane < kProdLanes) {
            if (lane == 0) prefetch_tmap(&tmX);
            // X may be the output of the preceding grid on the stream
            grid_dependency_wait();
            const uint64_t pol_x = policy_evict_last();
            int last = -1;
            Cursor cur(u0 + lane, p.KB);
            Ring<kXStages> rx(lane);
            for (int i0 = 0; i0 < nunits; i0 += kProdLanes, cur.step(kProdLanes, p.KB), rx.step(kProdLanes)) {
                const int i = i0 + lane;
                const int s = rx.slot;
                const bool mine = i < nunits;
                const bool ok = !mine || i < kXStages || wait_bounded(xempty(s), rx.phase ^ 1u, wc);
                if (!__all_sync(kProdMask, ok)) break;
                if (mine) {
                    const uint32_t st = base + L::kXOff + s * L::kXSlot;
                    mbar_arrive_expect_tx(xfull(s), L::kXSlot);
                    tma_load_2d(st, &tmX, xfull(s), cur.kr * 128, 0, pol_x);
                    tma_load_2d(st + L::kXBox, &tmX, xfull(s), cur.kr * 128 + 64, 0, pol_x);
                    last = i;
                }
            }
            // the last kXStages units issued, as for the weights
            const int newest = __reduce_max_sync(kProdMask, last);
            for (int i = last; i >= 0 && i > newest - kXStages; i -= kProdLanes)
                drain_wait(xfull(i % kXStages), (i / kXStages) & 1, p.timeout_ns);
        }
    } else if (warp == 1 || warp == kWarpMma2) {
        // ------------------------------------------------------------ MMA issuers
        // Issuer j takes units i with i % 2 == j and accumulates them into its
        // own accumulator of the piece's buffer b = piece % 2 (two issuers never
        // write one accumulator).  The whole warp runs the loop and its waits;
        // one elected lane issues the MMAs and the commits: X slot free and A
        // buffer free after every unit, accumulator complete after the
        // issuer's last unit of the piece.
        //
        // Before its first unit of piece p >= 2 an issuer waits for the fold to
        // have drained piece p - 2 (the same buffer).  Only the first and the
        // last piece of a CTA's range can be a single unit (every other piece
        // is a whole tile of KB >= 2 units, or every piece is a single unit and
        // each issuer keeps to one buffer), so an issuer that skipped piece
        // p - 2 did so for p - 2 = 0 and the parity wait is unambiguous.
        {
            const bool elected = elect_one();
            const int j = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc = idesc_f16(NMMA, F::kBf16);
            const uint64_t desc0 = smem_desc_sw128(base + L::kXOff);
            const int first_tile = static_cast<int>(u0 / p.KB);
            int last = -1;
            int last_a = 0;
            uint32_t last_aph = 0;
            int piece = -1;
            Ring<kXStages> rx(j);
            Ring<kNA> ra(j);
            Cursor cur(u0 + j, p.KB);
            for (int i = j; i < nunits; i += kIssuers, rx.step(kIssuers), ra.step(kIssuers), cur.step(kIssuers, p.KB)) {
                const int s = rx.slot;
                const int a = ra.slot;
                const int pc = cur.tile - first_tile;
                const int b = pc & 1;
                const bool fresh = pc != piece;   // the issuer's first unit of this piece
                if (fresh) {
                    piece = pc;
                    if (pc >= 2 && !warp_wait(dempty(b), static_cast<uint32_t>(((pc >> 1) - 1) & 1), wc)) break;
                }
                if (!warp_wait(xfull(s), rx.phase, wc)) break;
                if (!warp_wait(afull(a), ra.phase, wc)) break;
                tc_fence_after();
                // the issuer's last unit of the piece: its next unit is past the
                // range or in the next tile
                const bool closes = i + kIssuers >= nunits || cur.kb + kIssuers >= p.KB;
                // the descriptor's start-address field counts 16-byte units
                const uint64_t xd = desc0 + static_cast<uint64_t>((s * L::kXSlot) >> 4);
                const uint32_t dt = tmem + kDCol0 + (2 * b + j) * NMMA;
                const uint32_t at = tmem + a * 64;
                if (elected) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_ts_f16(dt, at + k * 8, xd + (((k >> 2) * L::kXBox + (k & 3) * 32) >> 4), idesc,
                                   (k > 0 || !fresh) ? 1u : 0u);
                    tc_commit(xempty(s));
                    tc_commit(afree(a));
                    if (closes) tc_commit(dfull(b, j));
                }
                __syncwarp();
                last = i;
                last_a = a;
                last_aph = ra.phase;
            }
            if (last >= 0 && elected) drain_wait(afree(last_a), last_aph, p.timeout_ns);
        }
    } else if (warp < kWarpDeq0) {
        // ------------------------------------------------------------ fold / epilogue
        // One pass per piece: wait for the accumulators of the issuers that
        // had units in it, add them, release the buffer, store or reduce.
        const int q = warp & 3;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const int first_tile = static_cast<int>(u0 / p.KB);
        const int split_info = split_info_lane(p, u0, u1, lane);
        // Y and the workspace may still be in use by the preceding grid
        grid_dependency_wait();
        uint32_t done[2][2] = {{0u, 0u}, {0u, 0u}};   // completions seen per accumulator
        auto load_acc = [&](int b, int j, uint32_t (&v)[NMMA]) {
            const uint32_t col = tl + kDCol0 + (2 * b + j) * NMMA;
            uint32_t (&v0)[16] = *reinterpret_cast<uint32_t (*)[16]>(&v[0]);
            tmem_ld_x16(col, v0);
            if constexpr (NMMA == 32) {
                uint32_t (&v1)[16] = *reinterpret_cast<uint32_t (*)[16]>(&v[16]);
                tmem_ld_x16(col + 16, v1);
            }
        };
        int ps = 0;
        int kb0 = static_cast<int>(u0 % p.KB);
        bool deferred = false;   // the first tile's reduction waits for the end of the range
        for (int pc = 0; ps < nunits; ++pc) {
            const int tile = first_tile + pc;
            const int b = pc & 1;
            int pe = ps + (p.KB - kb0) - 1;   // last unit of the piece
            if (pe > nunits - 1) pe = nunits - 1;
            const int kb_end = kb0 + (pe - ps);
            const bool two = pe > ps;
            const int j0 = ps & 1;
            if (!warp_wait(dfull(b, j0), done[b][j0] & 1u, wc)) break;
            ++done[b][j0];
            if (two) {
                if (!warp_wait(dfull(b, j0 ^ 1), done[b][j0 ^ 1] & 1u, wc)) break;
                ++done[b][j0 ^ 1];
            }
            tc_fence_after();
            uint32_t v[NMMA], w[NMMA];
            load_acc(b, j0, v);
            if (two) load_acc(b, j0 ^ 1, w);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty(b));
            float outer[NMMA];
#pragma unroll
            for (int m = 0; m < NMMA; ++m)
                outer[m] = two ? __fadd_rn(__uint_as_float(v[m]), __uint_as_float(w[m])) : __uint_as_float(v[m]);
            // after the CTA's last unit the X ring is idle: the reduction may use it
            const bool last = pe == nunits - 1;
            if (end_piece<NMMA, F>(p, outer, tile, kb_end, u0 + pe, u0, first_tile, split_info, q, lane,
                                   last ? gbase + L::kXOff : nullptr))
                deferred = true;
            if (last && deferred) finish_tile<NMMA, F>(p, first_tile, 0, split_info, q, lane, gbase + L::kXOff);
            ps = pe + 1;
            kb0 = 0;
        }
    } else {
        // ------------------------------------------------------------ dequant
        const int q = warp & 3;
        const int grp = (warp - kWarpDeq0) >> 2;   // takes units i with i % kDeqGroups == grp
        const int row = q * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
        typename F::Deq dq(p, u0, grp, kDeqGroups, nunits, row);
        // Rings of the unit being converted (weight stage, A buffer); the
        // group's units are kDeqGroups apart.
        Ring<kWStages> rw(grp);
        Ring<kNA> ra(grp);
        // unit i, whose scale sits in queue slot `slot`; false when a wait gave up
        auto unit = [&](int i, int slot) -> bool {
            const int a = ra.slot;
            const uint32_t aph = ra.phase;
            const int sw = rw.slot;
            const uint32_t wph = rw.phase;
            ra.step(kDeqGroups);
            rw.step(kDeqGroups);
            dq.prepare(p, i, nunits, row, slot);
            if (!warp_wait(wfull(sw), wph, wc)) return false;
            dq.load(gbase + sw * F::kStageBytes, row);
            // unit i - kNA (this group's) is done with its A buffer once its MMAs are
            if (i >= kNA && !warp_wait(afree(a), aph ^ 1u, wc)) return false;
            __syncwarp();
            tc_fence_after();
#pragma unroll
            for (int qtr = 0; qtr < 4; ++qtr) {
                uint32_t o[16];
                dq.convert(qtr, o);
                tmem_st_x16(tl + a * 64 + qtr * 16, o);
            }
            // Unit i's weight stage is refilled as soon as it is released, so the
            // release must not be performed before every lane's shared-memory
            // loads of it have returned.  It comes after the TMEM stores of the
            // converted weights, which need those loads: both the stores and the
            // arrive are ordered memory operations (neither the compiler nor the
            // in-order issue can put the arrive first), and a store cannot issue
            // before the registers it reads are written.
            __syncwarp();
            if (lane == 0) mbar_arrive(wempty(sw));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(a));
            return true;
        };
        // unrolled so that every scale-queue slot index is a constant
        constexpr int kU = F::Deq::kUnroll;
        bool ok = true;
        for (int i0 = grp; i0 < nunits && ok; i0 += kDeqGroups * kU) {
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                const int i = i0 + kDeqGroups * j;
                if (i < nunits && ok) ok = unit(i, j);
            }
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

template <int NMMA, class F>
cudaError_t launch(const Params& prm, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                   bool overlap, cudaStream_t st) {
    using L = Layout<NMMA, F::kStageBytes>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(qgemm_kernel<NMMA, F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s.G));
    cfg.blockDim = dim3(Roles<NMMA>::kThreads);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, qgemm_kernel<NMMA, F>, tmW, tmX, prm);
}

// Common parameter block for a schedule and workspace.
inline Params base_params(const Schedule& s, void* Y, int64_t ldy, int M, int N, int K, void* ws,
                          const LaunchCtl& c) {
    Params p{};
    p.nseg = 1;
    p.seg[0].tile0 = 0;
    p.seg[0].n = N;
    p.seg[0].S = nullptr;
    p.seg[0].Y = Y;
    p.seg[0].ldy = ldy;
    p.M = M;
    p.N = N;
    p.K = K;
    p.KB = s.KU;
    p.U = s.U;
    p.G = s.G;
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.part = reinterpret_cast<float*>(w);
    p.cnt = w ? reinterpret_cast<uint32_t*>(w + workspace_partial_bytes(s)) : nullptr;
    p.timeout_ns = c.timeout_ns;
    p.fault_unit = c.fault_unit;
    p.status = c.status;
    return p;
}

}  // namespace gemm
}  // namespace qg
