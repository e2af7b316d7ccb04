// W8A16 FP8 block-scaled decode GEMM for sm_103a.
//
//   Y[m, n] = bf16( sum_kb  s[n/128, kb] * ( sum_{k in kb} x[m,k] * e4m3(W[n,k]) ) )
//
// The two-level fold ("atlas" m16_tc module page, section NUMERICS): each
// 128-wide K block is reduced on the tensor core into its own FP32
// accumulator, then multiplied by that block's FP32 scale once and added to an
// FP32 outer accumulator held in registers.
//
// The weights are never converted.  A 128 x 128 E4M3 tile goes from HBM to
// shared memory by TMA (128-byte swizzle, the tensor core's K-major layout)
// and is the A operand of tcgen05.mma kind::f8f6f4 as it is.  The activations
// are the ones turned into E4M3: for each (row m, K block) a power of two 2^e
// brings max |x| into [128, 256), and every scaled x splits into two E4M3
// values, x * 2^e = hi + lo / 16, exact for every element within 2^13 of the
// row's block maximum (below that the error is at most 2^-14 * 2^-e, under
// 2^-21 of the block's largest |x|; see split_e4m3x2).  The hi and lo planes
// are the MMA's B rows 0..NX-1 and NX..2NX-1 (swap-AB: the 128 weight rows
// are the MMA's M side, the activation rows its narrow N side), so one MMA
// pass of N = 2 NX gives both partial sums; every product is exact in the
// tensor core and accumulates in FP32.  The fold then forms
//   inner[m] = (hi_sum[m] + lo_sum[m] / 16) * 2^-e[m]
// and adds inner[m] * s to the outer accumulator: the same two-level fold,
// with the block sum taken in a different order.
//
// One persistent CTA per SM, 480 threads (15 warps):
//   warp 0       weight producer: one 16 KB TMA tile per unit (evict-first)
//                into a ring of 10 (NX = 16) / 8 (NX = 32) stages.
//   warps 1, 2   MMA issuers, alternate units: 4 tcgen05.mma kind::f8f6f4
//                (M = 128, N = 2 NX, K = 32) from one lane, then commits
//                that free the unit's weight stage and X planes and mark its
//                accumulator ready once the MMAs complete.
//   warps 3-6    fold / epilogue, one per TMEM lane quadrant (warp % 4).
//   warps 7-14   X split: four groups of 2 warps taking every fourth unit, 32
//                (64 for 32 rows) elements of a row per thread.  Each
//                thread copies its own share of a unit's BF16 X slice two of
//                its group's units ahead (cp.async through the load/store
//                path: a TMA copy would queue behind the weight tiles already
//                in flight and arrive microseconds later), converts the
//                current unit from registers, writes the hi/lo E4M3 planes in
//                the swizzled K-major layout and s * 2^-e per row beside them
//                (s = the unit's block scale), then takes the row maxima and
//                exponents of its group's next unit.
// A unit is 128 weight rows x one 128-wide K block.  The schedule (tiles of
// 128 rows, split-K pieces, last-arriver reduction) is the shared one of
// qg_gemm.cuh.
#include "qg_gemm.cuh"

namespace qg {
namespace {

using gemm::Cursor;
using gemm::Params;

constexpr int kWarpMma0 = 1;      // warps 1, 2
constexpr int kIssuers = 2;
constexpr int kWarpFold0 = 3;     // warps 3..6: TMEM lane quadrant warp % 4
constexpr int kFoldWarps = 4;
constexpr int kWarpConv0 = 7;     // then the split warps

// X split: four groups of two warps, taking units i with i % 4 == g; a
// thread owns kEpt elements of one row (32 at up to 16 rows, 64 at 32).
template <int NX>
struct Split {
    static constexpr int kEpt = NX == 16 ? 32 : 64;   // X elements per split thread and unit
    static constexpr int kLpr = 128 / kEpt;           // split lanes per row
    static constexpr int kWarps = NX * kLpr / 32;     // per group: 2
    static constexpr int kGroups = 4;
    static constexpr int kThreads = 32 * (kWarpConv0 + kGroups * kWarps);
};

template <int NX>
struct Fp8Layout {
    static constexpr int kN = 2 * NX;            // MMA N: hi plane, then lo plane
    static constexpr int kWBytes = 128 * 128;    // one E4M3 unit
    static constexpr int kXbSlot = NX * 256;     // BF16 X slice, [16-byte chunk j][split thread of the group]
    static constexpr int kX8Slot = kN * 128;     // both planes, 128-byte rows
    // per group: two BF16 X slots, so that a unit's copy is issued one of the
    // group's units before its scan (the slot is refilled as soon as the scan
    // has read it into registers)
    static constexpr int kXbStages = 2;
    // X plane slots: a slot is refilled once the MMAs that read it complete, so
    // the ring has to cover the split latency plus the MMA latency
    static constexpr int kX8Stages = NX == 16 ? 8 : 4;
    static constexpr int kNA = NX == 16 ? 8 : 4; // TMEM accumulators of kN columns
    static constexpr int kTmemCols = kNA * kN;
    // Row factors s * 2^-e of a unit live in their own ring, kFacStages deep: the
    // split group writes unit i's factors only after the MMAs of unit
    // i - kX8Stages completed, which were issued after the fold released unit
    // i - kX8Stages - kNA's accumulator, having read its factors; so the fold is
    // done with every unit before i - kX8Stages - kNA >= i - kFacStages.
    static constexpr int kFacStages = NX == 16 ? 16 : 8;
    static constexpr int kFacBytes = kFacStages * NX * 4;
    static constexpr int kMaxWStages = 16;
    static constexpr int kFixed = Split<NX>::kGroups * kXbStages * kXbSlot + kX8Stages * kX8Slot + kFacBytes +
                                  8 * (2 * kMaxWStages + 2 * kX8Stages + 2 * kNA) + 64 + 1024;
    static constexpr int kWFit = (232448 - kFixed) / kWBytes;
    // even: every use of a weight stage (and of an X plane slot and an
    // accumulator) then falls to the same MMA issuer, so each issuer waits on
    // the phases of a barrier in order
    static constexpr int kWStages = (kWFit < kMaxWStages ? kWFit : kMaxWStages) & ~1;
    static constexpr int kXbOff = kWStages * kWBytes;
    static constexpr int kX8Off = kXbOff + Split<NX>::kGroups * kXbStages * kXbSlot;
    static constexpr int kFacOff = kX8Off + kX8Stages * kX8Slot;
    static constexpr int kBarOff = kFacOff + kFacBytes;
    static constexpr int kNumBars = 2 * kWStages + 2 * kX8Stages + 2 * kNA;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 64 + 1024;   // + alignment slack
    static_assert(kX8Off % 1024 == 0 && kX8Slot % 1024 == 0, "keep the 1024-byte swizzle alignment");
    static_assert(kWStages >= 8 && kWStages % kIssuers == 0, "weight ring");
    // the same for the X plane slots and the accumulators, and for the split
    // groups, which take every kGroups-th unit
    static_assert(kX8Stages % kIssuers == 0 && kNA % kIssuers == 0, "ring ownership");
    static_assert(kX8Stages % Split<NX>::kGroups == 0, "ring ownership");
    static_assert(kTmemCols == 256, "TMEM allocation");
    static_assert(kFacStages >= kX8Stages + kNA, "factor ring");
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(kFacOff - kXbOff >= 4 * gemm::scratch_quadrant<NX>(), "reduction scratch in the X slots");
};

struct Bf16Store {
    __device__ static void store(void* Y, int64_t idx, float v) {
        static_cast<__nv_bfloat16*>(Y)[idx] = __float2bfloat16_rn(v);
    }
};

static_assert(gemm::kMaxSegs == kMaxFp8Segs, "segment tables");

// Index of the segment holding `tile` (constant-index selects).
__device__ __forceinline__ int seg_index(const Params& p, int tile) {
    int r = 0;
#pragma unroll
    for (int j = 1; j < gemm::kMaxSegs; ++j)
        if (j < p.nseg && tile >= p.seg[j].tile0) r = j;
    return r;
}

template <int NX>
__global__ void __launch_bounds__(Split<NX>::kThreads, 1)
    fp8_kernel(const __grid_constant__ Fp8Maps tm, const Params p) {
    using L = Fp8Layout<NX>;
    constexpr int kN = L::kN;
    constexpr int kWStages = L::kWStages;
    constexpr int kX8Stages = L::kX8Stages;
    constexpr int kNA = L::kNA;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + L::kBarOff;
    auto wfull = [&](int s) { return bar0 + 8u * s; };
    auto wempty = [&](int s) { return bar0 + 8u * (kWStages + s); };
    constexpr int kBarX8 = 2 * kWStages;
    auto x8full = [&](int s) { return bar0 + 8u * (kBarX8 + s); };
    auto x8empty = [&](int s) { return bar0 + 8u * (kBarX8 + kX8Stages + s); };
    constexpr int kBarD = kBarX8 + 2 * kX8Stages;
    auto dfull = [&](int a) { return bar0 + 8u * (kBarD + a); };
    auto dempty = [&](int a) { return bar0 + 8u * (kBarD + kNA + a); };
    float* facs = reinterpret_cast<float*>(gbase + L::kFacOff);   // [kFacStages][NX]: s * 2^-e
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
            mbar_init(wempty(s), 1);            // commit: the unit's MMAs are complete
        }
        for (int s = 0; s < kX8Stages; ++s) {
            mbar_init(x8full(s), Split<NX>::kWarps);
            mbar_init(x8empty(s), 1);           // commit: the unit's MMAs are complete
        }
        for (int a = 0; a < kNA; ++a) {
            mbar_init(dfull(a), 1);
            mbar_init(dempty(a), kFoldWarps);
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
    // The next grid on the stream may be scheduled now; its CTAs start as ours
    // exit, and only its weight stream runs before it waits for this grid.
    grid_dependents_launch();

    if (warp == 0) {
        // ------------------------------------------------------------ weight producer
        if (lane == 0) {
            for (int j = 0; j < p.nseg; ++j) prefetch_tmap(&tm.m[j]);
            const uint64_t pol_w = policy_evict_first();
            int issued = 0;
            Cursor cur(u0, p.KB);
            for (int i = 0; i < nunits; ++i, cur.step(p.KB)) {
                const int s = i % kWStages;
                if (i >= kWStages && !wait_bounded(wempty(s), ((i / kWStages) - 1) & 1, wc)) break;
                if (cta == 0 && i == p.fault_unit) continue;   // failure-path test hook
                // the unit's segment: its own weight map, rows counted from its first tile
                const int sj = seg_index(p, cur.tile);
                const int row0 = (cur.tile - gemm::seg_of(p, cur.tile).tile0) * 128;
                mbar_arrive_expect_tx(wfull(s), L::kWBytes);
                tma_load_2d(base + s * L::kWBytes, &tm.m[sj], wfull(s), cur.kr * 128, row0, pol_w);
                issued = i + 1;
            }
            // Every copy this thread started must land before the CTA can exit.
            for (int i = issued - kWStages < 0 ? 0 : issued - kWStages; i < issued; ++i) {
                if (cta == 0 && i == p.fault_unit) continue;
                gemm::drain_wait(wfull(i % kWStages), (i / kWStages) & 1, p.timeout_ns);
            }
        }
    } else if (warp >= kWarpConv0) {
        // ------------------------------------------------------------ X split
        // Group g takes units i with i % kG == g.  Thread (r, c) of a group:
        // row r, elements [kEpt c, kEpt c + kEpt) of the unit's 128-wide slice;
        // the kLpr lanes of a row are adjacent lanes.  Each thread copies and reads
        // back only its own chunks, so the staging ring needs no barrier: a
        // thread's wait on its own copy groups is enough.
        constexpr int kEpt = Split<NX>::kEpt;
        constexpr int kLpr = Split<NX>::kLpr;
        constexpr int CH_IN = kEpt / 8;        // 16-byte BF16 chunks read
        constexpr int CH_OUT = kEpt / 16;      // 16-byte E4M3 chunks written per plane
        constexpr int kGT = 32 * Split<NX>::kWarps;   // threads per group
        constexpr int kG = Split<NX>::kGroups;
        const int g = (warp - kWarpConv0) / Split<NX>::kWarps;
        const int ct = ((warp - kWarpConv0) % Split<NX>::kWarps) * 32 + lane;
        const int r = ct / kLpr;
        const int c = ct % kLpr;
        const uint32_t sw = static_cast<uint32_t>(r & 7);
        const int xring = L::kXbOff + g * L::kXbStages * L::kXbSlot + ct * 16;   // byte offset
        const __nv_bfloat16* xrow = static_cast<const __nv_bfloat16*>(p.X) + static_cast<int64_t>(r) * p.ldx;
        // X may be the output of the preceding grid on the stream
        grid_dependency_wait();
        Cursor pf(u0 + g, p.KB);   // the group's unit copied next
        Cursor sq(u0 + g, p.KB);   // the group's unit scanned next
        auto prefetch = [&](int i) {
            if (i < nunits) {
                const uint32_t slot = base + static_cast<uint32_t>(xring + ((i / kG) % L::kXbStages) * L::kXbSlot);
                const int k0 = pf.kr * 128 + c * kEpt;   // K % 8 == 0: a chunk is in or out
                const bool rok = r < p.M;
#pragma unroll
                for (int j = 0; j < CH_IN; ++j) {
                    const bool ok = rok && k0 + j * 8 < p.K;
                    cp_async_16(slot + j * (kGT * 16), ok ? static_cast<const void*>(xrow + k0 + j * 8) : p.X,
                                ok ? 16u : 0u);
                }
                pf.step(kG, p.KB);
            }
            cp_async_commit();   // one group per unit, empty past the end
        };
        // Unit i's slice into registers, its row maximum and exponent: 2^e
        // with max |x| * 2^e in [128, 256), e = 134 - (BF16 biased exponent of
        // the maximum), capped so that 2^e and 2^-e stay normal; and the unit's
        // block scale.
        auto scan = [&](int i, uint4 (&xin)[CH_IN], uint32_t& pw2, int& e, float& sblk) {
            const gemm::Seg sg = gemm::seg_of(p, sq.tile);
            sblk = __ldg(sg.S + static_cast<int64_t>(sq.tile - sg.tile0) * p.lds + sq.kr);
            sq.step(kG, p.KB);
            const uint8_t* xs = gbase + xring + ((i / kG) % L::kXbStages) * L::kXbSlot;
#pragma unroll
            for (int j = 0; j < CH_IN; ++j) xin[j] = *reinterpret_cast<const uint4*>(xs + j * (kGT * 16));
            // max(|a|, |b|) per half, sign bits set aside below
            uint32_t m2 = bf16x2_absmax(xin[0].x, xin[0].y);
            m2 = bf16x2_absmax(m2, bf16x2_absmax(xin[0].z, xin[0].w));
#pragma unroll
            for (int j = 1; j < CH_IN; ++j) {
                m2 = bf16x2_absmax(m2, bf16x2_absmax(xin[j].x, xin[j].y));
                m2 = bf16x2_absmax(m2, bf16x2_absmax(xin[j].z, xin[j].w));
            }
            m2 &= 0x7FFF7FFFu;
            uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
            for (int o = 1; o < kLpr; o <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            e = split_exponent(mx);
            pw2 = bf16x2_pow2(e);
        };
        // The group's units i = g, g + kG, ...: unit i is converted from
        // registers while the copies of units i + kG and i + 2 kG are in flight;
        // then unit i + kG, copied one iteration earlier, is scanned.
        prefetch(g);
        prefetch(g + kG);
        uint4 xc[CH_IN];
        uint32_t pc = 0;
        int ec = 0;
        float scur = 0.0f;
        if (g < nunits) {
            cp_async_wait<1>();
            scan(g, xc, pc, ec, scur);
        }
        for (int i = g; i < nunits; i += kG) {
            const int s8 = i % kX8Stages;
            // into the slot unit i was read from
            prefetch(i + 2 * kG);
            if (i >= kX8Stages && !gemm::warp_wait(x8empty(s8), ((i / kX8Stages) - 1) & 1, wc)) break;
            uint8_t* xo = gbase + L::kX8Off + s8 * L::kX8Slot;
#pragma unroll
            for (int h = 0; h < CH_OUT; ++h) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    // elements 16h + 4 q4 .. +3 of this thread: BF16 words 8h + 2 q4, +1
                    const int wi = 8 * h + 2 * q4;
                    const uint4& src = xc[wi >> 2];
                    const uint32_t w0 = (wi & 3) == 0 ? src.x : src.z;
                    const uint32_t w1 = (wi & 3) == 0 ? src.y : src.w;
                    split_e4m3x4(bf16x2_mul(w0, pc), bf16x2_mul(w1, pc), hw[q4], lw[q4]);
                }
                const uint32_t oc = static_cast<uint32_t>(c * CH_OUT + h);   // 16-element chunk (0..7)
                const int rh = r, rl = NX + r;
                *reinterpret_cast<uint4*>(xo + (rh >> 3) * 1024 + (rh & 7) * 128 + ((oc ^ sw) << 4)) =
                    make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(xo + (rl >> 3) * 1024 + (rl & 7) * 128 + ((oc ^ sw) << 4)) =
                    make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            // s * 2^-e: exact, a power-of-two multiple of the FP32 block scale
            if (c == 0)
                facs[(i % L::kFacStages) * NX + r] = __fmul_rn(scur, __uint_as_float(static_cast<uint32_t>(127 - ec) << 23));
            // the planes are read by the tensor core (async proxy)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(x8full(s8));
            if (i + kG < nunits) {
                cp_async_wait<1>();   // all but the newest copy (unit i + 2 kG) have landed
                scan(i + kG, xc, pc, ec, scur);
            }
        }
    } else if (warp >= kWarpMma0 && warp < kWarpMma0 + kIssuers) {
        // ------------------------------------------------------------ MMA issuers
        // The whole warp runs the loop and its waits; one elected lane issues.
        const bool elected = elect_one();
        const int first = warp - kWarpMma0;
        constexpr uint32_t idesc = idesc_f8_e4m3(kN);
        const uint64_t dw0 = smem_desc_sw128(base);
        const uint64_t dx0 = smem_desc_sw128(base + L::kX8Off);
        int last = -1;
        for (int i = first; i < nunits; i += kIssuers) {
            const int sw = i % kWStages;
            const int s8 = i % kX8Stages;
            const int a = i % kNA;
            if (!gemm::warp_wait(wfull(sw), (i / kWStages) & 1, wc)) break;
            if (!gemm::warp_wait(x8full(s8), (i / kX8Stages) & 1, wc)) break;
            if (i >= kNA && !gemm::warp_wait(dempty(a), ((i / kNA) - 1) & 1, wc)) break;
            tc_fence_after();
            // descriptor start addresses count 16-byte units; one MMA takes 32 K
            // bytes of both operands
            const uint64_t ad = dw0 + static_cast<uint64_t>((sw * L::kWBytes) >> 4);
            const uint64_t bd = dx0 + static_cast<uint64_t>((s8 * L::kX8Slot) >> 4);
            const uint32_t dt = tmem + a * kN;
            if (elected) {
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_ss_f8(dt, ad + 2 * j, bd + 2 * j, idesc, j > 0 ? 1u : 0u);
                tc_commit(wempty(sw));
                tc_commit(x8empty(s8));
                tc_commit(dfull(a));
            }
            __syncwarp();
            last = i;
        }
        if (last >= 0 && elected) gemm::drain_wait(dfull(last % kNA), (last / kNA) & 1, p.timeout_ns);
    } else if (warp >= kWarpFold0 && warp < kWarpFold0 + kFoldWarps) {
        // ------------------------------------------------------------ fold / epilogue
        const int q = warp & 3;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const int first_tile = static_cast<int>(u0 / p.KB);
        const int split_info = gemm::split_info_lane(p, u0, u1, lane);
        // Y and the workspace may still be in use by the preceding grid
        grid_dependency_wait();
        bool deferred = false;   // the first tile's reduction waits for the end of the range
        float outer[NX];
#pragma unroll
        for (int m = 0; m < NX; ++m) outer[m] = 0.0f;
        Cursor cur(u0, p.KB);
        for (int i = 0; i < nunits; ++i, cur.step(p.KB)) {
            const int a = i % kNA;
            if (!gemm::warp_wait(dfull(a), (i / kNA) & 1, wc)) break;
            tc_fence_after();
            // hi columns [0, NX), lo columns [NX, 2 NX); 16 rows of X at a time,
            // with the unit's row factors s * 2^-e (valid until the fold reaches
            // unit i + kFacStages - kX8Stages - kNA > i, see kFacStages):
            //   outer += (hi + lo / 16) * s * 2^-e
            const float4* f4 = reinterpret_cast<const float4*>(facs + (i % L::kFacStages) * NX);
            auto fold16 = [&](int m0, const uint32_t (&vh)[16], const uint32_t (&vl)[16]) {
#pragma unroll
                for (int m4 = 0; m4 < 4; ++m4) {
                    const float4 f = f4[m0 / 4 + m4];
                    const float fm[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int jj = 4 * m4 + j;
                        const float t = __fmaf_rn(__uint_as_float(vl[jj]), 0.0625f, __uint_as_float(vh[jj]));
                        outer[m0 + jj] = __fmaf_rn(t, fm[j], outer[m0 + jj]);
                    }
                }
            };
            uint32_t vh[16], vl[16];
            tmem_ld_x16(tl + a * kN, vh);
            tmem_ld_x16(tl + a * kN + NX, vl);
            tmem_wait_ld();
            if constexpr (NX == 32) {
                fold16(0, vh, vl);
                tmem_ld_x16(tl + a * kN + 16, vh);
                tmem_ld_x16(tl + a * kN + NX + 16, vl);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty(a));
            fold16(NX - 16, vh, vl);

            if (cur.kb != p.KB - 1 && i != nunits - 1) continue;
            // after the CTA's last unit the X staging and plane slots are idle:
            // the reduction may use them
            const bool last = i == nunits - 1;
            if (gemm::end_piece<NX, Bf16Store>(p, outer, cur.tile, cur.kb, u0 + i, u0, first_tile, split_info, q,
                                               lane, last ? gbase + L::kXbOff : nullptr))
                deferred = true;
            if (last && deferred)
                gemm::finish_tile<NX, Bf16Store>(p, first_tile, 0, split_info, q, lane, gbase + L::kXbOff);
#pragma unroll
            for (int m = 0; m < NX; ++m) outer[m] = 0.0f;
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

template <int NX>
cudaError_t launch_nx(const Params& prm, const Schedule& s, const Fp8Maps& maps, bool overlap, cudaStream_t st) {
    using L = Fp8Layout<NX>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(fp8_kernel<NX>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s.G));
    cfg.blockDim = dim3(Split<NX>::kThreads);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, fp8_kernel<NX>, maps, prm);
}

}  // namespace

cudaError_t launch_fp8(const Fp8Args& a, const Schedule& s, const Fp8Maps& maps, const LaunchCtl& c,
                       cudaStream_t st) {
    gemm::Params p = gemm::base_params(s, a.seg[0].Y, a.seg[0].ldy, a.M, s.T * 128, a.K, a.ws, c);
    p.nseg = a.nseg;
    int tile0 = 0;
    for (int j = 0; j < a.nseg; ++j) {
        p.seg[j].tile0 = tile0;
        p.seg[j].n = a.seg[j].N;
        p.seg[j].S = a.seg[j].S;
        p.seg[j].Y = a.seg[j].Y;
        p.seg[j].ldy = a.seg[j].ldy;
        tile0 += (a.seg[j].N + 127) / 128;
    }
    p.S = a.seg[0].S;
    p.lds = a.lds;
    p.X = a.X;
    p.ldx = a.ldx;
    if (s.nmma == 16) return launch_nx<16>(p, s, maps, c.overlap, st);
    return launch_nx<32>(p, s, maps, c.overlap, st);
}

}  // namespace qg
