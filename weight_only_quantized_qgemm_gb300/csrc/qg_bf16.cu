// Dense BF16 decode GEMM for sm_103a (the unquantised tier beside the FP8 one
// on the "atlas" m16_tc page, graded by the same numerics contract):
//
//   Y[m, n] = bf16( sum_k x[m, k] * w[n, k] )        (FP32 accumulation)
//
// The weights need no conversion: a 128-row x 128-K BF16 unit arrives by TMA
// (two 64-element boxes, 128-byte swizzle, the tensor core's K-major layout)
// and is the A operand of tcgen05.mma kind::f16 as it lands; X is the B
// operand (swap-AB: 128 weight rows on the MMA's M side, the M <= 32
// activation rows its narrow N side).  There is no per-block scale, so the
// MMAs of a tile piece (the units of one tile in a CTA's range) accumulate in
// TMEM and the fold warps read each piece once.
//
// One persistent CTA per SM, 256 threads:
//   warp 0      weight producer: two TMA boxes per unit (L2 evict-first)
//               into a ring of 32 KB stages.
//   warp 1      X producer: the unit's 128-wide X slice (two boxes) into a
//               ring, after the grid dependency wait.
//   warp 2      MMA issuer: 8 tcgen05.mma (M = 128, N = NX, K = 16) per unit
//               from one elected lane, into the piece's accumulator (two
//               piece buffers alternate).
//   warps 4-7   fold / epilogue, one per TMEM lane quadrant: read a piece's
//               accumulator once, store the tile or its split-K partial.
// The work split (tiles of 128 rows, units of 128 K, stream-K pieces,
// last-arriver reduction) is the shared one of qg_gemm.cuh.
#include "qg_gemm.cuh"

namespace qg {
namespace {

using gemm::Cursor;
using gemm::Params;

constexpr int kWarpWProd = 0;
constexpr int kWarpXProd = 1;
constexpr int kWarpMma = 2;
constexpr int kWarpFold0 = 4;   // warps 4..7: TMEM lane quadrant warp % 4
constexpr int kThreads = 256;

template <int NX>
struct Bf16Layout {
    static constexpr int kWBytes = 128 * 128 * 2;   // one unit of BF16 weights: two 16 KB boxes
    static constexpr int kWBox = 128 * 128;         // bytes of one 64-K box of 128 rows
    static constexpr int kXSlot = NX * 256;         // two 64-K boxes of NX rows
    static constexpr int kXBox = NX * 128;
    static constexpr int kXStages = 8;
    static constexpr int kTmemCols = 2 * NX < 32 ? 32 : 2 * NX;   // two piece accumulators
    static constexpr int kFixed = kXStages * kXSlot + 8 * (2 * 8 + 2 * kXStages + 4) + 64 + 1024;
    static constexpr int kWStages = (232448 - kFixed) / kWBytes;
    static constexpr int kXOff = kWStages * kWBytes;
    static constexpr int kBarOff = kXOff + kXStages * kXSlot;
    static constexpr int kNumBars = 2 * kWStages + 2 * kXStages + 4;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 64 + 1024;   // + alignment slack
    static_assert(kWStages >= 4 && kWStages <= 8, "weight ring");
    static_assert(kXOff % 1024 == 0 && kXSlot % 1024 == 0, "keep the 1024-byte swizzle alignment");
    // the final split-K reduction stages its pieces in the idle weight ring
    static_assert(kWStages * kWBytes >= 4 * gemm::scratch_quadrant<NX>(), "reduction scratch");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

struct Bf16Store {
    __device__ static void store(void* Y, int64_t idx, float v) {
        static_cast<__nv_bfloat16*>(Y)[idx] = __float2bfloat16_rn(v);
    }
};

template <int NX>
__global__ void __launch_bounds__(kThreads, 1)
    bf16_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const Params p) {
    using L = Bf16Layout<NX>;
    constexpr int kWStages = L::kWStages;
    constexpr int kXStages = L::kXStages;
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
    auto dfull = [&](int b) { return bar0 + 8u * (kBarD + b); };
    auto dempty = [&](int b) { return bar0 + 8u * (kBarD + 2 + b); };
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
            mbar_init(xempty(s), 1);   // commit: the unit's MMAs are complete
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(dfull(b), 1);    // commit: the piece's last MMAs are complete
            mbar_init(dempty(b), 4);   // the four fold warps
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
    // the next grid on the stream may be scheduled now (it streams its weights
    // before it waits for this one)
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
                const uint32_t dst = base + s * L::kWBytes;
                mbar_arrive_expect_tx(wfull(s), L::kWBytes);
                tma_load_2d(dst, &tmW, wfull(s), cur.kr * 128, cur.tile * 128, pol_w);
                tma_load_2d(dst + L::kWBox, &tmW, wfull(s), cur.kr * 128 + 64, cur.tile * 128, pol_w);
                issued = i + 1;
            }
            // every copy started must land before the CTA can exit
            for (int i = issued - kWStages < 0 ? 0 : issued - kWStages; i < issued; ++i) {
                if (cta == 0 && i == p.fault_unit) continue;
                gemm::drain_wait(wfull(i % kWStages), (i / kWStages) & 1, p.timeout_ns);
            }
        }
    } else if (warp == kWarpXProd) {
        // ------------------------------------------------------------ X producer
        if (lane == 0) {
            prefetch_tmap(&tmX);
            // X may be the output of the preceding grid on the stream
            grid_dependency_wait();
            const uint64_t pol_x = policy_evict_last();
            int issued = 0;
            Cursor cur(u0, p.KB);
            for (int i = 0; i < nunits; ++i, cur.step(p.KB)) {
                const int s = i % kXStages;
                if (i >= kXStages && !wait_bounded(xempty(s), ((i / kXStages) - 1) & 1, wc)) break;
                const uint32_t dst = base + L::kXOff + s * L::kXSlot;
                mbar_arrive_expect_tx(xfull(s), L::kXSlot);
                tma_load_2d(dst, &tmX, xfull(s), cur.kr * 128, 0, pol_x);
                tma_load_2d(dst + L::kXBox, &tmX, xfull(s), cur.kr * 128 + 64, 0, pol_x);
                issued = i + 1;
            }
            for (int i = issued - kXStages < 0 ? 0 : issued - kXStages; i < issued; ++i)
                gemm::drain_wait(xfull(i % kXStages), (i / kXStages) & 1, p.timeout_ns);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        // Piece p accumulates in buffer p % 2; before the first unit of piece
        // p >= 2 the issuer waits for the fold to have drained piece p - 2.
        const bool elected = elect_one();
        constexpr uint32_t idesc = idesc_f16(NX, true);
        const uint64_t dw0 = smem_desc_sw128(base);
        const uint64_t dx0 = smem_desc_sw128(base + L::kXOff);
        const int first_tile = static_cast<int>(u0 / p.KB);
        int piece = -1;
        int last = -1, last_b = 0;
        Cursor cur(u0, p.KB);
        for (int i = 0; i < nunits; ++i, cur.step(p.KB)) {
            const int sw = i % kWStages;
            const int sx = i % kXStages;
            const int pc = cur.tile - first_tile;
            const int b = pc & 1;
            const bool fresh = pc != piece;
            if (fresh) {
                piece = pc;
                if (pc >= 2 && !gemm::warp_wait(dempty(b), static_cast<uint32_t>(((pc >> 1) - 1) & 1), wc)) break;
            }
            if (!gemm::warp_wait(wfull(sw), (i / kWStages) & 1, wc)) break;
            if (!gemm::warp_wait(xfull(sx), (i / kXStages) & 1, wc)) break;
            tc_fence_after();
            const bool closes = i == nunits - 1 || cur.kb == p.KB - 1;
            // descriptor start addresses count 16-byte units; one MMA takes 16
            // K (32 bytes) of both operands
            const uint64_t ad = dw0 + static_cast<uint64_t>((sw * L::kWBytes) >> 4);
            const uint64_t bd = dx0 + static_cast<uint64_t>((sx * L::kXSlot) >> 4);
            const uint32_t dt = tmem + b * NX;
            if (elected) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t a = ad + static_cast<uint64_t>(((k >> 2) * L::kWBox + (k & 3) * 32) >> 4);
                    const uint64_t x = bd + static_cast<uint64_t>(((k >> 2) * L::kXBox + (k & 3) * 32) >> 4);
                    mma_ss_f16(dt, a, x, idesc, (k > 0 || !fresh) ? 1u : 0u);
                }
                tc_commit(wempty(sw));
                tc_commit(xempty(sx));
                if (closes) tc_commit(dfull(b));
            }
            __syncwarp();
            last = i;
            last_b = b;
        }
        (void)last_b;
        if (last >= 0 && elected) gemm::drain_wait(wempty(last % kWStages), (last / kWStages) & 1, p.timeout_ns);
    } else if (warp >= kWarpFold0) {
        // ------------------------------------------------------------ fold / epilogue
        const int q = warp & 3;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const int first_tile = static_cast<int>(u0 / p.KB);
        const int split_info = gemm::split_info_lane(p, u0, u1, lane);
        // Y and the workspace may still be in use by the preceding grid
        grid_dependency_wait();
        bool deferred = false;   // the first tile's reduction waits for the end of the range
        uint32_t done[2] = {0u, 0u};
        int ps = 0;
        int kb0 = static_cast<int>(u0 % p.KB);
        for (int pc = 0; ps < nunits; ++pc) {
            const int tile = first_tile + pc;
            const int b = pc & 1;
            int pe = ps + (p.KB - kb0) - 1;   // last unit of the piece
            if (pe > nunits - 1) pe = nunits - 1;
            const int kb_end = kb0 + (pe - ps);
            if (!gemm::warp_wait(dfull(b), done[b] & 1u, wc)) break;
            ++done[b];
            tc_fence_after();
            uint32_t v[NX];
            tmem_ld_x16(tl + b * NX, *reinterpret_cast<uint32_t (*)[16]>(&v[0]));
            if constexpr (NX == 32) tmem_ld_x16(tl + b * NX + 16, *reinterpret_cast<uint32_t (*)[16]>(&v[16]));
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty(b));
            float outer[NX];
#pragma unroll
            for (int m = 0; m < NX; ++m) outer[m] = __uint_as_float(v[m]);
            // after the CTA's last unit the weight ring is idle: the reduction may use it
            const bool last = pe == nunits - 1;
            if (gemm::end_piece<NX, Bf16Store>(p, outer, tile, kb_end, u0 + pe, u0, first_tile, split_info, q, lane,
                                               last ? gbase : nullptr))
                deferred = true;
            if (last && deferred) gemm::finish_tile<NX, Bf16Store>(p, first_tile, 0, split_info, q, lane, gbase);
            ps = pe + 1;
            kb0 = 0;
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
cudaError_t launch_nx(const Params& prm, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                      bool overlap, cudaStream_t st) {
    using L = Bf16Layout<NX>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(bf16_kernel<NX>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s.G));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, bf16_kernel<NX>, tmW, tmX, prm);
}

}  // namespace

cudaError_t launch_bf16(const Bf16Args& a, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                        const LaunchCtl& c, cudaStream_t st) {
    gemm::Params p = gemm::base_params(s, a.Y, a.ldy, a.M, a.N, a.K, a.ws, c);
    if (s.nmma == 16) return launch_nx<16>(p, s, tmW, tmX, c.overlap, st);
    return launch_nx<32>(p, s, tmW, tmX, c.overlap, st);
}

}  // namespace qg
