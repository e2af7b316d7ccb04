// W3A16 learned-LUT format for the decode GEMM pipeline (qg_gemm.cuh);
// FLUTE "optimized_w3" page, sections Core contributions and Results,
// re-designed for tcgen05.
//
//   d[n, k] = fp16_rne(qmap[code[n, k]] * scale[n, k/128])
//   Y[m, n] = fp16( sum_k x[m, k] * d[n, k] )          (FP32 accumulation)
//
// Weights arrive pre-packed (pack_lut3): one contiguous 8 KB block per
// (128-row tile, 128-wide K group) unit, one code per nibble, 16-byte chunks
// ordered so that the 32 lanes owning 32 consecutive rows read 512 contiguous
// bytes.  The dequantiser keeps, per (row, group), the scaled 8-entry table as
// two FP16 byte planes in registers and looks codes up with byte permutes
// whose selector is the code word itself (8 values = 1 shift + 8 permutes; no
// shared-memory table).  The scale is applied once per table entry, which
// gives the same FP16 values as scaling every weight.  There is no per-block
// fold scale: the MMAs of a tile piece accumulate in TMEM (FP32) and the fold
// warps add the two MMA issuers' accumulators once per piece.
#include <type_traits>

#include "qg_gemm.cuh"

namespace qg {
namespace {

// One thread dequantises one weight row (128 codes, one scale group) of a
// unit: the scaled 8-entry table, then the codes by byte permutes.  The codes
// of one unit and its table are held at a time: loading the next unit's codes
// early would need a second set of registers, and at this kernel's register
// budget that set spills.
struct DeqCore {
    uint4 qm;
    uint4 c[4];
    LutPlanes t;
    __device__ explicit DeqCore(const gemm::Params& p) : qm(__ldg(p.qmap)) {}
    __device__ void load_codes(const uint8_t* stage, int row, uint32_t sc) {
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = *reinterpret_cast<const uint4*>(stage + ((j * 128 + row) << 4));
        const uint32_t sc2 = sc | (sc << 16);
        t = lut_planes(f16x2_mul(qm.x, sc2), f16x2_mul(qm.y, sc2), f16x2_mul(qm.z, sc2), f16x2_mul(qm.w, sc2));
    }
    // columns 16*qtr .. 16*qtr+15 of the row's A fragment (K 32*qtr .. 32*qtr+31)
    __device__ void convert(int qtr, uint32_t (&o)[16]) const {
        const uint4 cw = c[qtr];
        const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t r4[4];
            lut3x8_to_f16(w4[w], t, r4);
#pragma unroll
            for (int e = 0; e < 4; ++e) o[4 * w + e] = r4[e];
        }
    }
};

// Scales from global memory: the thread's scale for a unit is fetched kUnroll
// of its units in advance into a fixed slot of scq (the caller unrolls its
// loop by kUnroll), so the load latency stays off the dequant.
struct DeqLoadedScales : DeqCore {
    static constexpr int kUnroll = 2;
    uint32_t sc = 0;
    uint32_t scq[kUnroll];
    gemm::Cursor ahead;   // the unit whose scale is fetched next
    int G;                // dequant groups: this thread's units are G apart
    __device__ static uint32_t scale_of(const gemm::Params& p, const gemm::Cursor& c, int row) {
        const int n = c.tile * 128 + row;
        return n < p.N ? static_cast<uint32_t>(__ldg(p.lut_scales + static_cast<int64_t>(n) * p.ld_lut_scales + c.kr))
                       : 0u;
    }
    // this thread handles units grp, grp + G, grp + 2 G, ... (G dequant
    // groups); slot j of scq holds the scale of its j-th unit modulo kUnroll
    __device__ DeqLoadedScales(const gemm::Params& p, long long u0, int grp, int groups, int nunits, int row)
        : DeqCore(p), ahead(u0 + grp, p.KB), G(groups) {
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) {
            const int i = grp + G * j;
            scq[j] = i < nunits ? scale_of(p, ahead, row) : 0u;
            ahead.step(G, p.KB);
        }
    }
    // called for each of the group's units in order, before load(); slot is
    // the unit's place in the scale queue (a compile-time constant)
    __device__ void prepare(const gemm::Params& p, int i, int nunits, int row, int slot) {
        sc = scq[slot];
        const int inext = i + G * kUnroll;
        scq[slot] = inext < nunits ? scale_of(p, ahead, row) : 0u;
        ahead.step(G, p.KB);
    }
    __device__ void load(const uint8_t* stage, int row) { load_codes(stage, row, sc); }
};

// Scales copied into the weight stage by the producer (a [128 rows x 8 K
// groups] box holding the unit's group): the thread reads its row's entry.
struct DeqStagedScales : DeqCore {
    static constexpr int kUnroll = 2;
    static constexpr int kScaleOff = 8192;
    gemm::Cursor now;   // the unit prepared next
    int kr = 0;         // K group of the unit being converted
    int G;
    __device__ DeqStagedScales(const gemm::Params& p, long long u0, int grp, int groups, int, int)
        : DeqCore(p), now(u0 + grp, p.KB), G(groups) {}
    __device__ void prepare(const gemm::Params& p, int, int, int, int) {
        kr = now.kr;
        now.step(G, p.KB);
    }
    __device__ void load(const uint8_t* stage, int row) {
        const uint32_t sc = *reinterpret_cast<const uint16_t*>(stage + kScaleOff + row * 16 + (kr & 7) * 2);
        load_codes(stage, row, sc);
    }
};

// kStagedScales: the producer also copies each unit's scales with a tensor
// map over the [N, K/128] scale matrix (needs a row pitch that is a multiple
// of 16 bytes, i.e. K % 1024 == 0, and a 16-byte aligned base); otherwise the
// dequant warps load their scales from global memory.
template <bool kStagedScales>
struct Lut3Fmt {
    static constexpr int kWBytes = 8192;                 // the codes of one unit
    static constexpr int kScaleBoxBytes = 128 * 8 * 2;   // [128 rows x 8 groups] FP16
    static constexpr int kStageBytes = kWBytes + (kStagedScales ? kScaleBoxBytes : 0);
    static constexpr bool kBf16 = false;
    static constexpr bool kUsesTensorMapW = kStagedScales;   // the first tensor map holds the scales
    static_assert(DeqStagedScales::kScaleOff == kWBytes, "scale box placement");

    // One unit's copies into its stage: the codes, one contiguous bulk copy,
    // and with staged scales the box of rows [128 tile, 128 tile + 128) and
    // K groups [kb & ~7, (kb & ~7) + 8) (its first coordinate a multiple of 8
    // groups, 16 bytes; rows past N and groups past K/128 read as zero).
    __device__ static void load_w(uint32_t dst, const CUtensorMap* tmS, const gemm::Params& p, uint32_t bar, int tile,
                                  int kb, uint64_t pol, uint64_t pol_s) {
        const size_t off = (static_cast<size_t>(tile) * p.KT + (kb >> 1)) * 16384 + (kb & 1) * kWBytes;
        bulk_load(dst, p.Wq + off, kWBytes, bar, pol);
        if constexpr (kStagedScales) tma_load_2d(dst + kWBytes, tmS, bar, kb & ~7, tile * 128, pol_s);
    }
    __device__ static void store(void* Y, int64_t idx, float v) {
        static_cast<__half*>(Y)[idx] = __float2half_rn(v);
    }
    using Deq = std::conditional_t<kStagedScales, DeqStagedScales, DeqLoadedScales>;
};

}  // namespace

cudaError_t launch_lut3(const Lut3Args& a, const Schedule& s, const CUtensorMap& tmX, const CUtensorMap* tmS,
                        const LaunchCtl& c, cudaStream_t st) {
    gemm::Params p = gemm::base_params(s, a.Y, a.ldy, a.M, a.N, a.K, a.ws, c);
    p.Wq = static_cast<const uint8_t*>(a.Wq);
    p.qmap = static_cast<const uint4*>(a.qmap);
    p.lut_scales = static_cast<const uint16_t*>(a.scales);
    p.ld_lut_scales = a.ldsc;
    p.KT = (a.K + 255) / 256;
    if (tmS) {
        if (s.nmma == 16) return gemm::launch<16, Lut3Fmt<true>>(p, s, *tmS, tmX, c.overlap, st);
        return gemm::launch<32, Lut3Fmt<true>>(p, s, *tmS, tmX, c.overlap, st);
    }
    CUtensorMap unused{};
    if (s.nmma == 16) return gemm::launch<16, Lut3Fmt<false>>(p, s, unused, tmX, c.overlap, st);
    return gemm::launch<32, Lut3Fmt<false>>(p, s, unused, tmX, c.overlap, st);
}

}  // namespace qg
