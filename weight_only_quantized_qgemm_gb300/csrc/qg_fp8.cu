// W8A16 FP8 block-scaled format for the decode GEMM pipeline (qg_gemm.cuh).
//
//   Y[m, n] = bf16( sum_kb  s[n/128, kb] * ( sum_{k in kb} x[m,k] * e4m3(W[n,k]) ) )
//
// The two-level fold ("atlas" m16_tc module page, section NUMERICS): each
// 128-wide K block is reduced on the tensor core into its own FP32
// accumulator, then multiplied by that block's FP32 scale once and added to an
// FP32 outer accumulator held in registers.  Weights stream as 128 x 128 E4M3
// tiles through a 2-D TMA map with the 128-byte swizzle (one row per lane is
// then read conflict-free) and become BF16 exactly in registers; the scale is
// never applied to individual weights.
#include "qg_gemm.cuh"

namespace qg {
namespace {

struct Fp8Fmt {
    static constexpr int kWBytes = 128 * 128;
    static constexpr bool kBf16 = true;
    static constexpr bool kUsesTensorMapW = true;

    __device__ static void load_w(uint32_t dst, const CUtensorMap* tmW, const gemm::Params&, uint32_t bar,
                                  int tile, int kb, uint64_t pol) {
        tma_load_2d(dst, tmW, bar, kb * 128, tile * 128, pol);
    }
    static constexpr bool kHasFoldScale = true;
    __device__ static const float* fold_scale_ptr(const gemm::Params& p, int tile, int kb) {
        return p.S + static_cast<int64_t>(tile) * p.lds + kb;
    }
    __device__ static float fold(float outer, float inner, float sc) {
        return __fadd_rn(outer, __fmul_rn(inner, sc));
    }
    __device__ static void store(void* Y, int64_t idx, float v) {
        static_cast<__nv_bfloat16*>(Y)[idx] = __float2bfloat16_rn(v);
    }

    // One thread dequantises one weight row (128 codes) of a unit.  Two
    // register slots: the pipeline loads the group's next unit into one while
    // it converts the current unit from the other.
    struct Deq {
        static constexpr int kUnroll = 2;
        uint4 c[2][8];
        __device__ Deq(const gemm::Params&, long long, int, int, int) {}
        __device__ void prepare(const gemm::Params&, int, int, int, int) {}
        __device__ void load(int slot, const uint8_t* stage, int row) {
            const uint8_t* wrow = stage + row * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                c[slot][j] = *reinterpret_cast<const uint4*>(wrow + ((j ^ (row & 7)) << 4));
        }
        // columns 16*qtr .. 16*qtr+15 of the row's A fragment (K 32*qtr .. 32*qtr+31)
        __device__ void convert(int slot, int qtr, uint32_t (&o)[16]) const {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint4 w = c[slot][2 * qtr + j];
                e4m3x4_to_bf16(w.x, o[8 * j + 0], o[8 * j + 1]);
                e4m3x4_to_bf16(w.y, o[8 * j + 2], o[8 * j + 3]);
                e4m3x4_to_bf16(w.z, o[8 * j + 4], o[8 * j + 5]);
                e4m3x4_to_bf16(w.w, o[8 * j + 6], o[8 * j + 7]);
            }
        }
    };
};

}  // namespace

cudaError_t launch_fp8(const Fp8Args& a, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                       const LaunchCtl& c, cudaStream_t st) {
    gemm::Params p = gemm::base_params(s, a.Y, a.ldy, a.M, a.N, a.K, a.ws, c);
    p.S = a.S;
    p.lds = a.lds;
    if (s.nmma == 16) return gemm::launch<16, Fp8Fmt>(p, s, tmW, tmX, c.overlap, st);
    return gemm::launch<32, Fp8Fmt>(p, s, tmW, tmX, c.overlap, st);
}

}  // namespace qg
