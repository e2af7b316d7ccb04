// Internal interface of the W8A8 kernels (qg_w8a8.cu) for the C ABI.
#pragma once

#include "qg_internal.h"

namespace qg {

// W8A8: E4M3 activations Xq [M, ldxq] with per-(128-K block, row) scales
// Sx [KB, ldsx] (ldsx >= M rounded up to 32), E4M3 weights W [N, K] with
// block scales S [ceil(N/128), ceil(K/128)], BF16 Y [M, ldy].
struct W8a8Args {
    const float* Sx;
    int64_t ldsx;
    const float* S;
    void* Y;
    int64_t ldy;
    int M, N, K;
    void* ws;
    // Y as a BF16 [M, N] tensor map (row pitch ldy * 2 bytes, boxes of 32
    // columns x 16 rows, no swizzle) when y_tma != 0, which needs Y 16-byte
    // aligned and ldy and N multiples of 8; else the kernel stores Y directly
    CUtensorMap tmY;
    int y_tma;
};

// The W8A8 kernel's activation rows per tile (its MMA N) for a batch size.
constexpr int kMaxTileRows = 128;
inline int w8a8_tile_rows(int M) { return M <= 64 ? 64 : kMaxTileRows; }

// Workspace of a W8A8 schedule (s.nmma = the tile's activation rows, s.T its
// tiles): split-K partial sums, two slots of 128 x kMaxTileRows FP32 per CTA
// (w8a8_partial_bytes, the same for every W8A8 shape), then one arrival
// counter per (tile, fold warp) (nmma / 16 per tile); 0 when no tile is split.
size_t w8a8_partial_bytes(const Schedule& s);
size_t w8a8_workspace_bytes(const Schedule& s, bool split);

// tmW: the weight map ([N, K] E4M3, 128 x 128 boxes); tmX: the activation
// map ([M, K] E4M3, boxes of 128 K x s.nmma rows).  The schedule's tiles are
// ceil(N/128) x ceil(M/s.nmma), weight-tile-major.
cudaError_t launch_w8a8(const W8a8Args& a, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                        const LaunchCtl& c, cudaStream_t st);
cudaError_t launch_quantize_act(const void* X, int64_t ldx, void* Xq, int64_t ldxq, float* Sx, int64_t ldsx, int M,
                                int K, const LaunchCtl& c, cudaStream_t st);

}  // namespace qg
