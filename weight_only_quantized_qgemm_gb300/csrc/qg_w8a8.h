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
};

// tmW: the weight map ([N, K] E4M3, 128 x 128 boxes); tmX: the activation
// map ([M, K] E4M3, boxes of 128 K x 32 rows).  The schedule's tiles are
// ceil(N/128) x ceil(M/32), weight-tile-major.
cudaError_t launch_w8a8(const W8a8Args& a, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                        const LaunchCtl& c, cudaStream_t st);
cudaError_t launch_quantize_act(const void* X, int64_t ldx, void* Xq, int64_t ldxq, float* Sx, int64_t ldsx, int M,
                                int K, const LaunchCtl& c, cudaStream_t st);

}  // namespace qg
