// Internal interface between the C ABI (qg_api.cu) and the kernel translation
// units.  Not installed; not part of the public header.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/qgemm.h"

namespace qg {

// Work decomposition shared by both GEMM kernels.  The output is cut into
// T tiles of 128 weight rows; each tile's K range into KU units.  The
// T * KU units, tile-major, are split evenly over G CTAs (CTA c owns units
// [c*U/G, (c+1)*U/G)).  A tile whose units are spread over several CTAs is
// finished by the last of them to arrive (split-K / stream-K).
struct Schedule {
    int T = 0;        // tiles
    int KU = 0;       // units per tile
    long long U = 0;  // T * KU
    int G = 0;        // CTAs
    int nmma = 16;    // MMA N (16 or 32)
    int max_ctas = 0; // CTAs the device holds at once (one per SM): bounds G
};

// Workspace layout for a schedule that splits tiles: split-K partial sums
// (scratch; two slots per CTA), sized for the largest grid and MMA width the
// device runs, so that the arrival counters behind them sit at the same
// offset for every shape and never overlap another shape's partial sums;
// then 4 arrival counters per tile, which are zero between calls.
size_t workspace_partial_bytes(const Schedule& s);   // = offset of the counters
size_t workspace_bytes(const Schedule& s);           // 0 when no tile is split

// Offset and size of the arrival counters of a call (0, 0 when it needs no
// workspace), for callers that must clear them.
void workspace_counters(int kind, int M, int N, int K, size_t* offset, size_t* bytes);

// One FP8 weight matrix of a call and its output (a call holds 1 to
// kMaxFp8Segs of them sharing X; see qgemm_fp8_block_multi).
constexpr int kMaxFp8Segs = 4;
struct Fp8Seg {
    const uint8_t* W;
    const float* S;
    void* Y;
    int64_t ldy;
    int N;
};

struct Fp8Args {
    const void* X;
    int64_t ldx;
    int nseg;
    Fp8Seg seg[kMaxFp8Segs];
    int64_t lds;      // ceil(K/128): the row pitch of every segment's scales
    int M, K;
    void* ws;
};

// The weight tensor map of each segment (128 x 128 E4M3 boxes).
struct Fp8Maps {
    CUtensorMap m[kMaxFp8Segs];
};

struct Lut3Args {
    const void* X;
    int64_t ldx;
    const void* Wq;
    const void* qmap;
    const void* scales;
    int64_t ldsc;
    void* Y;
    int64_t ldy;
    int M, N, K;
    void* ws;
};

struct Bf16Args {
    const void* X;
    int64_t ldx;
    const void* W;
    void* Y;
    int64_t ldy;
    int M, N, K;
    void* ws;
};

struct LaunchCtl {
    uint64_t timeout_ns;
    int fault_unit;
    uint32_t* status;    // device status word
    int num_sms;
    bool overlap;        // launch with programmatic stream serialization
};

cudaError_t launch_fp8(const Fp8Args& a, const Schedule& s, const Fp8Maps& maps, const LaunchCtl& c,
                       cudaStream_t st);
// tmS: the scale-matrix tensor map ([N, K/128] FP16, boxes of 128 rows x 8
// groups), or null to have the kernel load scales from global memory.
cudaError_t launch_lut3(const Lut3Args& a, const Schedule& s, const CUtensorMap& tmX, const CUtensorMap* tmS,
                        const LaunchCtl& c, cudaStream_t st);

// tmW: the weight map ([N, K] BF16, boxes of 64 K x 128 rows); tmX: the
// activation map ([M, K] BF16, boxes of 64 K x MMA-N rows).
cudaError_t launch_bf16(const Bf16Args& a, const Schedule& s, const CUtensorMap& tmW, const CUtensorMap& tmX,
                        const LaunchCtl& c, cudaStream_t st);
cudaError_t launch_split_probe(const void* X, int64_t blocks, void* hi, void* lo, int* exponent, cudaStream_t st);
cudaError_t launch_dequant_lut3(const void* Wq, const void* qmap, const void* scales, void* D,
                                int N, int K, cudaStream_t st);
cudaError_t launch_zero_rows(void* Y, int64_t ldy, int M, int N, cudaStream_t st);

uint32_t* device_status_ptr();

// True when calls launch with programmatic stream serialization
// (qg_set_weight_prefetch_overlap).
bool overlap_enabled();

inline bool aligned_16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Argument checks shared by the FP8 entry points (qgemm_fp8_block, the host
// and no-alloc variants): QG_OK or the status qgemm_fp8_block returns.
qg_status check_fp8_args(const void* X, int64_t ldx, const void* W, const void* W_scale, const void* Y, int64_t ldy,
                         int M, int N, int K);

// Zero the arrival counters of the no-alloc entry point's scratch array on
// the current device (if that entry point has used it there), on `st`, and
// wait for it.  Called after a timeout is reported.
cudaError_t noalloc_clear_counters(cudaStream_t st);

}  // namespace qg
