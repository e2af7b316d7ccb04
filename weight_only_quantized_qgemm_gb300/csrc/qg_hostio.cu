// qgemm_fp8_block_host: the W8A16 FP8 block-scaled GEMM with X and Y in
// pinned host memory.  A staging kernel pulls X over the host link into a
// caller-owned device buffer, and the GEMM's epilogue stores Y straight into
// host memory.  The only copy engine is the SM's load/store path: no copy
// call sits between two kernels, so the GEMM keeps its programmatic
// launch overlap (weight prefetch during the staging kernel) and no
// device-to-host copy follows it.
#include "../../include/qgemm.h"
#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr int kStageThreads = 128;
constexpr int kStagePer = 4;   // 16-byte chunks per thread

// Copy `rows` rows of `row16` 16-byte chunks from src (row stride src_ld16
// chunks) to dst (row stride dst_ld16).  Both the loads and the stores come
// after the dependency wait: the preceding grid on the stream may write the
// source (a chained caller passes one call's Y_host as the next call's
// X_host) and may still read the destination.  The next grid is released at
// once, so the GEMM behind this kernel starts streaming its weights while X
// crosses the host link.
__global__ void __launch_bounds__(kStageThreads) stage_rows_kernel(const uint4* src, int64_t src_ld16, uint4* dst,
                                                                   int64_t dst_ld16, int rows, int64_t row16) {
    grid_dependents_launch();
    grid_dependency_wait();
    const int64_t total = static_cast<int64_t>(rows) * row16;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kStageThreads;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kStageThreads + threadIdx.x;
    uint4 v[kStagePer];
#pragma unroll
    for (int j = 0; j < kStagePer; ++j) {
        const int64_t i = i0 + j * stride;
        if (i < total) {
            const int64_t r = i / row16;
            v[j] = src[r * src_ld16 + (i - r * row16)];
        }
    }
#pragma unroll
    for (int j = 0; j < kStagePer; ++j) {
        const int64_t i = i0 + j * stride;
        if (i < total) {
            const int64_t r = i / row16;
            dst[r * dst_ld16 + (i - r * row16)] = v[j];
        }
    }
}

// Device address of a buffer the GPU can reach (pinned host, device or
// managed memory); null for pageable host memory and unknown pointers.
const void* device_view(const void* p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();   // the failed query is recorded as the last error; clear it
        return nullptr;
    }
    if (attr.type == cudaMemoryTypeUnregistered) return nullptr;
    return attr.devicePointer;   // the address of p itself, not of its allocation
}

}  // namespace
}  // namespace qg

extern "C" qg_status qgemm_fp8_block_host(const void* X_host, int64_t ldx, const uint8_t* W, const float* W_scale,
                                          void* Y_host, int64_t ldy, int M, int N, int K, void* X_stage,
                                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    // the GEMM's own checks, with the host buffers standing for X and Y
    qg_status v = qg::check_fp8_args(X_host, ldx, W, W_scale, Y_host, ldy, M, N, K);
    if (v != QG_OK || M == 0 || N == 0) return v;
    if (!X_stage) return QG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(X_stage) & 15u) != 0) return QG_ERR_MISALIGNED;
    const void* Xd = qg::device_view(X_host);
    void* Yd = const_cast<void*>(qg::device_view(Y_host));
    if (!Xd || !Yd) return QG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Xd) & 15u) != 0 || (reinterpret_cast<uintptr_t>(Yd) & 1u) != 0)
        return QG_ERR_MISALIGNED;
    // Validate the workspace too before the staging kernel is enqueued, so
    // that a refused call enqueues nothing.
    if (K > 0) {
        const size_t need = qg_workspace_bytes(QG_KIND_FP8_BLOCK, M, N, K);
        if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
            return QG_ERR_WORKSPACE;
        const int64_t row16 = static_cast<int64_t>(K) / 8;
        const int64_t total = static_cast<int64_t>(M) * row16;
        const int64_t per_cta = static_cast<int64_t>(qg::kStageThreads) * qg::kStagePer;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>((total + per_cta - 1) / per_cta));
        cfg.blockDim = dim3(qg::kStageThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        if (qg::overlap_enabled()) {
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        if (cudaLaunchKernelEx(&cfg, qg::stage_rows_kernel, static_cast<const uint4*>(Xd), ldx / 8,
                               static_cast<uint4*>(X_stage), row16, M, row16) != cudaSuccess)
            return QG_ERR_CUDA;
    }
    return qgemm_fp8_block(X_stage, K, W, W_scale, Yd, ldy, M, N, K, workspace, workspace_bytes, stream);
}
