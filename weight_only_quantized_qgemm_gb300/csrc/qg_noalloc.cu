// qgemm_fp8_block_noalloc: the W8A16 FP8 block-scaled GEMM for callers that
// cannot allocate device memory.  The split-K scratch that qgemm_fp8_block
// takes from the caller lives here instead, in a fixed file-scope device
// array that every GPU loading the library holds until the process exits.
#include <mutex>

#include "../../include/qgemm.h"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

struct ScratchSlot {
    std::once_flag once;
    void* ptr = nullptr;
    cudaError_t err = cudaSuccess;
};
ScratchSlot g_scratch[kMaxDevices];

// Device address of the scratch array on the current device.  In host code
// the array's name only stands for the symbol, so the address is asked from
// the runtime once per device, with that device current.
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    ScratchSlot* s = &g_scratch[dev];
    std::call_once(s->once, [s]() {
        s->err = cudaGetSymbolAddress(&s->ptr, g_noalloc_scratch);
        if (s->err != cudaSuccess) s->ptr = nullptr;
    });
    return s->ptr;
}

}  // namespace
}  // namespace qg

extern "C" qg_status qgemm_fp8_block_noalloc(const void* X, int64_t ldx, const uint8_t* W, const float* W_scale,
                                             void* Y, int64_t ldy, int M, int N, int K, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return QG_OK;
    const size_t need = qg_workspace_bytes(QG_KIND_FP8_BLOCK, M, N, K);
    if (need > qg::kNoAllocScratchBytes) return QG_ERR_WORKSPACE;
    void* scratch = qg::scratch_on_current_device();
    if (!scratch) return QG_ERR_CUDA;
    // The array keeps whatever the previous call left (a call that timed out
    // leaves its arrival counters set); the counters must start at zero, so
    // this call's are cleared first.  The partial sums need no clearing.
    size_t cnt_off = 0, cnt_bytes = 0;
    qg::workspace_counters(QG_KIND_FP8_BLOCK, M, N, K, &cnt_off, &cnt_bytes);
    if (cnt_bytes > 0 &&
        cudaMemsetAsync(static_cast<unsigned char*>(scratch) + cnt_off, 0, cnt_bytes, stream) != cudaSuccess)
        return QG_ERR_CUDA;
    return qgemm_fp8_block(X, ldx, W, W_scale, Y, ldy, M, N, K, scratch, qg::kNoAllocScratchBytes, stream);
}
