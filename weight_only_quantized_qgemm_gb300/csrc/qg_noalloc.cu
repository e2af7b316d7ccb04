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

// Zero-initialised when the module loads; every successful call leaves its
// arrival counters at zero again.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

struct ScratchSlot {
    std::once_flag once;
    void* ptr = nullptr;
    cudaError_t err = cudaSuccess;
};
ScratchSlot g_scratch[kMaxDevices];

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Device address of the scratch array on the current device.  In host code
// the array's name only stands for the symbol, so the address is asked from
// the runtime once per device, with that device current.
void* scratch_on_current_device() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    ScratchSlot* s = &g_scratch[dev];
    std::call_once(s->once, [s]() {
        s->err = cudaGetSymbolAddress(&s->ptr, g_noalloc_scratch);
        if (s->err != cudaSuccess) s->ptr = nullptr;
    });
    return s->ptr;
}

}  // namespace

cudaError_t noalloc_clear_counters(cudaStream_t st) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    ScratchSlot* s = &g_scratch[dev];
    // only a device on which the entry point has run can hold counters of it
    if (s->ptr == nullptr) return cudaSuccess;
    // the counters of every shape sit behind the partial sums of the largest
    // grid the device runs (see workspace_partial_bytes)
    size_t off = 0, bytes = 0;
    workspace_counters(QG_KIND_FP8_BLOCK, 1, 128 * 1024, 4096, &off, &bytes);
    if (off == 0 || off >= kNoAllocScratchBytes) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(static_cast<unsigned char*>(s->ptr) + off, 0, kNoAllocScratchBytes - off, st);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(st);
}

}  // namespace qg

extern "C" qg_status qgemm_fp8_block_noalloc(const void* X, int64_t ldx, const uint8_t* W, const float* W_scale,
                                             void* Y, int64_t ldy, int M, int N, int K, cudaStream_t stream) {
    // every argument is checked before anything is enqueued
    const qg_status v = qg::check_fp8_args(X, ldx, W, W_scale, Y, ldy, M, N, K);
    if (v != QG_OK || M == 0 || N == 0) return v;
    const size_t need = qg_workspace_bytes(QG_KIND_FP8_BLOCK, M, N, K);
    if (need > qg::kNoAllocScratchBytes) return QG_ERR_WORKSPACE;
    void* scratch = need > 0 ? qg::scratch_on_current_device() : nullptr;
    if (need > 0 && !scratch) return QG_ERR_CUDA;
    return qgemm_fp8_block(X, ldx, W, W_scale, Y, ldy, M, N, K, scratch, qg::kNoAllocScratchBytes, stream);
}
