// Exactness-gated tuning of the dispatch table (FLUTE "optimized_w3" page,
// Results: candidates are checked against a reference before they are timed).
// For one shape, candidate grids run on the caller's buffers; a candidate
// whose output strays from the built-in schedule's output beyond a gate is
// discarded, the others are timed back to back with CUDA events, and the
// fastest becomes the shape's dispatch-table entry.
#include <cmath>
#include <cstring>
#include <vector>

#include "../../include/qgemm.h"
#include "qg_internal.h"
#include "qg_w8a8.h"

namespace qg {
namespace {

// BF16 or FP16 bit pattern -> float.
float half_bits_to_float(uint16_t h, bool bf16) {
    if (bf16) {
        uint32_t u = static_cast<uint32_t>(h) << 16;
        float f;
        std::memcpy(&f, &u, 4);
        return f;
    }
    const uint32_t s = (h >> 15) & 1u, e = (h >> 10) & 31u, m = h & 1023u;
    float v;
    if (e == 0) v = std::ldexp(static_cast<float>(m), -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = std::ldexp(static_cast<float>(m | 1024u), static_cast<int>(e) - 25);
    return s ? -v : v;
}

// The gate: every value finite, and the candidate within a relative
// Frobenius distance of 1e-3 and a largest deviation of 1e-2 of the
// reference's largest magnitude.  Reassociating the FP32 split-K sum moves
// results by a few units in the last place; a schedule that drops, repeats or
// misplaces a piece moves them by the size of the values themselves.
bool gate(const std::vector<uint16_t>& got, const std::vector<uint16_t>& ref, bool bf16) {
    double num = 0, den = 0, dmax = 0, rmax = 0;
    for (size_t i = 0; i < got.size(); ++i) {
        const double a = half_bits_to_float(got[i], bf16), b = half_bits_to_float(ref[i], bf16);
        if (!std::isfinite(a) || !std::isfinite(b)) return false;
        num += (a - b) * (a - b);
        den += b * b;
        dmax = std::fmax(dmax, std::fabs(a - b));
        rmax = std::fmax(rmax, std::fabs(b));
    }
    if (den == 0) return num == 0;
    return std::sqrt(num / den) <= 1e-3 && dmax <= 1e-2 * rmax;
}

// Candidate grids: one CTA per tile, 2..8 CTAs per tile, fractions of the
// SMs, and (more tiles than SMs) the largest grid over which whole tiles
// divide evenly, each at most the SM count and the number of work units.
std::vector<int> candidates(int T, long long U, int sms) {
    std::vector<int> c;
    auto add = [&](long long g) {
        if (g < 1 || g > sms || g > U) return;
        for (int x : c)
            if (x == g) return;
        c.push_back(static_cast<int>(g));
    };
    for (int k = 1; k <= 8; ++k) add(static_cast<long long>(k) * T);
    for (int e = 8; e >= 4; --e) add(static_cast<long long>(sms) * e / 8);
    if (T > sms)
        for (int d = sms; d >= 1; --d)
            if (T % d == 0) {
                add(d);
                break;
            }
    return c;
}

struct Tuner {
    int kind, M, N, K;
    int T;          // the shape's tiles
    long long U;    // its work units
    void* Y;
    void* Y_ref;
    int64_t ldy;
    size_t ws_bytes;
    int calls;
    cudaStream_t stream;
    bool bf16;

    std::vector<uint16_t> fetch(const void* buf) const {
        std::vector<uint16_t> h(static_cast<size_t>(M) * N);
        // rows of N values with row stride ldy
        if (cudaMemcpy2D(h.data(), static_cast<size_t>(N) * 2, buf, static_cast<size_t>(ldy) * 2,
                         static_cast<size_t>(N) * 2, M, cudaMemcpyDeviceToHost) != cudaSuccess)
            h.clear();
        return h;
    }

    // run(out, i): one call writing `out`, i-th of a timed sequence.
    template <class Run>
    qg_status tune(Run run, int* best_ctas, float* best_us) {
        qg_dispatch_set(kind, M, N, K, 0);
        const int builtin = qg_dispatch_get(kind, M, N, K);
        qg_status st = run(Y_ref, 0);
        if (st != QG_OK) return st;
        if (qg_last_device_status(stream) != QG_OK) return QG_ERR_CUDA;
        const std::vector<uint16_t> ref = fetch(Y_ref);
        if (ref.empty()) return QG_ERR_CUDA;
        int sms = 0, dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return QG_ERR_CUDA;
        std::vector<int> cand = candidates(T, U, sms);
        bool has_builtin = false;
        for (int g : cand) has_builtin |= g == builtin;
        if (!has_builtin) cand.push_back(builtin);
        cudaEvent_t e0, e1;
        if (cudaEventCreate(&e0) != cudaSuccess) return QG_ERR_CUDA;
        if (cudaEventCreate(&e1) != cudaSuccess) {
            cudaEventDestroy(e0);
            return QG_ERR_CUDA;
        }
        int best = builtin;
        float best_t = INFINITY;
        qg_status result = QG_OK;
        for (int g : cand) {
            if (qg_dispatch_set(kind, M, N, K, g) != QG_OK) continue;
            if (qg_workspace_bytes(kind, M, N, K) > ws_bytes) continue;   // needs more scratch than given
            if ((st = run(Y, 0)) != QG_OK) {
                result = st;
                break;
            }
            if (qg_last_device_status(stream) != QG_OK) {
                result = QG_ERR_CUDA;
                break;
            }
            const std::vector<uint16_t> got = fetch(Y);
            if (got.empty()) {
                result = QG_ERR_CUDA;
                break;
            }
            if (!gate(got, ref, bf16)) continue;
            for (int i = 0; i < 8; ++i) run(Y, i);   // warm-up
            cudaEventRecord(e0, stream);
            for (int i = 0; i < calls; ++i) run(Y, i);
            cudaEventRecord(e1, stream);
            if (cudaEventSynchronize(e1) != cudaSuccess) {
                result = QG_ERR_CUDA;
                break;
            }
            float ms = 0;
            cudaEventElapsedTime(&ms, e0, e1);
            if (qg_last_device_status(stream) != QG_OK) {
                result = QG_ERR_CUDA;
                break;
            }
            const float us = ms * 1000.0f / calls;
            if (us < best_t) {
                best_t = us;
                best = g;
            }
        }
        cudaEventDestroy(e0);
        cudaEventDestroy(e1);
        // the built-in rule stays in charge when it is the fastest
        qg_dispatch_set(kind, M, N, K, best == builtin ? 0 : best);
        if (result != QG_OK) return result;
        if (best_ctas) *best_ctas = best;
        if (best_us) *best_us = best_t;
        return QG_OK;
    }
};

// Tiles and work units of a shape (the dispatch rule's decomposition).
void shape_units(int kind, int M, int N, int K, int* T, long long* U) {
    const int tn = (N + 127) / 128;
    if (kind == QG_KIND_W8A8) {
        const int R = w8a8_tile_rows(M);
        *T = tn * ((M + R - 1) / R);
        *U = static_cast<long long>(*T) * ((K + 255) / 256);
    } else {
        *T = tn;
        *U = static_cast<long long>(tn) * ((K + 127) / 128);
    }
}

Tuner make_tuner(int kind, int M, int N, int K, void* Y, int64_t ldy, void* Y_ref, void* workspace,
                 size_t workspace_bytes, int calls, cudaStream_t stream, bool bf16) {
    Tuner t{kind, M, N, K, 0, 0, Y, Y_ref, ldy, workspace ? workspace_bytes : 0, calls, stream, bf16};
    shape_units(kind, M, N, K, &t.T, &t.U);
    return t;
}

}  // namespace
}  // namespace qg

extern "C" qg_status qg_tune_fp8(const void* X, int64_t ldx, const uint8_t* const* W_copies, int ncopies,
                                 const float* W_scale, void* Y, int64_t ldy, void* Y_ref, int M, int N, int K,
                                 void* workspace, size_t workspace_bytes, int calls, int* best_ctas, float* best_us,
                                 cudaStream_t stream) {
    if (!W_copies || ncopies < 1 || !Y_ref || calls < 1) return QG_ERR_INVALID_ARG;
    for (int i = 0; i < ncopies; ++i) {
        const qg_status v = qg::check_fp8_args(X, ldx, W_copies[i], W_scale, Y, ldy, M, N, K);
        if (v != QG_OK) return v;
    }
    if (M == 0 || N == 0 || K == 0) return QG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Y_ref) & 1u) != 0) return QG_ERR_MISALIGNED;
    qg::Tuner t = qg::make_tuner(QG_KIND_FP8_BLOCK, M, N, K, Y, ldy, Y_ref, workspace, workspace_bytes, calls, stream,
                                 true);
    auto run = [&](void* out, int i) {
        return qgemm_fp8_block(X, ldx, W_copies[i % ncopies], W_scale, out, ldy, M, N, K, workspace,
                               workspace_bytes, stream);
    };
    return t.tune(run, best_ctas, best_us);
}

extern "C" qg_status qg_tune_lut3(const void* X, int64_t ldx, const void* const* Wq_copies, int ncopies,
                                  const void* qmap, const void* scales, void* Y, int64_t ldy, void* Y_ref, int M,
                                  int N, int K, void* workspace, size_t workspace_bytes, int calls, int* best_ctas,
                                  float* best_us, cudaStream_t stream) {
    if (!Wq_copies || ncopies < 1 || !Y_ref || calls < 1) return QG_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return QG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Y_ref) & 1u) != 0) return QG_ERR_MISALIGNED;
    qg::Tuner t = qg::make_tuner(QG_KIND_LUT3, M, N, K, Y, ldy, Y_ref, workspace, workspace_bytes, calls, stream,
                                 false);
    auto run = [&](void* out, int i) {
        return qgemm_lut3(X, ldx, Wq_copies[i % ncopies], qmap, scales, out, ldy, M, N, K, workspace,
                          workspace_bytes, stream);
    };
    return t.tune(run, best_ctas, best_us);
}

extern "C" qg_status qg_tune_bf16(const void* X, int64_t ldx, const void* const* W_copies, int ncopies, void* Y,
                                  int64_t ldy, void* Y_ref, int M, int N, int K, void* workspace,
                                  size_t workspace_bytes, int calls, int* best_ctas, float* best_us,
                                  cudaStream_t stream) {
    if (!W_copies || ncopies < 1 || !Y_ref || calls < 1) return QG_ERR_INVALID_ARG;
    if (M < 1 || M > 32 || N < 1 || K < 1) return M > 32 ? QG_ERR_UNSUPPORTED_SHAPE : QG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Y_ref) & 1u) != 0) return QG_ERR_MISALIGNED;
    qg::Tuner t = qg::make_tuner(QG_KIND_BF16, M, N, K, Y, ldy, Y_ref, workspace, workspace_bytes, calls, stream,
                                 true);
    auto run = [&](void* out, int i) {
        return qgemm_bf16(X, ldx, W_copies[i % ncopies], out, ldy, M, N, K, workspace, workspace_bytes, stream);
    };
    return t.tune(run, best_ctas, best_us);
}

extern "C" qg_status qg_tune_w8a8(const uint8_t* Xq, int64_t ldxq, const float* X_scale, int64_t ldsx,
                                  const uint8_t* const* W_copies, int ncopies, const float* W_scale, void* Y,
                                  int64_t ldy, void* Y_ref, int M, int N, int K, void* workspace,
                                  size_t workspace_bytes, int calls, int* best_ctas, float* best_us,
                                  cudaStream_t stream) {
    if (!W_copies || ncopies < 1 || !Y_ref || calls < 1) return QG_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return QG_ERR_INVALID_ARG;
    if (M > 65536) return QG_ERR_UNSUPPORTED_SHAPE;
    if ((reinterpret_cast<uintptr_t>(Y_ref) & 1u) != 0) return QG_ERR_MISALIGNED;
    qg::Tuner t = qg::make_tuner(QG_KIND_W8A8, M, N, K, Y, ldy, Y_ref, workspace, workspace_bytes, calls, stream,
                                 true);
    auto run = [&](void* out, int i) {
        return qgemm_w8a8_block(Xq, ldxq, X_scale, ldsx, W_copies[i % ncopies], W_scale, out, ldy, M, N, K,
                                workspace, workspace_bytes, stream);
    };
    return t.tune(run, best_ctas, best_us);
}
