/*
 * qgemm.h -- C ABI of libqgemm: weight-only quantized decode GEMMs on GB300
 * (sm_103a).
 *
 *   Y[M, N] = X[M, K] . dequant(W)[N, K]^T,   1 <= M <= 32
 *
 * Two weight formats:
 *
 *  1. W8A16 FP8 block-scaled ("atlas" m16_tc module page, sections WHY and
 *     NUMERICS; "arc" PR 215, weight_block_size [128, 128]).  W holds OCP
 *     E4M3FN codes, one FP32 scale per [128 x 128] block of W; X and Y are
 *     BF16.  Every 128-wide K block is reduced in FP32, multiplied by its
 *     block scale once, and added to an FP32 outer accumulator (the two-level
 *     fold); Y is the BF16 round-to-nearest-even of the outer sum.  The
 *     reduction order inside a block and across K ranges is the tensor core's
 *     and the split-K schedule's, so results match a strict-K-order reference
 *     within 2 BF16 ULP per element, or within an absolute floor for outputs
 *     that cancel to near zero (same page, red-cell section).
 *
 *  2. W3A16 learned LUT (FLUTE "optimized_w3" page, sections Core
 *     contributions and Results).  W holds 3-bit codes packed one per nibble
 *     (layout below); an 8-entry FP16 map qmap and one FP16 scale per
 *     (row, 128-wide K group) dequantise a code as fp16_rne(qmap[c] * scale);
 *     X and Y are FP16, the sum is FP32.
 *
 * Conventions shared by all GEMM entry points
 *  - All matrix pointers are device pointers; the caller owns every buffer.
 *    The library allocates nothing per call.
 *  - Row-major: X row m starts at X + m*ldx elements, Y row m at Y + m*ldy.
 *    Callers flatten [B, S, K] activations to [B*S, K] first.
 *  - Calls are asynchronous on `stream` (NULL = legacy default stream); Y is
 *    overwritten, never accumulated into.
 *  - Arguments are validated before anything is launched: a non-OK status
 *    means nothing was enqueued.  M == 0 or N == 0 is a no-op returning
 *    QG_OK; K == 0 writes zeros to Y.
 *  - Kernel waits are bounded (default 1 s, see qg_set_wait_timeout_ns).  A
 *    wait that runs out makes the kernel record QG_ERR_TIMEOUT in a device
 *    status word, release its resources and return; read it with
 *    qg_last_device_status().  After such an error the workspace contents are
 *    undefined and must be zero-filled again before reuse.
 *  - NaN codes (E4M3 0x7F / 0xFF) and non-finite X produce unspecified values.
 *  - One workspace may serve one in-flight call at a time.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* the same type as cudaStream_t */

typedef enum {
    QG_OK = 0,
    QG_ERR_INVALID_ARG = 1,       /* null pointer, negative size, ld < row length */
    QG_ERR_UNSUPPORTED_SHAPE = 2, /* M > 32, K % 16 (FP8) or K % 128 (LUT3) != 0 */
    QG_ERR_MISALIGNED = 3,        /* a pointer or row stride breaks the 16-byte rule */
    QG_ERR_CUDA = 4,              /* a CUDA runtime call or kernel launch failed */
    QG_ERR_TIMEOUT = 5,           /* a bounded in-kernel wait ran out */
    QG_ERR_WORKSPACE = 6          /* workspace missing or smaller than qg_workspace_bytes */
} qg_status;

enum { QG_KIND_FP8_BLOCK = 0, QG_KIND_LUT3 = 1 };

/*
 * Bytes of device workspace a call of the given kind and shape needs on the
 * current device (0 if none).  The workspace holds split-K partial sums
 * (scratch, sized for the device's largest grid) followed by per-tile arrival
 * counters (the last 16 * ceil(N/128) bytes, rounded up to 256).  It must be
 * zero-filled once before its first use; every successful call leaves its
 * counters at zero again, so one workspace serves later calls of any shape
 * without clearing.
 */
size_t qg_workspace_bytes(int kind, int M, int N, int K);

/*
 * W8A16 FP8 block-scaled GEMM.
 *   X        device, BF16 [M, ldx], 16-byte aligned, ldx >= K, ldx % 8 == 0
 *   W        device, E4M3 codes [N, K] row-major (row stride K bytes),
 *            16-byte aligned
 *   W_scale  device, FP32 [ceil(N/128), ceil(K/128)] row-major; entry
 *            (i, j) scales W[128i : 128i+128, 128j : 128j+128]
 *   Y        device, BF16 [M, ldy], ldy >= N
 *   M, N, K  1 <= M <= 32, N >= 1, K % 16 == 0 (ragged N and K tails are
 *            handled; the last block row/column may be partial)
 *   workspace, workspace_bytes  device buffer of at least
 *            qg_workspace_bytes(QG_KIND_FP8_BLOCK, M, N, K) bytes (may be NULL
 *            when that is 0)
 */
qg_status qgemm_fp8_block(const void *X, int64_t ldx,
                          const uint8_t *W, const float *W_scale,
                          void *Y, int64_t ldy,
                          int M, int N, int K,
                          void *workspace, size_t workspace_bytes,
                          struct CUstream_st *stream);

/*
 * The W8A16 FP8 block-scaled GEMM for callers that cannot allocate device
 * memory -- for example a plug-in running inside a host framework that owns
 * all device memory and hands it no allocator, or code that must not allocate
 * while it serves requests.  (The paper has no counterpart of this entry
 * point; it is an addition of this library.)
 *
 * Arguments and results are those of qgemm_fp8_block without the workspace:
 * the split-K scratch is a fixed 8 MiB array inside the library, which every
 * GPU that loads the library holds until the process exits.  The call
 * allocates nothing.
 *  - A shape whose scratch need (qg_workspace_bytes) exceeds 8 MiB returns
 *    QG_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on a device looks up the array's device address (one
 *    runtime query, with that device current); make that first call before
 *    any stream capture.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's contents; each call clears the part it uses on `stream` first.
 *    Calls whose execution overlaps on the GPU (different streams, or
 *    concurrent host threads) race on the array and give wrong results:
 *    serialise them.
 */
qg_status qgemm_fp8_block_noalloc(const void *X, int64_t ldx,
                                  const uint8_t *W, const float *W_scale,
                                  void *Y, int64_t ldy,
                                  int M, int N, int K,
                                  struct CUstream_st *stream);

/*
 * The W8A16 FP8 block-scaled GEMM with X and Y in host memory -- for a
 * caller whose activations arrive from, and whose results go back to, the
 * host every call.  (The paper has no counterpart of this entry point; it is
 * an addition of this library.)
 *
 * Arguments and results are those of qgemm_fp8_block, except:
 *   X_host   pinned (page-locked) host memory, BF16 [M, ldx], 16-byte
 *            aligned, ldx >= K, ldx % 8 == 0; device or managed memory also
 *            works
 *   Y_host   pinned host memory, BF16 [M, ldy], ldy >= N; device or managed
 *            memory also works
 *   X_stage  device, at least M * K * 2 bytes, 16-byte aligned: scratch the
 *            call copies X into (row stride K); owned by the caller and
 *            serving one in-flight call at a time, like the workspace
 * A staging kernel reads X_host over the host link into X_stage, and the
 * GEMM stores Y directly into Y_host; no copy call is enqueued.  Pageable
 * (unregistered) host memory, or a pointer the runtime does not know,
 * returns QG_ERR_INVALID_ARG before anything is enqueued.  Y_host is
 * complete once `stream` has been synchronised; the call is asynchronous
 * like the others, so neither host buffer may be touched before that.
 */
qg_status qgemm_fp8_block_host(const void *X_host, int64_t ldx,
                               const uint8_t *W, const float *W_scale,
                               void *Y_host, int64_t ldy,
                               int M, int N, int K,
                               void *X_stage,
                               void *workspace, size_t workspace_bytes,
                               struct CUstream_st *stream);

/*
 * W3A16 learned-LUT GEMM.
 *   X        device, FP16 [M, ldx], 16-byte aligned, ldx >= K, ldx % 8 == 0
 *   Wq       device, pack_lut3() output for an [N, K] code matrix
 *            (qg_lut3_packed_bytes(N, K) bytes), 16-byte aligned
 *   qmap     device, 8 FP16 values (the learned map), 16-byte aligned
 *   scales   device, FP16 [N, K/128] row-major, one per (row, 128-wide K group)
 *   Y        device, FP16 [M, ldy], ldy >= N
 *   M, N, K  1 <= M <= 32, N >= 1, K % 128 == 0
 *   workspace as for qgemm_fp8_block, with kind QG_KIND_LUT3.
 */
qg_status qgemm_lut3(const void *X, int64_t ldx,
                     const void *Wq, const void *qmap, const void *scales,
                     void *Y, int64_t ldy,
                     int M, int N, int K,
                     void *workspace, size_t workspace_bytes,
                     struct CUstream_st *stream);

/*
 * Packed size, in bytes, of an [N, K] 3-bit code matrix:
 * ceil(N/128) * ceil(K/256) * 16384.
 */
size_t qg_lut3_packed_bytes(int N, int K);

/*
 * Offline packer (host memory, synchronous, deterministic).  codes is an
 * [N, K] row-major byte matrix with values 0..7; packed receives
 * qg_lut3_packed_bytes(N, K) bytes.  Codes above 7 give QG_ERR_INVALID_ARG.
 *
 * Layout ("nibble + fragment" order; FLUTE optimized_w3 page, Core
 * contributions item 2, re-derived for this library's kernel): the matrix is
 * cut into tiles of 128 rows x 256 codes, stored tile-row-major (tile
 * (tn, tk) is block number tn * ceil(K/256) + tk, 16384 bytes each, so one
 * K-step of one 128-row tile is one contiguous bulk copy).  Inside a tile, the
 * 16-byte chunk holding codes k = 32q .. 32q+31 of row r sits at byte offset
 * (q * 128 + r) * 16, so the 32 lanes of a warp that own 32 consecutive rows
 * read 512 contiguous bytes.  A chunk is four little-endian 32-bit words;
 * word w holds the codes of k = 32q + 8w + i in nibble i (bits 4i .. 4i+3),
 * top bit zero, so a word is directly the byte-permute selector of the
 * dequantiser.  Rows >= N and columns >= K are filled with code 0.
 */
qg_status pack_lut3(const uint8_t *codes, void *packed, int N, int K);

/* Inverse of pack_lut3 (host, test aid): writes the [N, K] codes back. */
qg_status unpack_lut3(const void *packed, uint8_t *codes, int N, int K);

/*
 * Dequantise n E4M3 codes to BF16 on the device with exactly the conversion
 * the FP8 GEMM uses (no scale applied).  codes and out_bf16 are device
 * pointers; n >= 0.  Exposed so that the conversion can be checked code by
 * code.
 */
qg_status qg_dequant_e4m3_bf16(const uint8_t *codes, void *out_bf16, int64_t n,
                               struct CUstream_st *stream);

/*
 * Dequantise a packed LUT3 matrix to FP16 D[N, K] (row-major, device) with
 * exactly the conversion the LUT3 GEMM uses: D[n, k] =
 * fp16_rne(qmap[code] * scales[n, k/128]).
 */
qg_status qg_dequant_lut3(const void *Wq, const void *qmap, const void *scales,
                          void *D, int N, int K, struct CUstream_st *stream);

/*
 * Synchronises `stream`, returns the device status word recorded by kernels
 * since the last call (QG_OK if none failed), and clears it.  The word is per
 * process and device, shared by all streams.
 */
qg_status qg_last_device_status(struct CUstream_st *stream);

/* Upper bound, in nanoseconds, of every in-kernel wait of later launches
 * (default 1e9; values below 1000 are raised to 1000). */
void qg_set_wait_timeout_ns(uint64_t ns);

/*
 * Failure-path test hook.  With unit >= 0, the next GEMM launches have their
 * first CTA skip the weight load of its unit-th work unit, so that the wait
 * for it runs out and the kernel reports QG_ERR_TIMEOUT.  unit < 0 turns it
 * off (the default).
 */
void qg_set_fault_injection(int unit);

/*
 * Overlap of consecutive GEMMs on a stream (off by default).  When enabled,
 * the GEMM kernels are launched with programmatic stream serialization: a
 * GEMM may start, and begin streaming its W and scales, while the kernel
 * before it on the stream is still finishing; it waits for that kernel before
 * it reads X or touches Y and the workspace.  Enable it only when W and the
 * scales are not written by the work immediately preceding the GEMM on the
 * same stream (true for model weights in decode).  Applies to later launches.
 */
void qg_set_weight_prefetch_overlap(int enable);

/* Short English description of a status code (static storage). */
const char *qg_status_string(qg_status status);

/* Library version, e.g. "0.1.0". */
const char *qg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H */
