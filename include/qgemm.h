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
 *  3. Unquantised BF16 (the BF16 lm_head tier graded by the same numerics
 *     contract on the "atlas" m16_tc page): W, X and Y are BF16, the sum is
 *     FP32, Y is its BF16 round-to-nearest-even.
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
    QG_ERR_UNSUPPORTED_SHAPE = 2, /* M > 32 (65536 for W8A8), K % 16 (FP8, W8A8), K % 128 (LUT3)
                                     or K % 8 (BF16) != 0 */
    QG_ERR_MISALIGNED = 3,        /* a pointer or row stride breaks the 16-byte rule */
    QG_ERR_CUDA = 4,              /* a CUDA runtime call or kernel launch failed */
    QG_ERR_TIMEOUT = 5,           /* a bounded in-kernel wait ran out */
    QG_ERR_WORKSPACE = 6          /* workspace missing or smaller than qg_workspace_bytes */
} qg_status;

enum { QG_KIND_FP8_BLOCK = 0, QG_KIND_LUT3 = 1, QG_KIND_BF16 = 2, QG_KIND_W8A8 = 3 };

/*
 * Bytes of device workspace a call of the given kind and shape needs on the
 * current device (0 if none).  The workspace holds split-K partial sums
 * (scratch, sized for the device's largest grid) followed by per-tile arrival
 * counters (the last 16 * ceil(N/128) bytes, rounded up to 256; for
 * QG_KIND_W8A8, R / 4 bytes for each of its ceil(N/128) * ceil(M/R) tiles,
 * R = 64 for M <= 64, else 128).  It must be
 * zero-filled once before its first use; every successful call leaves its
 * counters at zero again, so one workspace serves later calls of any shape
 * without clearing.  The W8A8 kind lays its workspace out differently (wider
 * partial sums): a workspace serves either QG_KIND_W8A8 calls or calls of
 * the other kinds, not both, unless it is zero-filled again in between.
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
 * Several FP8 block-scaled GEMMs that share X, in one launch: for each
 * segment j, Y_j = X . dequant(W_j)^T -- e.g. the Q, K and V projections of
 * one attention layer ("atlas" m16_tc page, the section on splitting the
 * lever per projection family; its w8a16_gemm_m16_strided kernel).  The
 * segments' 128-row tiles are concatenated into one grid, so the shapes
 * share one launch, one split-K schedule and one per-call start-up cost, and
 * each segment's rows are stored into its own Y with its own row stride.
 * Every segment's result is what qgemm_fp8_block gives for it alone, within
 * the same comparison rule (only the split-K order of the sums can differ).
 *
 *   X, ldx, M, K   as for qgemm_fp8_block, shared by every segment
 *   segments[j]    W, W_scale, Y, ldy and N (>= 1) of segment j, each as
 *                  for qgemm_fp8_block; 1 <= nseg <= QG_MAX_SEGMENTS
 *   workspace      at least qg_workspace_bytes(QG_KIND_FP8_BLOCK, M, R, K)
 *                  bytes, R = the sum over segments of 128 * ceil(N_j / 128);
 *                  the dispatch table is consulted with that same R
 * Arguments are checked segment by segment, in order, before anything is
 * enqueued; the first failing check's status is returned.
 */
#define QG_MAX_SEGMENTS 4

typedef struct qg_fp8_segment {
    const uint8_t *W;       /* device, E4M3 [N, K] row-major, 16-byte aligned */
    const float *W_scale;   /* device, FP32 [ceil(N/128), ceil(K/128)] row-major */
    void *Y;                /* device, BF16 [M, ldy] */
    int64_t ldy;            /* >= N */
    int N;                  /* >= 1 */
} qg_fp8_segment;

qg_status qgemm_fp8_block_multi(const void *X, int64_t ldx,
                                const qg_fp8_segment *segments, int nseg,
                                int M, int K,
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
 * allocates nothing and enqueues nothing but the GEMM kernel.
 *  - Arguments are checked as qgemm_fp8_block checks them, before anything
 *    is enqueued; then a shape whose scratch need (qg_workspace_bytes)
 *    exceeds 8 MiB returns QG_ERR_WORKSPACE, also before anything is enqueued.
 *  - The first call on a device that needs scratch looks up the array's
 *    device address (one runtime query, with that device current); make
 *    that first call before any stream capture.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's contents.  Its arrival counters start at zero and every
 *    successful call leaves them at zero.  A call that runs out of time
 *    (QG_ERR_TIMEOUT) leaves some set: qg_last_device_status, which reports
 *    that timeout, also clears them (on its stream, synchronously), so read
 *    the status after an error before the next call.
 *  - Calls whose execution overlaps on the GPU (different streams, or
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
 * Dense BF16 GEMM (no quantisation), e.g. an output projection (lm_head) at
 * decode batch sizes.
 *   X        device, BF16 [M, ldx], 16-byte aligned, ldx >= K, ldx % 8 == 0
 *   W        device, BF16 [N, K] row-major (row stride K elements), 16-byte
 *            aligned
 *   Y        device, BF16 [M, ldy], ldy >= N
 *   M, N, K  1 <= M <= 32, N >= 1, K % 8 == 0 (ragged N and K tails are
 *            handled)
 *   workspace as for qgemm_fp8_block, with kind QG_KIND_BF16.
 * Results match the strict-K-order FP32 sum within the header's comparison
 * rule (2 BF16 ULP, or the absolute floor for outputs that cancel).
 */
qg_status qgemm_bf16(const void *X, int64_t ldx, const void *W,
                     void *Y, int64_t ldy,
                     int M, int N, int K,
                     void *workspace, size_t workspace_bytes,
                     struct CUstream_st *stream);

/*
 * FP8 activation quantiser of the W8A8 path (block-scaled FP8 GEMMs take FP8
 * activations as well as FP8 weights: "arc" PR page, the cuBLASLt
 * block-scale section).  For every row m and 128-wide K block kb (the last
 * one may be partial):
 *   X_scale[kb * ldsx + m] = max |X[m, k in kb]| / 448 (FP32 division; 1 for
 *                            an all-zero block)
 *   Xq[m * ldxq + k]       = E4M3 code of X[m, k] / X_scale (FP32 division,
 *                            round to nearest even, saturating at +-448)
 * and X_scale[kb * ldsx + m] = 0 for m in [M, ldsx).  Bit-exact: the same
 * FP32 operations in the same order on every device.
 *   X        device, BF16 [M, ldx], 16-byte aligned, ldx >= K, ldx % 8 == 0
 *   Xq       device, E4M3 codes [M, ldxq], 16-byte aligned, ldxq >= K,
 *            ldxq % 16 == 0
 *   X_scale  device, FP32 [ceil(K/128), ldsx], 16-byte aligned,
 *            ldsx >= M rounded up to a multiple of 32, ldsx % 4 == 0
 *   M, K     0 <= M <= 65536, K % 16 == 0
 * Finite inputs only (the codes of Inf and NaN are unspecified).
 */
qg_status qg_quantize_act_e4m3(const void *X, int64_t ldx, uint8_t *Xq, int64_t ldxq,
                               float *X_scale, int64_t ldsx, int M, int K,
                               struct CUstream_st *stream);

/*
 * W8A8 block-scaled GEMM, for batches beyond the decode tier (M > 32, though
 * any M >= 1 is accepted):
 *   Y[m, n] = bf16( sum_kb f(kb, m, n) * sum_{k in kb} xq[m, k] * w[n, k] ),
 *   f(kb, m, n) = X_scale[kb * ldsx + m] * W_scale[n/128, kb]
 * each 128-wide block sum accumulated in FP32 and folded once, with its
 * factor, onto an FP32 outer sum (the two-level fold of qgemm_fp8_block).
 *   Xq, ldxq, X_scale, ldsx  as written by qg_quantize_act_e4m3
 *   W, W_scale, Y, ldy       as for qgemm_fp8_block
 *   M, N, K  1 <= M <= 65536, N >= 1, K % 16 == 0
 *   workspace as for qgemm_fp8_block, with kind QG_KIND_W8A8.
 * Y is written through TMA stores when it is 16-byte aligned and ldy and N
 * are multiples of 8, by plain stores otherwise (same values; only elements
 * of Y[0..M-1][0..N-1] are written either way).
 * Results match the strict-order FP32 fold within the header's comparison
 * rule.
 */
qg_status qgemm_w8a8_block(const uint8_t *Xq, int64_t ldxq, const float *X_scale, int64_t ldsx,
                           const uint8_t *W, const float *W_scale,
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
 * Test aid: the FP8 GEMM's activation split on its own, through the same
 * device functions as the GEMM's split warps.  The weights are never
 * converted (E4M3 goes to the tensor core as stored); instead every
 * (row, 128-wide K block) of BF16 X is scaled by a power of two and split
 * into two E4M3 planes:
 *   e  = min(126, 134 - biased BF16 exponent of the block's largest |x|)
 *        (so the largest |x| * 2^e lies in [128, 256)),
 *   x * 2^e = hi + lo / 16,
 * exactly whenever |x * 2^e| >= 2^-6, and to within 2^-14 below that.
 *   X         device, BF16 [blocks, 128] (one block per row), 16-byte aligned
 *   hi, lo    device, E4M3 codes [blocks, 128], 16-byte aligned
 *   exponent  device, int32 [blocks]: e of each block
 * Non-finite X gives unspecified codes.
 */
qg_status qg_debug_fp8_split(const void *X, int64_t blocks, void *hi, void *lo, int *exponent,
                             struct CUstream_st *stream);

/*
 * Dequantise a packed LUT3 matrix to FP16 D[N, K] (row-major, device) with
 * exactly the conversion the LUT3 GEMM uses: D[n, k] =
 * fp16_rne(qmap[code] * scales[n, k/128]).
 */
qg_status qg_dequant_lut3(const void *Wq, const void *qmap, const void *scales,
                          void *D, int N, int K, struct CUstream_st *stream);

/*
 * Dispatch table.  Each call picks its grid (the number of persistent CTAs,
 * at most one per SM) per (kind, M, N, K): from this process-wide table when
 * it holds an entry for the shape, else from a built-in cost rule (one CTA
 * per 128-row tile when the tiles fit on the SMs and that is cheaper, else
 * stream-K over the SMs).  Any grid gives a result within the comparison rule
 * of the header (only the order of the FP32 split-K sum changes), and a given
 * grid gives the same bits on every call.  Entries are set by a caller that
 * measured the candidates (a tuner, or a test forcing split-K and unsplit
 * runs of one shape).  A changed entry can change qg_workspace_bytes for the
 * shape; the table is shared by all threads and devices.
 *
 * qg_dispatch_set: ctas in 1 .. SM count of the current device sets the
 *   entry (a grid larger than the shape's work units is cut to their
 *   number); ctas == 0 removes it.  M in 1..32 (1..65536 for QG_KIND_W8A8).
 * qg_dispatch_get: the grid the next call of the shape launches on the
 *   current device (0 for invalid arguments).
 * qg_dispatch_rule: the grid the built-in cost rule picks for the shape on
 *   a device with `sms` SMs, whatever the table holds (host only, no CUDA
 *   call; 0 for invalid arguments).
 * qg_dispatch_clear: removes every entry.
 */
qg_status qg_dispatch_set(int kind, int M, int N, int K, int ctas);
int qg_dispatch_get(int kind, int M, int N, int K);
int qg_dispatch_rule(int kind, int M, int N, int K, int sms);
void qg_dispatch_clear(void);

/*
 * The largest workspace any grid of a shape with N output rows may need on
 * the current device (for a multi-segment call, N = the sum of 128 *
 * ceil(N_j / 128)): a workspace of this size serves every dispatch-table
 * entry of such shapes, as qg_tune_* requires.
 */
size_t qg_workspace_bytes_max(int N);

/*
 * The same bound for QG_KIND_W8A8 shapes with M activation rows and N output
 * rows (any K, any grid); 0 for invalid arguments.
 */
size_t qg_workspace_bytes_max_w8a8(int M, int N);

/*
 * Tuning of the dispatch table for one shape: an exactness-gated search
 * (FLUTE "optimized_w3" page, Results: a candidate is accepted only after
 * its output is checked).  The built-in schedule's output, written to Y_ref
 * (a device buffer shaped like Y), is the reference.  Candidate grids (one CTA
 * per 128-row tile, 2..8 CTAs per tile, 4/8..8/8 of the SMs, and, with more
 * tiles than SMs, the largest grid over which whole tiles divide evenly; each
 * at most the SM count) then run on the caller's buffers; a candidate whose output is
 * not finite, or differs from the reference by more than a relative
 * Frobenius distance of 1e-3 or anywhere by more than 1e-2 of the
 * reference's largest magnitude (a reordered FP32 sum moves results by a
 * few units in the last place; a misplaced piece moves them by their own
 * size), is discarded.  The others are timed over `calls` back-to-back calls
 * (CUDA events on `stream`, current launch-overlap setting), the weights
 * rotating over the ncopies equal copies given (copies totalling more than
 * twice the L2 size make the timings stream from HBM), and the fastest
 * becomes the shape's dispatch-table entry (the entry is removed when the
 * built-in grid is the fastest).  Candidates that need more than
 * workspace_bytes of workspace are skipped (qg_workspace_bytes_max(N) serves
 * all).  Synchronous.  *best_ctas and *best_us (either may be NULL) receive
 * the grid chosen and its time per call.  Arguments are those of the GEMM
 * entry point for each W copy.
 */
qg_status qg_tune_fp8(const void *X, int64_t ldx, const uint8_t *const *W_copies, int ncopies,
                      const float *W_scale, void *Y, int64_t ldy, void *Y_ref,
                      int M, int N, int K, void *workspace, size_t workspace_bytes,
                      int calls, int *best_ctas, float *best_us, struct CUstream_st *stream);

qg_status qg_tune_lut3(const void *X, int64_t ldx, const void *const *Wq_copies, int ncopies,
                       const void *qmap, const void *scales, void *Y, int64_t ldy, void *Y_ref,
                       int M, int N, int K, void *workspace, size_t workspace_bytes,
                       int calls, int *best_ctas, float *best_us, struct CUstream_st *stream);

/*
 * The same search for the dense BF16 GEMM (workspace bound
 * qg_workspace_bytes_max(N)) and for the W8A8 GEMM on quantised activations
 * (workspace bound qg_workspace_bytes_max_w8a8(M, N); candidate grids count
 * that kind's tiles of 128 x R rows and units of two K blocks).
 */
qg_status qg_tune_bf16(const void *X, int64_t ldx, const void *const *W_copies, int ncopies,
                       void *Y, int64_t ldy, void *Y_ref, int M, int N, int K,
                       void *workspace, size_t workspace_bytes,
                       int calls, int *best_ctas, float *best_us, struct CUstream_st *stream);

qg_status qg_tune_w8a8(const uint8_t *Xq, int64_t ldxq, const float *X_scale, int64_t ldsx,
                       const uint8_t *const *W_copies, int ncopies, const float *W_scale,
                       void *Y, int64_t ldy, void *Y_ref, int M, int N, int K,
                       void *workspace, size_t workspace_bytes,
                       int calls, int *best_ctas, float *best_us, struct CUstream_st *stream);

/*
 * Test aid: the work split of a shape's schedule, computed on the device by
 * the same functions the GEMM kernels use.  Work units are (128-row tile,
 * 128-wide K block) pairs numbered tile-major, ceil(N/128) * ceil(K/128) in
 * all (QG_KIND_W8A8: tiles of 128 rows x R activation rows as in
 * qg_workspace_bytes, units of two K blocks, ceil(K/256) per tile).  Writes
 * the CTA count to *ctas (host); then, unless ranges or info is
 * null, launches one small kernel on `stream` that writes, for every CTA g:
 *   ranges[2g], ranges[2g+1]   device int64: its units [first, end)
 *   info[6g .. 6g+2]           device int32: for its first tile, the first
 *                              and last CTA holding units of the tile and the
 *                              partial-sum slot (0 or 1) of the first one
 *   info[6g+3 .. 6g+5]         the same for its last tile
 * capacity: the number of CTAs the arrays hold.
 */
qg_status qg_debug_schedule(int kind, int M, int N, int K, int *ctas, int64_t *ranges, int *info, int capacity,
                            struct CUstream_st *stream);

/*
 * Synchronises `stream`, returns the device status word recorded by kernels
 * since the last call (QG_OK if none failed), and clears it.  The word is per
 * process and device, shared by all streams.  On QG_ERR_TIMEOUT it also
 * zeroes the arrival counters of qgemm_fp8_block_noalloc's scratch array on
 * the current device (a caller-owned workspace must be zero-filled by its
 * owner).
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
