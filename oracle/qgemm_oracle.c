/*
 * CPU oracle for the weight-only quantized decode GEMM -- TEST INFRASTRUCTURE.
 *
 * Only the test suite, the package's smoke check and the benchmark's CPU
 * baseline leg may call this library.  It shares no code, header, table or
 * constant with the CUDA path, and the CUDA path never calls it.
 *
 * Everything here is a literal, slow restatement of what the method computes:
 *
 *  - FP8 E4M3 decode (OCP 8-bit floating point, E4M3FN flavour: bias 7,
 *    no infinities, S.1111.111 is NaN, exponent field 0 is subnormal m*2^-9).
 *  - The W8A16 block-scaled GEMM with the two-level fold described on the
 *    "atlas" m16_tc module page (section "NUMERICS"): every 128-wide K block is
 *    summed in its own FP32 accumulator in strict K order, that block sum is
 *    multiplied by the block's FP32 scale once, and the product is added to an
 *    FP32 outer accumulator; K blocks are taken in ascending order; the output
 *    is rounded to BF16 (round to nearest, ties to even).
 *  - The 3-bit learned-LUT GEMM of the FLUTE "optimized_w3" page (section
 *    "Results", accuracy bullet): each weight is dequantised as
 *    fp16_rne(qmap[code] * scale[n, k/128]) before accumulation, the products
 *    with the FP16 activations are summed in FP32 in strict K order, and the
 *    sum is rounded to FP16.
 *  - The W8A8 block-scaled GEMM (FP8 activations as well as weights): the
 *    "arc" PR page's cuBLASLt block-scale section notes that block-scaled FP8
 *    needs FP8 activations and so an activation quantiser.  Activations are
 *    quantised per (row, 128-wide K block) with the weights' rule (scale =
 *    block amax / 448, codes = E4M3 round-to-nearest-even of x / scale,
 *    saturating at 448); the GEMM is the two-level fold with the product of
 *    the two block scales as the block factor.
 *  - The unquantised BF16 decode GEMM named beside the FP8 tier on the
 *    "atlas" m16_tc page (the numerics contract section: the BF16 lm_head
 *    tier graded by the same comparison): BF16 X and W, products summed in
 *    FP32 in strict K order, the sum rounded to BF16.
 *  - The tiled nibble packing of 3-bit codes (the layout documented in
 *    include/qgemm.h), written independently from that document.
 *
 * Build with -ffp-contract=off so that every multiply and add rounds on its
 * own (no fused multiply-add), as the definitions above require.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Scalar formats                                                      */
/* ------------------------------------------------------------------ */

/* OCP E4M3FN: value = (-1)^s * 2^(e-7) * (1 + m/8) for e > 0,
 *             (-1)^s * 2^-6 * (m/8) for e == 0; e == 15 && m == 7 is NaN. */
float oracle_e4m3_to_float(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    float mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexpf((float)m / 8.0f, -6);
    else
        mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return s ? -mag : mag;
}

float oracle_bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
float oracle_fp16_to_float(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    float mag;
    if (e == 31)
        mag = m ? NAN : INFINITY;
    else if (e == 0)
        mag = ldexpf((float)m, -24);
    else
        mag = ldexpf(1.0f + (float)m / 1024.0f, e - 15);
    return s ? -mag : mag;
}

/*
 * Round a finite, non-negative double `a` to a binary floating-point format
 * with `p` significand bits (hidden bit included), minimum normal exponent
 * `emin` (so the subnormal quantum is 2^(emin-p+1)), ties to even.  The result
 * is returned as a double (exactly representable); overflow is the caller's
 * business.  nearbyint() rounds to nearest even in the default mode.
 */
static double round_to_format(double a, int p, int emin)
{
    int ex;
    double q, ulp;
    if (a == 0.0)
        return 0.0;
    frexp(a, &ex);              /* a = f * 2^ex, f in [0.5, 1) */
    ex -= 1;                    /* a in [2^ex, 2^(ex+1)) */
    if (ex < emin)
        ex = emin;              /* subnormal range: fixed quantum */
    ulp = ldexp(1.0, ex - (p - 1));
    q = nearbyint(a / ulp);
    return q * ulp;
}

/* float -> BF16 bits, round to nearest even (8 significand bits, emin -126). */
uint16_t oracle_float_to_bf16_rne(float f)
{
    uint32_t u;
    double a, r;
    uint16_t sign;
    int ex;
    memcpy(&u, &f, 4);
    sign = (uint16_t)((u >> 16) & 0x8000);
    if (isnan(f))
        return (uint16_t)(sign | 0x7FC0);
    a = fabs((double)f);
    if (isinf(f))
        return (uint16_t)(sign | 0x7F80);
    r = round_to_format(a, 8, -126);
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -126))              /* subnormal: m * 2^-133 */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -133)));
    frexp(r, &ex);
    ex -= 1;
    return (uint16_t)(sign | (uint16_t)((ex + 127) << 7) |
                      (uint16_t)((r / ldexp(1.0, ex) - 1.0) * 128.0));
}

/* float -> FP16 bits, round to nearest even (11 significand bits, emin -14). */
uint16_t oracle_float_to_fp16_rne(float f)
{
    uint32_t u;
    double a, r;
    uint16_t sign;
    int ex;
    memcpy(&u, &f, 4);
    sign = (uint16_t)((u >> 16) & 0x8000);
    if (isnan(f))
        return (uint16_t)(sign | 0x7E00);
    a = fabs((double)f);
    if (isinf(f))
        return (uint16_t)(sign | 0x7C00);
    r = round_to_format(a, 11, -14);
    if (r >= 65536.0)
        return (uint16_t)(sign | 0x7C00);
    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -14))               /* subnormal: m * 2^-24 */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
    frexp(r, &ex);
    ex -= 1;
    return (uint16_t)(sign | (uint16_t)((ex + 15) << 10) |
                      (uint16_t)((r / ldexp(1.0, ex) - 1.0) * 1024.0));
}

/* Array forms of the scalar conversions above (same functions, element by element). */
void oracle_e4m3_to_float_array(int64_t n, const uint8_t *in, float *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = oracle_e4m3_to_float(in[i]);
}

void oracle_fp16_to_float_array(int64_t n, const uint16_t *in, float *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = oracle_fp16_to_float(in[i]);
}

void oracle_float_to_bf16_array(int64_t n, const float *in, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = oracle_float_to_bf16_rne(in[i]);
}

void oracle_float_to_fp16_array(int64_t n, const float *in, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = oracle_float_to_fp16_rne(in[i]);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* W8A16 FP8 block-scaled GEMM, two-level fold                          */
/* ------------------------------------------------------------------ */

/*
 * One output element Y[m, n] as an FP32 value (before BF16 rounding).
 *   X: BF16 bits, row m starts at X + m*ldx
 *   Wrow: E4M3 codes of weight row n (K codes)
 *   S: FP32 scales, [ceil(N/128), ceil(K/128)], row stride lds
 */
static float fp8_element(int K, const uint16_t *xrow, const uint8_t *wrow,
                         const float *srow)
{
    int kb, k, KB = (K + 127) / 128;
    float outer = 0.0f;
    for (kb = 0; kb < KB; ++kb) {
        int k0 = 128 * kb;
        int k1 = k0 + 128 < K ? k0 + 128 : K;
        float inner = 0.0f;
        for (k = k0; k < k1; ++k) {
            float prod = oracle_bf16_to_float(xrow[k]) * oracle_e4m3_to_float(wrow[k]);
            inner = inner + prod;
        }
        {
            float scaled = inner * srow[kb];
            outer = outer + scaled;
        }
    }
    return outer;
}

/*
 * Full product.  Y (BF16 bits, row stride ldy) and, if non-NULL, Yf (FP32
 * pre-rounding values, row stride ldy) receive M x N outputs.
 */
void oracle_qgemm_fp8_block(int M, int N, int K,
                            const uint16_t *X, int64_t ldx,
                            const uint8_t *W, int64_t ldw,
                            const float *S, int64_t lds,
                            uint16_t *Y, float *Yf, int64_t ldy, int nthreads)
{
    int n;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (n = 0; n < N; ++n) {
        int m;
        const uint8_t *wrow = W + (int64_t)n * ldw;
        const float *srow = S + (int64_t)(n / 128) * lds;
        for (m = 0; m < M; ++m) {
            float v = fp8_element(K, X + (int64_t)m * ldx, wrow, srow);
            if (Y)
                Y[(int64_t)m * ldy + n] = oracle_float_to_bf16_rne(v);
            if (Yf)
                Yf[(int64_t)m * ldy + n] = v;
        }
    }
}

/* Selected elements (ms[i], ns[i]) only; outputs are dense arrays of length count. */
void oracle_qgemm_fp8_block_sample(int M, int N, int K,
                                   const uint16_t *X, int64_t ldx,
                                   const uint8_t *W, int64_t ldw,
                                   const float *S, int64_t lds,
                                   const int32_t *ms, const int32_t *ns, int64_t count,
                                   uint16_t *Y, float *Yf, int nthreads)
{
    int64_t i;
    (void)M; (void)N;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
    for (i = 0; i < count; ++i) {
        int m = ms[i], n = ns[i];
        float v = fp8_element(K, X + (int64_t)m * ldx, W + (int64_t)n * ldw,
                              S + (int64_t)(n / 128) * lds);
        if (Y)
            Y[i] = oracle_float_to_bf16_rne(v);
        if (Yf)
            Yf[i] = v;
    }
}

/*
 * Absolute mass of the two-level sum, in double:
 *   A[m, n] = sum_kb |s[n/128, kb]| * sum_{k in kb} |x[m,k] * q[n,k]|.
 * It scales the absolute floor of the comparison criterion.  Either a full
 * M x N array (ms == NULL) or the listed elements.
 */
void oracle_fp8_abs_mass(int M, int N, int K,
                         const uint16_t *X, int64_t ldx,
                         const uint8_t *W, int64_t ldw,
                         const float *S, int64_t lds,
                         const int32_t *ms, const int32_t *ns, int64_t count,
                         double *A, int nthreads)
{
    int64_t i, total = ms ? count : (int64_t)M * N;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
    for (i = 0; i < total; ++i) {
        int m = ms ? ms[i] : (int)(i / N);
        int n = ms ? ns[i] : (int)(i % N);
        int kb, k, KB = (K + 127) / 128;
        double acc = 0.0;
        for (kb = 0; kb < KB; ++kb) {
            int k0 = 128 * kb, k1 = k0 + 128 < K ? k0 + 128 : K;
            double blk = 0.0;
            for (k = k0; k < k1; ++k)
                blk += fabs((double)oracle_bf16_to_float(X[(int64_t)m * ldx + k]) *
                            (double)oracle_e4m3_to_float(W[(int64_t)n * ldw + k]));
            acc += fabs((double)S[(int64_t)(n / 128) * lds + kb]) * blk;
        }
        A[i] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* E4M3 encoding, activation quantiser, W8A8 block-scaled GEMM          */
/* ------------------------------------------------------------------ */

/* float -> E4M3FN code: round to nearest even on the E4M3 grid (4
 * significand bits, smallest normal 2^-6, subnormal quantum 2^-9), values
 * that round beyond the largest finite value 448 saturate to +-448; NaN gives
 * the NaN code. */
uint8_t oracle_float_to_e4m3_rne_sat(float f)
{
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double r;
    int ex;
    if (isnan(f))
        return (uint8_t)(sign | 0x7F);
    r = round_to_format(fabs((double)f), 4, -6);
    if (r > 448.0)
        r = 448.0;
    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -6))                /* subnormal: m * 2^-9 */
        return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    frexp(r, &ex);
    ex -= 1;
    return (uint8_t)(sign | (uint8_t)((ex + 7) << 3) | (uint8_t)((r / ldexp(1.0, ex) - 1.0) * 8.0));
}

/*
 * Activation quantiser.  For every row m and 128-wide K block kb (the last
 * one possibly partial): amax = max |x| over the block, s = fl32(amax / 448)
 * (s = 1 for an all-zero block), q = e4m3(fl32(x / s)).  Xq: [M, K] codes
 * (row stride ldxq); Sx: [ceil(K/128), ldsx] scales, entry (kb, m).
 */
void oracle_quantize_act_e4m3(int M, int K, const uint16_t *X, int64_t ldx,
                              uint8_t *Xq, int64_t ldxq, float *Sx, int64_t ldsx)
{
    int m, kb, k, KB = (K + 127) / 128;
    for (m = 0; m < M; ++m) {
        for (kb = 0; kb < KB; ++kb) {
            int k0 = 128 * kb, k1 = k0 + 128 < K ? k0 + 128 : K;
            float amax = 0.0f, sc;
            for (k = k0; k < k1; ++k) {
                float a = fabsf(oracle_bf16_to_float(X[(int64_t)m * ldx + k]));
                if (a > amax)
                    amax = a;
            }
            sc = amax > 0.0f ? amax / 448.0f : 1.0f;
            Sx[(int64_t)kb * ldsx + m] = sc;
            for (k = k0; k < k1; ++k) {
                float q = oracle_bf16_to_float(X[(int64_t)m * ldx + k]) / sc;
                Xq[(int64_t)m * ldxq + k] = oracle_float_to_e4m3_rne_sat(q);
            }
        }
    }
}

/* One output of the W8A8 two-level fold, as FP32. */
static float w8a8_element(int K, const uint8_t *xrow, const float *sx, int64_t ldsx,
                          const uint8_t *wrow, const float *srow)
{
    int kb, k, KB = (K + 127) / 128;
    float outer = 0.0f;
    for (kb = 0; kb < KB; ++kb) {
        int k0 = 128 * kb;
        int k1 = k0 + 128 < K ? k0 + 128 : K;
        float inner = 0.0f;
        for (k = k0; k < k1; ++k) {
            float prod = oracle_e4m3_to_float(xrow[k]) * oracle_e4m3_to_float(wrow[k]);
            inner = inner + prod;
        }
        {
            float factor = sx[(int64_t)kb * ldsx] * srow[kb];
            float scaled = inner * factor;
            outer = outer + scaled;
        }
    }
    return outer;
}

/*
 * Y = bf16(sum_kb fl32(inner_kb * fl32(sx[kb, m] * sw[n/128, kb]))), K blocks
 * ascending, inner_kb the strict-K FP32 sum of the exact E4M3 x E4M3
 * products of the block.
 */
void oracle_qgemm_w8a8_block(int M, int N, int K,
                             const uint8_t *Xq, int64_t ldxq, const float *Sx, int64_t ldsx,
                             const uint8_t *W, int64_t ldw, const float *Sw, int64_t lds,
                             uint16_t *Y, float *Yf, int64_t ldy, int nthreads)
{
    int n;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (n = 0; n < N; ++n) {
        int m;
        for (m = 0; m < M; ++m) {
            float v = w8a8_element(K, Xq + (int64_t)m * ldxq, Sx + m, ldsx, W + (int64_t)n * ldw,
                                   Sw + (int64_t)(n / 128) * lds);
            if (Y)
                Y[(int64_t)m * ldy + n] = oracle_float_to_bf16_rne(v);
            if (Yf)
                Yf[(int64_t)m * ldy + n] = v;
        }
    }
}

/* A[m, n] = sum_kb |sx * sw| * sum_{k in kb} |xq * wq| in double. */
void oracle_w8a8_abs_mass(int M, int N, int K,
                          const uint8_t *Xq, int64_t ldxq, const float *Sx, int64_t ldsx,
                          const uint8_t *W, int64_t ldw, const float *Sw, int64_t lds,
                          double *A, int nthreads)
{
    int64_t i, total = (int64_t)M * N;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
    for (i = 0; i < total; ++i) {
        int m = (int)(i / N), n = (int)(i % N);
        int kb, k, KB = (K + 127) / 128;
        double acc = 0.0;
        for (kb = 0; kb < KB; ++kb) {
            int k0 = 128 * kb, k1 = k0 + 128 < K ? k0 + 128 : K;
            double blk = 0.0;
            for (k = k0; k < k1; ++k)
                blk += fabs((double)oracle_e4m3_to_float(Xq[(int64_t)m * ldxq + k]) *
                            (double)oracle_e4m3_to_float(W[(int64_t)n * ldw + k]));
            acc += fabs((double)Sx[(int64_t)kb * ldsx + m] * (double)Sw[(int64_t)(n / 128) * lds + kb]) * blk;
        }
        A[i] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* Dense BF16 GEMM                                                      */
/* ------------------------------------------------------------------ */

/* sum_k x[k] * w[k] in FP32, strictly ascending k (each product is exact). */
static float bf16_element(int K, const uint16_t *xrow, const uint16_t *wrow)
{
    int k;
    float acc = 0.0f;
    for (k = 0; k < K; ++k) {
        float prod = oracle_bf16_to_float(xrow[k]) * oracle_bf16_to_float(wrow[k]);
        acc = acc + prod;
    }
    return acc;
}

/* Y = bf16_rne(X[M,K] . W[N,K]^T); Yf (optional) the FP32 sums. */
void oracle_gemm_bf16(int M, int N, int K,
                      const uint16_t *X, int64_t ldx,
                      const uint16_t *W, int64_t ldw,
                      uint16_t *Y, float *Yf, int64_t ldy, int nthreads)
{
    int n;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (n = 0; n < N; ++n) {
        int m;
        for (m = 0; m < M; ++m) {
            float v = bf16_element(K, X + (int64_t)m * ldx, W + (int64_t)n * ldw);
            if (Y)
                Y[(int64_t)m * ldy + n] = oracle_float_to_bf16_rne(v);
            if (Yf)
                Yf[(int64_t)m * ldy + n] = v;
        }
    }
}

void oracle_gemm_bf16_sample(int M, int N, int K,
                             const uint16_t *X, int64_t ldx,
                             const uint16_t *W, int64_t ldw,
                             const int32_t *ms, const int32_t *ns, int64_t count,
                             uint16_t *Y, float *Yf, int nthreads)
{
    int64_t i;
    (void)M; (void)N;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
    for (i = 0; i < count; ++i) {
        float v = bf16_element(K, X + (int64_t)ms[i] * ldx, W + (int64_t)ns[i] * ldw);
        if (Y)
            Y[i] = oracle_float_to_bf16_rne(v);
        if (Yf)
            Yf[i] = v;
    }
}

/* A[m, n] = sum_k |x[m,k] * w[n,k]| in double (full array or listed elements). */
void oracle_bf16_abs_mass(int M, int N, int K,
                          const uint16_t *X, int64_t ldx,
                          const uint16_t *W, int64_t ldw,
                          const int32_t *ms, const int32_t *ns, int64_t count,
                          double *A, int nthreads)
{
    int64_t i, total = ms ? count : (int64_t)M * N;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
    for (i = 0; i < total; ++i) {
        int m = ms ? ms[i] : (int)(i / N);
        int n = ms ? ns[i] : (int)(i % N);
        int k;
        double acc = 0.0;
        for (k = 0; k < K; ++k)
            acc += fabs((double)oracle_bf16_to_float(X[(int64_t)m * ldx + k]) *
                        (double)oracle_bf16_to_float(W[(int64_t)n * ldw + k]));
        A[i] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* W3A16 learned-LUT GEMM                                               */
/* ------------------------------------------------------------------ */

/* d = fp16_rne(qmap[code] * scale); both factors are FP16, so the FP32
 * product is exact and a single rounding to FP16 follows. */
uint16_t oracle_lut3_dequant(uint8_t code, const uint16_t *qmap, uint16_t scale)
{
    float p = oracle_fp16_to_float(qmap[code & 7]) * oracle_fp16_to_float(scale);
    return oracle_float_to_fp16_rne(p);
}

/* Dequantised weight matrix D[N, K] (FP16 bits) from unpacked codes. */
void oracle_lut3_dequant_matrix(int N, int K, const uint8_t *codes, int64_t ldc,
                                const uint16_t *qmap, const uint16_t *scales, int64_t ldsc,
                                uint16_t *D, int64_t ldd)
{
    int n, k;
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k)
            D[(int64_t)n * ldd + k] = oracle_lut3_dequant(codes[(int64_t)n * ldc + k], qmap,
                                                          scales[(int64_t)n * ldsc + k / 128]);
}

static float lut3_element(int K, const uint16_t *xrow, const uint8_t *crow,
                          const uint16_t *qmap, const uint16_t *srow)
{
    int k;
    float acc = 0.0f;
    for (k = 0; k < K; ++k) {
        uint16_t d = oracle_lut3_dequant(crow[k], qmap, srow[k / 128]);
        float prod = oracle_fp16_to_float(xrow[k]) * oracle_fp16_to_float(d);
        acc = acc + prod;
    }
    return acc;
}

void oracle_qgemm_lut3(int M, int N, int K,
                       const uint16_t *X, int64_t ldx,
                       const uint8_t *codes, int64_t ldc,
                       const uint16_t *qmap, const uint16_t *scales, int64_t ldsc,
                       uint16_t *Y, float *Yf, int64_t ldy, int nthreads)
{
    int n;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (n = 0; n < N; ++n) {
        int m;
        for (m = 0; m < M; ++m) {
            float v = lut3_element(K, X + (int64_t)m * ldx, codes + (int64_t)n * ldc, qmap,
                                   scales + (int64_t)n * ldsc);
            if (Y)
                Y[(int64_t)m * ldy + n] = oracle_float_to_fp16_rne(v);
            if (Yf)
                Yf[(int64_t)m * ldy + n] = v;
        }
    }
}

void oracle_qgemm_lut3_sample(int M, int N, int K,
                              const uint16_t *X, int64_t ldx,
                              const uint8_t *codes, int64_t ldc,
                              const uint16_t *qmap, const uint16_t *scales, int64_t ldsc,
                              const int32_t *ms, const int32_t *ns, int64_t count,
                              uint16_t *Y, float *Yf, int nthreads)
{
    int64_t i;
    (void)M; (void)N;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
    for (i = 0; i < count; ++i) {
        float v = lut3_element(K, X + (int64_t)ms[i] * ldx, codes + (int64_t)ns[i] * ldc, qmap,
                               scales + (int64_t)ns[i] * ldsc);
        if (Y)
            Y[i] = oracle_float_to_fp16_rne(v);
        if (Yf)
            Yf[i] = v;
    }
}

/* A[m, n] = sum_k |x[m,k] * d[n,k]| in double (floor scale for the LUT path). */
void oracle_lut3_abs_mass(int M, int N, int K,
                          const uint16_t *X, int64_t ldx,
                          const uint8_t *codes, int64_t ldc,
                          const uint16_t *qmap, const uint16_t *scales, int64_t ldsc,
                          const int32_t *ms, const int32_t *ns, int64_t count,
                          double *A, int nthreads)
{
    int64_t i, total = ms ? count : (int64_t)M * N;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
    for (i = 0; i < total; ++i) {
        int m = ms ? ms[i] : (int)(i / N);
        int n = ms ? ns[i] : (int)(i % N);
        int k;
        double acc = 0.0;
        for (k = 0; k < K; ++k) {
            uint16_t d = oracle_lut3_dequant(codes[(int64_t)n * ldc + k], qmap,
                                             scales[(int64_t)n * ldsc + k / 128]);
            acc += fabs((double)oracle_fp16_to_float(X[(int64_t)m * ldx + k]) *
                        (double)oracle_fp16_to_float(d));
        }
        A[i] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* Tiled nibble packing of 3-bit codes                                  */
/* ------------------------------------------------------------------ */
/*
 * Layout (restated from its specification):
 *   tiles of 128 rows x 256 codes; tile (tn, tk) is the (tn * KT + tk)-th
 *   16384-byte block, KT = ceil(K/256);
 *   inside a tile, 16-byte chunk (q, r) for q = 0..7 (32 codes each along K)
 *   and r = 0..127 (row) sits at byte (q * 128 + r) * 16;
 *   a chunk is four little-endian 32-bit words; word w holds the codes of
 *   k = 256*tk + 32*q + 8*w + i in nibble i (bits 4i..4i+3);
 *   rows >= N and columns >= K hold code 0.
 */
int64_t oracle_lut3_packed_bytes(int N, int K)
{
    return (int64_t)((N + 127) / 128) * ((K + 255) / 256) * 16384;
}

static int64_t nibble_offset(int KT, int n, int k, int *shift)
{
    int tn = n / 128, r = n % 128, tk = k / 256, kk = k % 256;
    int q = kk / 32, w = (kk % 32) / 8, i = kk % 8;
    int64_t byte = (int64_t)(tn * KT + tk) * 16384 + (int64_t)(q * 128 + r) * 16 + w * 4 + i / 2;
    *shift = 4 * (i % 2);
    return byte;
}

void oracle_pack_lut3(int N, int K, const uint8_t *codes, uint8_t *packed)
{
    int KT = (K + 255) / 256, n, k, sh;
    memset(packed, 0, (size_t)oracle_lut3_packed_bytes(N, K));
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k) {
            int64_t b = nibble_offset(KT, n, k, &sh);
            packed[b] = (uint8_t)(packed[b] | ((codes[(int64_t)n * K + k] & 7) << sh));
        }
}

void oracle_unpack_lut3(int N, int K, const uint8_t *packed, uint8_t *codes)
{
    int KT = (K + 255) / 256, n, k, sh;
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k) {
            int64_t b = nibble_offset(KT, n, k, &sh);
            codes[(int64_t)n * K + k] = (uint8_t)((packed[b] >> sh) & 15);
        }
}
