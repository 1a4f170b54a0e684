/*
 * bqg_oracle.c -- the CPU oracle for block-quantized skinny GEMV.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes,
 * links or calls this file; only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load it.  It shares no header, helper
 * or table with the CUDA code.
 *
 * Everything here is written to be slow and obviously correct:
 *   - every weight/activation is decoded exactly to double,
 *   - every dot product is one plain left-to-right fp64 sum over k,
 *   - the quantizers are the block encodings taken step by step.
 *
 * Sources (web pages on block-quantized decode matvecs):
 *   [MI50]  "MI50 megakernel" (sebastianhaas.dev), hypothesis ledger:
 *           q4_0 stores 18-byte blocks (fp16 scale + 32 four-bit codes).
 *   [RX6700] "rx-6700xt-llama2-decode" (austxu.dev), Approach & Methodology:
 *           Q4_0 weight x Q8_1 activation integer-dot matvec; fused
 *           gate+up writing SwiGLU; shared-activation QKV.
 *   [SHAPE] "The Shape That Actually Matters" (amarbaro.com), Rounds 1-4:
 *           bf16 and 8-bit GEMV at M=1, K=4096, N=12288.
 *   [PROMPT] "llama-3x-prompt-speed", "the tile": 512-row prefill GEMM
 *           over dequantized weight tiles.
 * Block values follow the llama.cpp convention the pages build on:
 *   q8_0: w = q*d, q int8;  q4_0: w = (q-8)*d, q in 0..15;  q8_1: x = q*d.
 * Readings where the pages are silent are listed at each function.
 *
 * Parity status of each function is pinned by tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 32            /* elements per block, all three block formats */
#define Q8_0_BYTES 34    /* fp16 d + 32 x int8                          */
#define Q4_0_BYTES 18    /* fp16 d + 16 bytes of nibbles  [MI50]        */
#define Q8_1_BYTES 36    /* fp16 d + fp16 s + 32 x int8                 */

enum { FMT_BF16 = 0, FMT_Q8_0 = 1, FMT_Q4_0 = 2, FMT_Q8_1 = 3, FMT_F32 = 4 };

/* ------------------------------------------------------------------ */
/* IEEE binary16 / bfloat16 scalars, from the format definitions.      */
/* ------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double ref_fp16_to_double(uint16_t h)
{
    int sign = h >> 15;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);     /* (1.m) * 2^(e-15)     */
    return sign ? -v : v;
}

/* float -> binary16, round to nearest, ties to even.
 * The value is scaled so that one unit in the last place of the target
 * binade becomes 1, rounded to an integer with nearbyint (default mode is
 * round-to-nearest-even), and scaled back; the result is then encoded. */
uint16_t ref_fp16_from_float(float f)
{
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    if (isnan(f))
        return 0x7e00;
    double a = fabs((double)f);
    if (a >= 65520.0)                /* halfway above 65504 and beyond: inf */
        return sign | 0x7c00;
    int e;
    frexp(a, &e);                    /* a = fr * 2^e, fr in [0.5, 1)        */
    int ulp_exp = (e - 1 < -14) ? -24 : (e - 1) - 10;
    double n = nearbyint(ldexp(a, -ulp_exp));
    double v = ldexp(n, ulp_exp);    /* exactly representable in binary16   */
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -14))         /* subnormal: value = n * 2^-24        */
        return sign | (uint16_t)n;
    frexp(v, &e);
    int biased = (e - 1) + 15;
    uint16_t frac = (uint16_t)(ldexp(v, -(e - 1)) * 1024.0 - 1024.0);
    return sign | (uint16_t)(biased << 10) | frac;
}

/* bfloat16 is the top half of a binary32. */
double ref_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float fp16_to_float(uint16_t h) { return (float)ref_fp16_to_double(h); }

static uint16_t rd_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr_u16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }

/* ------------------------------------------------------------------ */
/* Block encoders.                                                      */
/* Readings (the pages name the formats but do not spell out rounding): */
/*  - the scale is computed in fp32 and rounded once to binary16 (RNE); */
/*  - codes divide by the STORED binary16 scale, in IEEE fp32, and      */
/*    round half away from zero (C roundf);                             */
/*  - a zero scale gives the zero code (q8: 0, q4_0: 8).                */
/* ------------------------------------------------------------------ */

static float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* q8_0 block: d = amax/127, q = round(x/d). */
static void encode_q8_0(const float *x, uint8_t *blk)
{
    float amax = 0.0f;
    for (int i = 0; i < QK; i++)
        if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    uint16_t dh = ref_fp16_from_float(amax / 127.0f);
    float d = fp16_to_float(dh);
    wr_u16(blk, dh);
    for (int i = 0; i < QK; i++) {
        float q = (d == 0.0f) ? 0.0f : clampf(roundf(x[i] / d), -127.0f, 127.0f);
        blk[2 + i] = (uint8_t)(int8_t)q;
    }
}

/* q8_1 block: as q8_0, plus s = d * sum(q) rounded to binary16.  The
 * product of a binary16 scale and |sum q| <= 4064 is exact in fp32.      */
static void encode_q8_1(const float *x, uint8_t *blk)
{
    float amax = 0.0f;
    for (int i = 0; i < QK; i++)
        if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    uint16_t dh = ref_fp16_from_float(amax / 127.0f);
    float d = fp16_to_float(dh);
    int sum = 0;
    for (int i = 0; i < QK; i++) {
        float q = (d == 0.0f) ? 0.0f : clampf(roundf(x[i] / d), -127.0f, 127.0f);
        blk[4 + i] = (uint8_t)(int8_t)q;
        sum += (int)q;
    }
    wr_u16(blk, dh);
    wr_u16(blk + 2, ref_fp16_from_float(d * (float)sum));
}

/* q4_0 block: m = the signed element of largest magnitude (first one on
 * ties), d = m / -8, q = clamp(round(x/d) + 8, 0, 15).  Byte j holds
 * element j in its low nibble and element j+16 in its high nibble.       */
static void encode_q4_0(const float *x, uint8_t *blk)
{
    float m = x[0];
    for (int i = 1; i < QK; i++)
        if (fabsf(x[i]) > fabsf(m)) m = x[i];
    uint16_t dh = ref_fp16_from_float(m / -8.0f);
    float d = fp16_to_float(dh);
    wr_u16(blk, dh);
    int q[QK];
    for (int i = 0; i < QK; i++)
        q[i] = (d == 0.0f) ? 8 : (int)clampf(roundf(x[i] / d) + 8.0f, 0.0f, 15.0f);
    for (int j = 0; j < 16; j++)
        blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

/* x: rows x K fp32, row-major.  out: rows x (K/32) blocks, row-major. */
int ref_quantize(int fmt, const float *x, int64_t rows, int64_t K, uint8_t *out)
{
    if (K % QK) return -1;
    int64_t nb = K / QK;
    int bytes = fmt == FMT_Q8_0 ? Q8_0_BYTES : fmt == FMT_Q4_0 ? Q4_0_BYTES
              : fmt == FMT_Q8_1 ? Q8_1_BYTES : 0;
    if (!bytes) return -2;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < nb; b++) {
            const float *src = x + r * K + b * QK;
            uint8_t *dst = out + (r * nb + b) * bytes;
            if (fmt == FMT_Q8_0) encode_q8_0(src, dst);
            else if (fmt == FMT_Q8_1) encode_q8_1(src, dst);
            else encode_q4_0(src, dst);
        }
    return 0;
}

/* Fused RMSNorm -> q8_1: the normalisation that precedes each projection,
 * folded into the activation encoder so that it is one step instead of two
 * ([MI50] hypothesis ledger: fusing neighbouring steps and epilogues;
 * [RX6700] Approach & Methodology: the Q8_1 activation of the matvec).
 * Reading (the pages name the fusion, not its arithmetic), per row:
 *     s   = sum_k x_k^2               in fp64, k in order (each square of a
 *                                     bf16 input is exact; the sum is exact
 *                                     while the squares span less than 2^37,
 *                                     as for N(0,1) rows, else fp64-rounded)
 *     r   = fp32( 1 / sqrt(s / K + eps) )    (fp64 sqrt and division)
 *     y_k = fp32( fp32(x_k * r) * gamma_k )  (gamma NULL: y_k = fp32(x_k * r))
 * and y is encoded into q8_1 blocks by encode_q8_1 above.
 * x: rows x K fp32 (bf16 inputs are passed exactly as fp32).  out: rows x K/32
 * blocks of 36 bytes. */
int ref_rmsnorm_q8_1(const float *x, const float *gamma, float eps, int64_t rows, int64_t K, uint8_t *out)
{
    if (K <= 0 || K % QK) return -1;
    float *y = (float *)malloc((size_t)K * sizeof(float));
    if (!y) return -3;
    int64_t nb = K / QK;
    for (int64_t r = 0; r < rows; r++) {
        const float *xr = x + r * K;
        double s = 0.0;
        for (int64_t k = 0; k < K; k++) s += (double)xr[k] * (double)xr[k];
        const float rr = (float)(1.0 / sqrt(s / (double)K + (double)eps));
        for (int64_t k = 0; k < K; k++) {
            float v = xr[k] * rr;
            if (gamma) v = v * gamma[k];
            y[k] = v;
        }
        for (int64_t b = 0; b < nb; b++) encode_q8_1(y + b * QK, out + (r * nb + b) * Q8_1_BYTES);
    }
    free(y);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Exact decoding of one row to double.                                 */
/* ------------------------------------------------------------------ */

static int64_t row_bytes(int fmt, int64_t K)
{
    switch (fmt) {
    case FMT_BF16: return 2 * K;
    case FMT_F32:  return 4 * K;
    case FMT_Q8_0: return (K / QK) * Q8_0_BYTES;
    case FMT_Q4_0: return (K / QK) * Q4_0_BYTES;
    case FMT_Q8_1: return (K / QK) * Q8_1_BYTES;
    }
    return -1;
}

static void decode_row(int fmt, const uint8_t *row, int64_t K, double *out)
{
    int64_t nb = K / QK;
    if (fmt == FMT_BF16) {
        for (int64_t k = 0; k < K; k++) out[k] = ref_bf16_to_double(rd_u16(row + 2 * k));
    } else if (fmt == FMT_F32) {
        for (int64_t k = 0; k < K; k++) { float f; memcpy(&f, row + 4 * k, 4); out[k] = f; }
    } else if (fmt == FMT_Q8_0) {
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = row + b * Q8_0_BYTES;
            double d = ref_fp16_to_double(rd_u16(blk));
            for (int i = 0; i < QK; i++) out[b * QK + i] = (double)(int8_t)blk[2 + i] * d;
        }
    } else if (fmt == FMT_Q4_0) {
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = row + b * Q4_0_BYTES;
            double d = ref_fp16_to_double(rd_u16(blk));
            for (int j = 0; j < 16; j++) {
                int lo = blk[2 + j] & 0x0f, hi = blk[2 + j] >> 4;
                out[b * QK + j] = (double)(lo - 8) * d;
                out[b * QK + j + 16] = (double)(hi - 8) * d;
            }
        }
    } else if (fmt == FMT_Q8_1) {
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = row + b * Q8_1_BYTES;
            double d = ref_fp16_to_double(rd_u16(blk));
            for (int i = 0; i < QK; i++) out[b * QK + i] = (double)(int8_t)blk[4 + i] * d;
        }
    }
}

/* rows x K values of any format -> double, row-major. */
int ref_dequantize(int fmt, const uint8_t *src, int64_t rows, int64_t K, double *out)
{
    if (K % QK && fmt != FMT_BF16 && fmt != FMT_F32) return -1;
    int64_t rb = row_bytes(fmt, K);
    if (rb < 0) return -2;
    for (int64_t r = 0; r < rows; r++) decode_row(fmt, src + r * rb, K, out + r * K);
    return 0;
}

/* ------------------------------------------------------------------ */
/* GEMV / skinny GEMM:  Y[m, n] = sum_k W[n, k] * X[m, k]   ([SHAPE])   */
/* W: N rows of K (row n = K/32 consecutive blocks);  X: M rows of K.  */
/* Only the selected rows n (rows[j], or all when rows == NULL) are     */
/* evaluated.  Y and A are M x nsel, row-major; A = sum_k |W X| is the  */
/* scale of the parity tolerance.  Summation: fp64, k = 0, 1, ..., K-1. */
/* nthreads > 1 spreads independent rows over OpenMP threads; each      */
/* row's sum is unchanged, so the result does not depend on it.         */
/* ------------------------------------------------------------------ */
int ref_gemv(int wfmt, const uint8_t *W, int xfmt, const uint8_t *X,
             int64_t M, int64_t N, int64_t K,
             const int64_t *rows, int64_t nsel,
             double *Y, double *A, int nthreads)
{
    if (K <= 0 || M <= 0 || N < 0) return -1;
    int64_t wrb = row_bytes(wfmt, K), xrb = row_bytes(xfmt, K);
    if (wrb < 0 || xrb < 0) return -2;
    if (rows == NULL) nsel = N;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(M * K));
    if (!xd) return -3;
    for (int64_t m = 0; m < M; m++) decode_row(xfmt, X + m * xrb, K, xd + m * K);
    int err = 0;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 16)
#endif
    for (int64_t j = 0; j < nsel; j++) {
        double *w = (double *)malloc(sizeof(double) * (size_t)K);
        if (!w) { err = -3; continue; }
        int64_t n = rows ? rows[j] : j;
        decode_row(wfmt, W + n * wrb, K, w);
        for (int64_t m = 0; m < M; m++) {
            double s = 0.0, a = 0.0;
            const double *x = xd + m * K;
            for (int64_t k = 0; k < K; k++) {
                s += w[k] * x[k];
                a += fabs(w[k] * x[k]);
            }
            Y[m * nsel + j] = s;
            if (A) A[m * nsel + j] = a;
        }
        free(w);
    }
    (void)nthreads;
    free(xd);
    return err;
}

/* Second reference (same loops, fp32 products and fp32 accumulation).
 * Used only to tell a rounding-order difference from a wrong result.   */
int ref_gemv_f32acc(int wfmt, const uint8_t *W, int xfmt, const uint8_t *X,
                    int64_t M, int64_t N, int64_t K, float *Y)
{
    int64_t wrb = row_bytes(wfmt, K), xrb = row_bytes(xfmt, K);
    if (wrb < 0 || xrb < 0) return -2;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(M * K));
    double *w = (double *)malloc(sizeof(double) * (size_t)K);
    if (!xd || !w) { free(xd); free(w); return -3; }
    for (int64_t m = 0; m < M; m++) decode_row(xfmt, X + m * xrb, K, xd + m * K);
    for (int64_t n = 0; n < N; n++) {
        decode_row(wfmt, W + n * wrb, K, w);
        for (int64_t m = 0; m < M; m++) {
            float s = 0.0f;
            for (int64_t k = 0; k < K; k++) {
                float p = (float)w[k] * (float)xd[m * K + k];
                s = s + p;
            }
            Y[m * N + n] = s;
        }
    }
    free(xd);
    free(w);
    return 0;
}

/* q4_0 weight x q8_1 activation, per-block integer dots  [RX6700]:
 *   sumi[n, b] = sum_{i<32} (qw_i - 8) * qx_i        (int64, |.| <= 32512)
 * For one activation row (M = 1).  dots: N x (K/32), row-major.         */
int ref_block_dots_q4_0_q8_1(const uint8_t *W, const uint8_t *Xq, int64_t N, int64_t K, int32_t *dots)
{
    if (K % QK) return -1;
    int64_t nb = K / QK;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *wb = W + (n * nb + b) * Q4_0_BYTES;
            const uint8_t *xb = Xq + b * Q8_1_BYTES;
            int64_t s = 0;
            for (int j = 0; j < 16; j++) {
                int lo = wb[2 + j] & 0x0f, hi = wb[2 + j] >> 4;
                s += (int64_t)(lo - 8) * (int8_t)xb[4 + j];
                s += (int64_t)(hi - 8) * (int8_t)xb[4 + j + 16];
            }
            dots[n * nb + b] = (int32_t)s;
        }
    return 0;
}

/* SwiGLU epilogue  [RX6700]:  h = silu(g) * u,  silu(g) = g / (1 + e^-g). */
void ref_swiglu(const double *g, const double *u, int64_t n, double *h)
{
    for (int64_t i = 0; i < n; i++) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* ------------------------------------------------------------------ */
/* The library's load-time weight layout ("repacked"), restated from    */
/* its published description so the oracle can check the repack        */
/* kernels byte for byte.  nb = K/32 blocks per row, T = ceil(nb/32)    */
/* tiles per row; a tile holds 32 consecutive blocks of one row.        */
/*   bf16 : row-major N x K, unchanged.                                 */
/*   q4_0 : tile = 576 B: slot s (block 32t+s) has its 16 code bytes at */
/*          16*s and its fp16 scale at 512 + 2*s.                       */
/*   q8_0 : tile = 1088 B: slot s has codes 0..15 at 16*s, codes 16..31 */
/*          at 512 + 16*s, and its fp16 scale at 1024 + 2*s.            */
/* Rows follow each other with stride T * tile bytes; unused slots of   */
/* the last tile are zero.                                              */
/* ------------------------------------------------------------------ */
static int64_t tile_bytes(int fmt) { return fmt == FMT_Q4_0 ? 576 : fmt == FMT_Q8_0 ? 1088 : 0; }

int64_t ref_repacked_size(int fmt, int64_t N, int64_t K)
{
    if (K % QK || N < 0) return -1;
    if (fmt == FMT_BF16) return N * K * 2;
    int64_t nb = K / QK, T = (nb + 31) / 32;
    if (!tile_bytes(fmt)) return -1;
    return N * T * tile_bytes(fmt);
}

int ref_repack(int fmt, const uint8_t *canon, int64_t N, int64_t K, uint8_t *packed)
{
    int64_t size = ref_repacked_size(fmt, N, K);
    if (size < 0) return -1;
    if (fmt == FMT_BF16) { memcpy(packed, canon, (size_t)size); return 0; }
    memset(packed, 0, (size_t)size);
    int64_t nb = K / QK, T = (nb + 31) / 32, tb = tile_bytes(fmt);
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++) {
            uint8_t *tile = packed + (n * T + b / 32) * tb;
            int64_t s = b % 32;
            if (fmt == FMT_Q4_0) {
                const uint8_t *blk = canon + (n * nb + b) * Q4_0_BYTES;
                memcpy(tile + 16 * s, blk + 2, 16);
                memcpy(tile + 512 + 2 * s, blk, 2);
            } else {
                const uint8_t *blk = canon + (n * nb + b) * Q8_0_BYTES;
                memcpy(tile + 16 * s, blk + 2, 16);
                memcpy(tile + 512 + 16 * s, blk + 18, 16);
                memcpy(tile + 1024 + 2 * s, blk, 2);
            }
        }
    return 0;
}

int ref_unrepack(int fmt, const uint8_t *packed, int64_t N, int64_t K, uint8_t *canon)
{
    int64_t size = ref_repacked_size(fmt, N, K);
    if (size < 0) return -1;
    if (fmt == FMT_BF16) { memcpy(canon, packed, (size_t)size); return 0; }
    int64_t nb = K / QK, T = (nb + 31) / 32, tb = tile_bytes(fmt);
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *tile = packed + (n * T + b / 32) * tb;
            int64_t s = b % 32;
            if (fmt == FMT_Q4_0) {
                uint8_t *blk = canon + (n * nb + b) * Q4_0_BYTES;
                memcpy(blk + 2, tile + 16 * s, 16);
                memcpy(blk, tile + 512 + 2 * s, 2);
            } else {
                uint8_t *blk = canon + (n * nb + b) * Q8_0_BYTES;
                memcpy(blk + 2, tile + 16 * s, 16);
                memcpy(blk + 18, tile + 512 + 16 * s, 16);
                memcpy(blk, tile + 1024 + 2 * s, 2);
            }
        }
    return 0;
}

/* Number of OpenMP threads the oracle would use (1 without OpenMP). */
int ref_openmp_max_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
