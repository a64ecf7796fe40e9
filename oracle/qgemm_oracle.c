/*
 * CPU oracle for the groupwise int4/int5 weight-only dequant-GEMM.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package entry point's smoke
 * check and the benchmark's CPU-baseline leg may load or call this code.  It
 * shares nothing with the CUDA library (no headers, no helpers, no tables):
 * its code unpacking, its fp16/bf16 decoding and its arithmetic are written
 * here from the definition and nowhere else.
 *
 * What it computes is the plain definition, in fp64, single-threaded:
 *
 *     Y[t][n] = sum_k  x[t][k] * ( s[n][k/64] * q[n][k] ),   k ascending
 *     A[t][n] = sum_k |x[t][k] * ( s[n][k/64] * q[n][k] )|
 *
 * - groupwise-int weights with one scale per 64 K-columns per row
 *   ("ninfer-3080 docs/performance.md", the cuBLAS prefill route section:
 *   cuBLAS reduces over all of K and so cannot apply a scale per 64 columns);
 * - the Q4 and Q5 codecs, Q5 carrying one more (high) bit per code
 *   (same page, the small-T kernels section on the Q5 counterpart);
 * - an fp64 oracle as the accuracy yardstick (same page, the A8 prefill
 *   routes section, which reports relative L2 against an FP64 oracle);
 * - codes are symmetric two's complement with no zero point: int4 in [-8, 7],
 *   int5 in [-16, 15]; scales are IEEE fp16; activations are bf16;
 * - the FP8 codec (the FP8-weight kernel the "Speculative decoding" page checks
 *   at verify widths) holds OCP E4M3 codes: sign, 4 exponent bits with bias 7,
 *   3 mantissa bits, subnormals at exponent 0, no infinities, and NaN for the
 *   two codes S.1111.111; with the same fp16 scale per 64 columns.
 *
 * Every product x * s * q is exact in fp64 (bf16 has 8 significant bits,
 * fp16 11, a code at most 5), so the only roundings are those of the running
 * sum, in ascending k.
 *
 * Canonical packing read here (the library's input format):
 * - int4: ceil(K/2) bytes per row; byte j holds code 2j in bits 0-3 and code
 *   2j+1 in bits 4-7.
 * - fp8: K bytes per row, byte k = the E4M3 code of column k.
 * - int5: ceil(5K/8) bytes per row; LSB-first bitstream, code k in bits
 *   5k .. 5k+4.
 * Scales: fp16 bit patterns, row-major [N][ceil(K/64)]; the last group of a
 * row may be shorter than 64 when K is not a multiple of 64 (the library
 * itself requires K % 64 == 0; the oracle accepts any K so that tiny
 * brute-force cases can run).
 * X: bf16 bit patterns, row-major [T][K].  Y, A: fp64, row-major [T][N].
 *
 * The two fused outputs of the pages' projections ("ninfer-3080
 * docs/performance.md": LinearAdd on the attention o_proj and GDN out_proj,
 * the SwiGLU gate/up pair on the MLP) are written out the same way:
 *
 *     linear add:  Y[t][n] = R[t][n] + sum_k x[t][k] * w[n][k]
 *     SwiGLU:      out[t][f] = silu(g[t][f]) * u[t][f],  silu(z) = z / (1 + e^-z)
 *
 * with g and u the plain results of the gate and the up matrix.
 *
 * The NVFP4 codec (the "nvfp4" weight profile of the pages' RTX 5090
 * publication index) is read here as the common NVFP4 definition: FP4 E2M1
 * codes (sign, 2 exponent bits with bias 1, 1 mantissa bit, a subnormal at
 * exponent 0: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), one unsigned E4M3
 * scale (4 exponent bits, bias 7, 3 mantissa bits, subnormals, no sign; the
 * code 0x7F and codes with bit 7 set are outside the codec) per 16
 * consecutive K-columns per row, and one fp32 scale for the whole tensor:
 *
 *     w[n][k] = e2m1(c[n][k]) * ue4m3(b[n][k/16]) * s_t
 *
 * Codes are packed two per byte like int4 (byte j: column 2j in bits 0-3,
 * 2j+1 in bits 4-7); block scales are bytes [N][ceil(K/16)].  Every product
 * x * w is exact in fp64 (8 + 2 + 4 + 24 significant bits).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_GROUP 64

/* IEEE binary16 -> double, from the field definitions. */
static double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* subnormal: m * 2^-24 */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), expo - 25);  /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 -> double: a bf16 pattern is the top half of an IEEE binary32. */
static double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int qgemm_oracle_row_bytes(int bits, int K)
{
    if ((bits != 4 && bits != 5 && bits != 8) || K < 0)
        return -1;
    return (int)(((long)K * bits + 7) / 8);
}

/* OCP FP8 E4M3 -> double, from the field definitions. */
static double oracle_e4m3_to_double(uint8_t b)
{
    int sign = b >> 7;
    int expo = (b >> 3) & 0x0f;
    int mant = b & 0x07;
    double v;
    if (expo == 15 && mant == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)mant, -9);                  /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + mant), expo - 10);     /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

int qgemm_oracle_groups(int K)
{
    return (K + ORACLE_GROUP - 1) / ORACLE_GROUP;
}

/* Two's-complement code k of one canonical row. */
static int oracle_code(int bits, const uint8_t *row, int k)
{
    if (bits == 4) {
        int byte = row[k >> 1];
        int nib = (k & 1) ? (byte >> 4) : (byte & 0x0f);
        return nib >= 8 ? nib - 16 : nib;
    } else {
        long bit = 5L * k;
        int v = 0;
        for (int b = 0; b < 5; ++b) {
            long p = bit + b;
            v |= ((row[p >> 3] >> (p & 7)) & 1) << b;
        }
        return v >= 16 ? v - 32 : v;
    }
}

/* Value of code k of one canonical row: the integer code, or the E4M3 value. */
static double oracle_value(int bits, const uint8_t *row, int k)
{
    if (bits == 8)
        return oracle_e4m3_to_double(row[k]);
    return (double)oracle_code(bits, row, k);
}

/* Integer codes [N][K] (unpacking only; fp8 codes come back as their bytes). */
int qgemm_oracle_unpack(int bits, int N, int K, const uint8_t *packed, int8_t *codes)
{
    int rb = qgemm_oracle_row_bytes(bits, K);
    if (rb < 0 || N < 0 || ((N > 0 && K > 0) && (!packed || !codes)))
        return -1;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            codes[(size_t)n * K + k] = bits == 8 ? (int8_t)packed[(size_t)n * rb + k]
                                                 : (int8_t)oracle_code(bits, packed + (size_t)n * rb, k);
    return 0;
}

/* Dequantised weights W[n][k] = s[n][k/64] * q[n][k], fp64 [N][K]. */
int qgemm_oracle_dequant(int bits, int N, int K, const uint8_t *packed,
                         const uint16_t *scales, double *W)
{
    int rb = qgemm_oracle_row_bytes(bits, K);
    int G = qgemm_oracle_groups(K);
    if (rb < 0 || N < 0)
        return -1;
    for (int n = 0; n < N; ++n) {
        const uint8_t *row = packed + (size_t)n * rb;
        for (int k = 0; k < K; ++k) {
            double s = oracle_half_to_double(scales[(size_t)n * G + k / ORACLE_GROUP]);
            W[(size_t)n * K + k] = s * oracle_value(bits, row, k);
        }
    }
    return 0;
}

/*
 * Y[t][n] and A[t][n] as defined in the header comment.  Row n is dequantised
 * once into a scratch row, then dotted with every activation column in
 * ascending k.  Returns 0, or -1 on bad arguments or allocation failure.
 */
int qgemm_oracle_gemm(int bits, int N, int K, int T, const uint8_t *packed,
                      const uint16_t *scales, const uint16_t *X, double *Y, double *A)
{
    int rb = qgemm_oracle_row_bytes(bits, K);
    int G = qgemm_oracle_groups(K);
    if (rb < 0 || N < 0 || T < 0)
        return -1;
    if (N == 0 || T == 0)
        return 0;
    double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!w)
        return -1;
    for (int n = 0; n < N; ++n) {
        const uint8_t *row = packed + (size_t)n * rb;
        for (int k = 0; k < K; ++k) {
            double s = oracle_half_to_double(scales[(size_t)n * G + k / ORACLE_GROUP]);
            w[k] = s * oracle_value(bits, row, k);
        }
        for (int t = 0; t < T; ++t) {
            const uint16_t *xr = X + (size_t)t * K;
            double acc = 0.0, mag = 0.0;
            for (int k = 0; k < K; ++k) {
                double p = oracle_bf16_to_double(xr[k]) * w[k];
                acc += p;
                mag += fabs(p);
            }
            Y[(size_t)t * N + n] = acc;
            if (A)
                A[(size_t)t * N + n] = mag;
        }
    }
    free(w);
    return 0;
}

/*
 * Y[t][n] = R[t][n] + (the gemm above), A[t][n] = |R[t][n]| + (its sum of
 * |products|).  R is fp32 (the library's residual type), read exactly.
 */
int qgemm_oracle_linear_add(int bits, int N, int K, int T, const uint8_t *packed,
                            const uint16_t *scales, const uint16_t *X, const float *R,
                            double *Y, double *A)
{
    if (!R)
        return -1;
    int st = qgemm_oracle_gemm(bits, N, K, T, packed, scales, X, Y, A);
    if (st != 0)
        return st;
    for (size_t i = 0; i < (size_t)T * (size_t)N; ++i) {
        Y[i] = (double)R[i] + Y[i];
        if (A)
            A[i] = fabs((double)R[i]) + A[i];
    }
    return 0;
}

/* out[i] = silu(g[i]) * u[i] with silu(z) = z / (1 + exp(-z)), in fp64. */
int qgemm_oracle_swiglu(int n, const double *g, const double *u, double *out)
{
    if (n < 0 || (n > 0 && (!g || !u || !out)))
        return -1;
    for (int i = 0; i < n; ++i)
        out[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
    return 0;
}

/* ------------------------------------------------------------------ NVFP4 */

#define ORACLE_NVFP4_BLOCK 16

/* FP4 E2M1 -> double, from the field definitions. */
static double oracle_e2m1_to_double(int nib)
{
    int sign = (nib >> 3) & 1;
    int expo = (nib >> 1) & 3;
    int mant = nib & 1;
    double v = expo == 0 ? 0.5 * mant                        /* subnormal: m/2 */
                         : ldexp(1.0 + 0.5 * mant, expo - 1); /* (1 + m/2) * 2^(e-1) */
    return sign ? -v : v;
}

/* Unsigned E4M3 -> double; NaN for the codes outside the codec. */
static double oracle_ue4m3_to_double(uint8_t b)
{
    int expo = (b >> 3) & 0x0f;
    int mant = b & 0x07;
    if ((b & 0x80) || (expo == 15 && mant == 7))
        return NAN;
    if (expo == 0)
        return ldexp((double)mant, -9);                      /* subnormal: m/8 * 2^-6 */
    return ldexp((double)(8 + mant), expo - 10);             /* (1 + m/8) * 2^(e-7) */
}

int qgemm_oracle_nvfp4_blocks(int K)
{
    return (K + ORACLE_NVFP4_BLOCK - 1) / ORACLE_NVFP4_BLOCK;
}

/* w[n][k] of an NVFP4 matrix into the scratch row w (K values). */
static void oracle_nvfp4_row(int K, const uint8_t *codes_row, const uint8_t *bs_row, double ts, double *w)
{
    for (int k = 0; k < K; ++k) {
        int byte = codes_row[k >> 1];
        int nib = (k & 1) ? (byte >> 4) : (byte & 0x0f);
        w[k] = oracle_e2m1_to_double(nib) * oracle_ue4m3_to_double(bs_row[k / ORACLE_NVFP4_BLOCK]) * ts;
    }
}

/* Dequantised NVFP4 weights W[n][k], fp64 [N][K]. */
int qgemm_oracle_dequant_nvfp4(int N, int K, const uint8_t *codes, const uint8_t *bscales, float tscale,
                               double *W)
{
    if (N < 0 || K < 0)
        return -1;
    int rb = (K + 1) / 2, nb = qgemm_oracle_nvfp4_blocks(K);
    for (int n = 0; n < N; ++n)
        oracle_nvfp4_row(K, codes + (size_t)n * rb, bscales + (size_t)n * nb, (double)tscale, W + (size_t)n * K);
    return 0;
}

/* Y[t][n] = sum_k x[t][k] * w[n][k] (k ascending) and A[t][n] = sum |x w|
 * for an NVFP4 matrix, as qgemm_oracle_gemm does for the other codecs. */
int qgemm_oracle_gemm_nvfp4(int N, int K, int T, const uint8_t *codes, const uint8_t *bscales, float tscale,
                            const uint16_t *X, double *Y, double *A)
{
    if (N < 0 || K < 0 || T < 0)
        return -1;
    if (N == 0 || T == 0)
        return 0;
    int rb = (K + 1) / 2, nb = qgemm_oracle_nvfp4_blocks(K);
    double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!w)
        return -1;
    for (int n = 0; n < N; ++n) {
        oracle_nvfp4_row(K, codes + (size_t)n * rb, bscales + (size_t)n * nb, (double)tscale, w);
        for (int t = 0; t < T; ++t) {
            const uint16_t *xr = X + (size_t)t * K;
            double acc = 0.0, mag = 0.0;
            for (int k = 0; k < K; ++k) {
                double p = oracle_bf16_to_double(xr[k]) * w[k];
                acc += p;
                mag += fabs(p);
            }
            Y[(size_t)t * N + n] = acc;
            if (A)
                A[(size_t)t * N + n] = mag;
        }
    }
    free(w);
    return 0;
}
