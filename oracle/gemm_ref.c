/*
 * Oracle: plain FP64 reference of the tiled dense GEMM and its fused epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code with the CUDA path.
 *
 * What it computes (the plain definition the tiled method reaches up to the
 * rounding order of its FP32 accumulator):
 *
 *   z[i][j] = act( alpha * sA * sB * sum_{k=0}^{K-1} dec(A[i][k]) * dec(B[j][k]) + bias[j] )
 *
 *   - C = A x B with one output tile C[m,n] per CTA task ("Deep dive into
 *     DeepGEMM", kumaling.xyz, panel "CTA <-> output tile: mapping first, then
 *     assignment", which reduces the GEMM to C = A x B).
 *   - A tile is the sum over its k-tiles ("H100 . Stream-K scheduling",
 *     runguoli.com course notes Lesson 8.1, section 1: C_tile = sum over k-tiles
 *     of A_tile_k . B_tile_k).  The oracle sums every k in ascending order in
 *     FP64; no k-tiling is applied here.
 *   - The epilogue order is Z = alpha*Acc, then + per-column bias, then the
 *     activation, then the output cast ("H100 . Kernel Design", Lesson 8,
 *     section 12.2, steps 2-4 and 7).  The FP8 tensor-wise scales sA, sB fold
 *     into alpha (same lesson, section 12.1 item 9 "scaling fusion"; WGMMA
 *     Part 2, section 11 "tensor-wise" scaling).
 *   - dec() is the exact value of a BF16 or FP8-e4m3 code (WGMMA Part 2,
 *     sections 9-10: e4m3 maximum 448, no infinity encoding).
 *
 * B is stored N x K (K contiguous), so the product is sum_k A[i][k] * B[j][k];
 * C is row-major M x N.  All arithmetic is IEEE FP64 with FMA contraction
 * disabled at compile time (-ffp-contract=off), so every product is rounded
 * and then added.  oracle_gemm_rows() only chooses which rows to compute (so a
 * large problem can be checked on a row sample); every element is the same
 * ascending-k loop.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_BF16 = 0, ORACLE_E4M3 = 1, ORACLE_E5M2 = 2 };

/* BF16: 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits.  The upper
 * half of an IEEE binary32. */
double oracle_decode_bf16(uint16_t code) {
    int sign = (code >> 15) & 1;
    int e = (code >> 7) & 0xFF;
    int m = code & 0x7F;
    double v;
    if (e == 0xFF) {
        v = (m == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)m, -126 - 7); /* subnormal: 0.m * 2^-126 */
    } else {
        v = ldexp(1.0 + (double)m / 128.0, e - 127);
    }
    return sign ? -v : v;
}

/* FP8 e4m3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits, no infinities, S.1111.111 is NaN, largest finite 1.75 * 2^8 = 448. */
double oracle_decode_e4m3(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) {
        v = NAN;
    } else if (e == 0) {
        v = ldexp((double)m, -6 - 3); /* subnormal: 0.m * 2^-6 */
    } else {
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    }
    return sign ? -v : v;
}

/* FP8 e5m2: 1 sign bit, 5 exponent bits (bias 15), 2 mantissa bits ("H100 .
 * WGMMA Part 2", section 9, and the Hopper summary of "H100 . Kernel Design":
 * wider range, less precision than e4m3).  It keeps the IEEE special values:
 * exponent field 31 is infinity (mantissa 0) or NaN; largest finite
 * 1.75 * 2^15 = 57344; subnormals 0.m * 2^-14. */
double oracle_decode_e5m2(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 2) & 0x1F;
    int m = code & 0x3;
    double v;
    if (e == 0x1F) {
        v = (m == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)m, -14 - 2);
    } else {
        v = ldexp(1.0 + (double)m / 4.0, e - 15);
    }
    return sign ? -v : v;
}

static double decode(int dtype, const void *base, int64_t idx) {
    if (dtype == ORACLE_BF16) return oracle_decode_bf16(((const uint16_t *)base)[idx]);
    if (dtype == ORACLE_E5M2) return oracle_decode_e5m2(((const uint8_t *)base)[idx]);
    return oracle_decode_e4m3(((const uint8_t *)base)[idx]);
}

void oracle_decode_array(int dtype, const void *codes, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = decode(dtype, codes, i);
}

/* FP64 -> BF16 bit pattern, round to nearest, ties to even, computed from the
 * value itself (no intermediate FP32 rounding).  BF16 values in the binade
 * [2^b, 2^(b+1)) are spaced 2^(b-7); below 2^-126 the spacing stays 2^-133
 * (subnormals).  A result that rounds to 2^128 or beyond is infinity. */
uint16_t oracle_round_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                       /* a = f * 2^e with f in [0.5, 1) */
    int b = e - 1;                      /* a in [2^b, 2^(b+1)) */
    if (b < -126) b = -126;
    double step = ldexp(1.0, b - 7);
    double r = nearbyint(a / step) * step;  /* ties to even (default mode) */
    if (r == 0.0) return sign;              /* below half the smallest subnormal: signed zero */
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
    frexp(r, &e);
    b = e - 1;
    if (b < -126) return sign | (uint16_t)(r / ldexp(1.0, -133));
    return sign | (uint16_t)(((b + 127) << 7) | (int)((r / ldexp(1.0, b) - 1.0) * 128.0));
}

/*
 * Rows rows[0..nrows) of the GEMM plus epilogue, with B already decoded: Bd holds
 * the exact FP64 values of B (N x K row-major), A holds dtype_a codes.  z_out and
 * absdot_out are nrows x N row-major (FP64).  absdot[r][j] = sum_k |alpha sA sB|
 * |a_ik| |b_jk|, the scale the error bound is quoted against.  rows == NULL means
 * rows 0..nrows-1.  Every element is the same ascending-k loop whichever entry
 * is called; this one lets a caller that computes many row samples of one B
 * decode it once.
 */
void oracle_gemm_rows_bdec(int64_t N, int64_t K, int dtype_a, const void *A, const double *Bd,
                           const int64_t *rows, int64_t nrows,
                           double alpha, double sA, double sB,
                           const float *bias, int relu,
                           double *z_out, double *absdot_out) {
    const double scale = alpha * sA * sB;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        double *Ad = (double *)malloc(sizeof(double) * (size_t)K);
        for (int64_t k = 0; k < K; ++k) Ad[k] = decode(dtype_a, A, i * K + k);
        for (int64_t j = 0; j < N; ++j) {
            const double *b = Bd + j * K;
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; ++k) {       /* ascending k */
                double p = Ad[k] * b[k];
                acc = acc + p;
                aacc = aacc + fabs(p);
            }
            double z = scale * acc;                  /* Z = alpha * Acc */
            if (bias) z = z + (double)bias[j];       /* + per-column bias */
            if (relu && z < 0.0) z = 0.0;            /* activation */
            z_out[r * N + j] = z;
            if (absdot_out) absdot_out[r * N + j] = fabs(scale) * aacc;
        }
        free(Ad);
    }
}

/*
 * The same with B given as dtype_b codes: B is decoded exactly (N x K doubles)
 * and the rows are computed as above.  A holds dtype_a codes (the two FP8
 * formats may be mixed).
 */
void oracle_gemm_rows(int64_t M, int64_t N, int64_t K, int dtype_a, int dtype_b,
                      const void *A, const void *B,
                      const int64_t *rows, int64_t nrows,
                      double alpha, double sA, double sB,
                      const float *bias, int relu,
                      double *z_out, double *absdot_out) {
    (void)M;
    double *Bd = (double *)malloc(sizeof(double) * (size_t)N * (size_t)K);
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k) Bd[j * K + k] = decode(dtype_b, B, j * K + k);
    oracle_gemm_rows_bdec(N, K, dtype_a, A, Bd, rows, nrows, alpha, sA, sB, bias, relu, z_out, absdot_out);
    free(Bd);
}
