/*
 * Float64 CPU oracle for single-precision GEMM:  C = alpha * A * B + beta * C.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark load this file. The CUDA library never
 * includes, links or calls it, and it shares no code with the CUDA library.
 *
 * What it computes (the plain definition; every GPU path must land within the
 * tolerance of this result):
 *
 *   The problem statement is the one of "NVIDIA_SGEMM_PRACTICE" (section
 *   "kernel 1": mysgemm(M, N, K, alpha, A, B, beta, C) with row-major A (MxK),
 *   B (KxN), C (MxN), each output element alpha * sum_k A[m][k] * B[k][n] +
 *   beta * C[m][n]).  The reference method is the CPU triple loop
 *   matrixMulCPU of "matmul_opt.cu" (cnblogs matmul-opt demo), which
 *   accumulates one output element over k in order.  Changes to that loop:
 *     - leading dimensions lda/ldb/ldc (the packed case is lda=K, ldb=ldc=N);
 *     - float64 accumulation: each product of two float32 values is exact in
 *       float64 (24 + 24 significant bits <= 53), so only the running sum
 *       rounds;
 *     - the alpha/beta epilogue of the problem statement;
 *     - a second accumulator, sum_k |A[m][k] * B[k][n]|, from which the
 *       per-element error scale |alpha| * sum_k |a*b| + |beta * c| is formed.
 *
 *   Readings where the pages are silent:
 *     - beta == 0: C is not read (BLAS convention), so NaN in the old C does
 *       not reach the result;
 *     - alpha == 0 or K == 0: A and B are not read; the result is beta * C.
 *
 * The loop order is m, k, n with one float64 accumulator per (m, n): for each
 * output element the products are still added in increasing k, exactly as in
 * the triple loop; the order only makes the inner loop walk memory forward.
 * OpenMP splits the work over output rows; rows never share an accumulator.
 *
 * Parity pins for this file live in tests/test_oracle_pins.py.
 *
 * Build: gcc -O3 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math).
 * ORACLE_PLANT selects a deliberately wrong variant; it exists only so the
 * tests can show that each pin catches a plausible mistake.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

/* Compute selected output rows.
 *
 *   rows == NULL : rows 0 .. nrows-1
 *   rows != NULL : rows[r] for r < nrows (each in [0, M))
 *   ref   : nrows x N, row-major, float64 results
 *   scale : nrows x N, |alpha| * sum_k |A[m][k] B[k][n]| + |beta C[m][n]|
 *   nthreads <= 0 : OpenMP default
 *
 * Returns 0, or a negative argument index (1-based) on invalid input.
 */
int oracle_sgemm_rows(int M, int N, int K, double alpha,
                      const float *A, long long lda,
                      const float *B, long long ldb,
                      double beta, const float *C, long long ldc,
                      const int *rows, int nrows,
                      double *ref, double *scale, int nthreads)
{
    if (M < 0) return -1;
    if (N < 0) return -2;
    if (K < 0) return -3;
    if (nrows < 0) return -14;
    if (nrows == 0 || N == 0) return 0;
    if (ref == NULL) return -15;
    if (scale == NULL) return -16;
    const int use_ab = (alpha != 0.0 && K > 0);
    if (use_ab && (A == NULL || B == NULL)) return -5;
    if (beta != 0.0 && C == NULL) return -10;
    if (rows != NULL) {
        for (int r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= M) return -13;
    } else if (nrows > M) {
        return -14;
    }
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    (void)nthreads;
#endif

#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int r = 0; r < nrows; ++r) {
        const long long m = rows ? rows[r] : r;
        double *s = ref + (long long)r * N;
        double *t = scale + (long long)r * N;
        for (int n = 0; n < N; ++n) { s[n] = 0.0; t[n] = 0.0; }
        if (use_ab) {
            for (int k = 0; k < K; ++k) {
#if ORACLE_PLANT == 1
                /* planted: A read transposed (A[k][m] instead of A[m][k]),
                 * indices wrapped so the read stays inside A */
                const double a = (double)A[(long long)(k % M) * lda + (m % K)];
#elif ORACLE_PLANT == 3
                /* planted: last k dropped */
                if (k == K - 1) break;
                const double a = (double)A[m * lda + k];
#else
                const double a = (double)A[m * lda + k];
#endif
                const float *brow = B + (long long)k * ldb;
                for (int n = 0; n < N; ++n) {
                    const double p = a * (double)brow[n];
                    s[n] += p;
                    t[n] += fabs(p);
                }
            }
        }
        const float *crow = (beta != 0.0) ? C + m * ldc : NULL;
        for (int n = 0; n < N; ++n) {
            const double ab = use_ab ? alpha * s[n] : 0.0;
#if ORACLE_PLANT == 2
            /* planted: beta term dropped */
            const double bc = 0.0 * (crow ? (double)crow[n] : 0.0);
#elif ORACLE_PLANT == 4
            /* planted: alpha and beta swapped */
            const double bc = crow ? alpha * (double)crow[n] : 0.0;
            s[n] = use_ab ? beta * s[n] + bc : bc;
            t[n] = fabs(beta) * t[n] + fabs(bc);
            continue;
#else
            const double bc = crow ? beta * (double)crow[n] : 0.0;
#endif
            s[n] = ab + bc;
            t[n] = fabs(alpha) * t[n] + fabs(bc);
        }
    }
    return 0;
}

/* Direct 2-D convolution (the deep-learning "convolution", i.e. a
 * cross-correlation: the filter is not flipped), the operation whose im2col
 * lowering gives the skinny GEMM shapes of "UNIVERSAL_SGEMM_CUDA" (its shape
 * list, e.g. M = 32 filters, K = 27 = 3 channels x 3 x 3, N = 32 images x
 * 224 x 224 output pixels).  The pages give the GEMM shapes only; this is the
 * plain definition of the layer they come from:
 *
 *   X: NCHW input, nb x C x H x W;  Wt: OIHW filter, F x C x KH x KW;
 *   Y: NCHW output, nb x F x OH x OW with
 *      OH = (H + 2 ph - dh (KH - 1) - 1) / sh + 1 (and likewise OW);
 *   Y[b][f][oh][ow] = alpha * sum_{c, kh, kw} Wt[f][c][kh][kw] *
 *                     X[b][c][oh sh + kh dh - ph][ow sw + kw dw - pw]
 *                     + beta * Y[b][f][oh][ow],
 *   input positions outside the image reading as zero.
 *
 * Each output element is summed in float64 over c, then kh, then kw (the
 * order of the im2col row index k = (c KH + kh) KW + kw), with the same
 * |product| sum as the GEMM oracle for the error scale.  beta == 0: Y is not
 * read.  ref / scale: nb x F x OH x OW, float64.  OpenMP over (b, f).
 *
 * Returns 0, or a negative argument index (1-based) on invalid input.
 */
int oracle_conv2d_nchw(int nb, int C, int H, int W, int F, int KH, int KW,
                       int sh, int sw, int ph, int pw, int dh, int dw,
                       double alpha, const float *X, const float *Wt,
                       double beta, const float *Y,
                       double *ref, double *scale, int nthreads)
{
    if (nb < 0) return -1;
    if (C < 0) return -2;
    if (H < 0) return -3;
    if (W < 0) return -4;
    if (F < 0) return -5;
    if (KH < 1) return -6;
    if (KW < 1) return -7;
    if (sh < 1) return -8;
    if (sw < 1) return -9;
    if (ph < 0) return -10;
    if (pw < 0) return -11;
    if (dh < 1) return -12;
    if (dw < 1) return -13;
    const long long OHn = (long long)H + 2LL * ph - (long long)dh * (KH - 1) - 1;
    const long long OWn = (long long)W + 2LL * pw - (long long)dw * (KW - 1) - 1;
    if (OHn < 0 || OWn < 0) return -3;
    const int OH = (int)(OHn / sh + 1), OW = (int)(OWn / sw + 1);
    if (nb == 0 || F == 0) return 0;
    const int use_ab = (alpha != 0.0 && C > 0);
    if (use_ab && X == NULL) return -15;
    if (use_ab && Wt == NULL) return -16;
    if (beta != 0.0 && Y == NULL) return -18;
    if (ref == NULL) return -19;
    if (scale == NULL) return -20;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    (void)nthreads;
#endif
    const long long plane = (long long)OH * OW;

#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long long bf = 0; bf < (long long)nb * F; ++bf) {
        const long long b = bf / F, f = bf % F;
        double *s = ref + bf * plane;
        double *t = scale + bf * plane;
        for (long long i = 0; i < plane; ++i) { s[i] = 0.0; t[i] = 0.0; }
        if (use_ab) {
            for (int c = 0; c < C; ++c) {
                const float *xc = X + (b * C + c) * (long long)H * W;
                for (int kh = 0; kh < KH; ++kh) {
                    for (int kw = 0; kw < KW; ++kw) {
#if ORACLE_PLANT == 5
                        /* planted: filter flipped (true convolution) */
                        const double w = (double)Wt[((f * C + c) * KH + (KH - 1 - kh)) * KW + (KW - 1 - kw)];
#else
                        const double w = (double)Wt[((f * C + c) * KH + kh) * KW + kw];
#endif
                        for (int oh = 0; oh < OH; ++oh) {
#if ORACLE_PLANT == 6
                            /* planted: padding applied on one side only */
                            const long long ih = (long long)oh * sh + (long long)kh * dh;
#elif ORACLE_PLANT == 7
                            /* planted: dilation ignored */
                            const long long ih = (long long)oh * sh + kh - ph;
#else
                            const long long ih = (long long)oh * sh + (long long)kh * dh - ph;
#endif
                            if (ih < 0 || ih >= H) continue;
                            for (int ow = 0; ow < OW; ++ow) {
#if ORACLE_PLANT == 7
                                const long long iw = (long long)ow * sw + kw - pw;
#else
                                const long long iw = (long long)ow * sw + (long long)kw * dw - pw;
#endif
                                if (iw < 0 || iw >= W) continue;
                                const double p = w * (double)xc[ih * W + iw];
                                s[(long long)oh * OW + ow] += p;
                                t[(long long)oh * OW + ow] += fabs(p);
                            }
                        }
                    }
                }
            }
        }
        const float *yo = (beta != 0.0) ? Y + bf * plane : NULL;
        for (long long i = 0; i < plane; ++i) {
            const double ab = use_ab ? alpha * s[i] : 0.0;
            const double bc = yo ? beta * (double)yo[i] : 0.0;
            s[i] = ab + bc;
            t[i] = fabs(alpha) * t[i] + fabs(bc);
        }
    }
    return 0;
}

/* Number of threads OpenMP would use by default (for reporting). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
