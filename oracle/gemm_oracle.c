/*
 * CPU oracle for the dense matrix multiply  C := alpha*A*B + beta*C.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the bench may load this file's library; the product path
 * never does.  It shares no source with the CUDA library.
 *
 * What it computes is the plain definition of the product:
 *   - "advanced SGEMM on NVIDIA GPUs" summary page (introduction): SGEMM
 *     computes C := alpha*A*B + beta*C;
 *   - same page, section on memory layout and PTX: row-major storage,
 *     element (r, c) of a matrix with leading dimension ld lives at
 *     ptr[r*ld + c]; A is M x K, B is K x N, C is M x N; ld may exceed the
 *     column count when the operand is a sub-matrix of a larger one;
 *   - "LeetGPU GEMM T4" page, baseline section: fp16 operands, a float
 *     accumulator, and the epilogue acc*alpha + C*beta rounded to half.
 *
 * The oracle keeps everything in double and returns the UNROUNDED result;
 * rounding to the output type is left to the tolerance check.  Inputs arrive
 * as float32 arrays: half operands are widened to float32 exactly before the
 * call, so nothing is lost.
 *
 * Conventions the pages leave open, and the reading taken here:
 *   - beta == 0: C is not read (the WMMA sections of the LeetGPU page skip the
 *     load of C when beta is zero; the SGEMM page loads C only when
 *     beta != 0).  C may then hold NaN.
 *   - alpha == 0 or K == 0: the result is beta*C; A and B are not read.
 *   - Summation order: k ascending for every element (i-k-j loop order over a
 *     double row buffer keeps that order per element).
 *
 * Rows are independent, so they are spread over OpenMP threads; the result
 * does not depend on the thread count.  Build with -ffp-contract=off so that
 * x86 and Arm hosts produce the same bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * out[r*ldo + j]    = alpha * sum_k A[i*lda+k] * B[k*ldb+j]  +  beta * C0[i*ldc+j]
 * absdot[r*ldo + j] = sum_k |A[i*lda+k]| * |B[k*ldb+j]|            (if absdot != NULL)
 *
 * where i = rows[r] when a row list is given (nrows entries), else i = r for
 * r in [0, M).  Returns 0, or -1 when a row buffer cannot be allocated.
 */
int oracle_gemm(int M, int N, int K, double alpha,
                const float* A, long lda, const float* B, long ldb,
                double beta, const float* C0, long ldc,
                double* out, double* absdot, long ldo,
                const int* rows, int nrows) {
    const int R = rows ? nrows : M;
    const int read_ab = (alpha != 0.0) && (K > 0);
    const int read_c = (beta != 0.0);
    int failed = 0;
    if (R <= 0 || N <= 0) return 0;

#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)N);
        double* acc_abs = absdot ? (double*)malloc(sizeof(double) * (size_t)N) : NULL;
        if (!acc || (absdot && !acc_abs)) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < R; ++r) {
                const long i = rows ? rows[r] : r;
                for (int j = 0; j < N; ++j) acc[j] = 0.0;
                if (acc_abs) for (int j = 0; j < N; ++j) acc_abs[j] = 0.0;
                if (read_ab) {
                    for (int k = 0; k < K; ++k) {
                        const double a = (double)A[i * lda + k];
                        const float* brow = B + (long)k * ldb;
                        for (int j = 0; j < N; ++j) acc[j] += a * (double)brow[j];
                        if (acc_abs) {
                            const double aa = fabs(a);
                            for (int j = 0; j < N; ++j) acc_abs[j] += aa * fabs((double)brow[j]);
                        }
                    }
                }
                double* o = out + (long)r * ldo;
                for (int j = 0; j < N; ++j) {
                    double v = read_ab ? alpha * acc[j] : 0.0;
                    if (read_c) v += beta * (double)C0[i * ldc + j];
                    o[j] = v;
                }
                if (acc_abs) {
                    double* oa = absdot + (long)r * ldo;
                    for (int j = 0; j < N; ++j) oa[j] = read_ab ? acc_abs[j] : 0.0;
                }
            }
        }
        free(acc);
        free(acc_abs);
    }
    return failed ? -1 : 0;
}

/*
 * Sum of all elements of an M x N row-major double matrix, in double, rows
 * then columns in ascending order ("From 306 ms to 86 ms", timing section:
 * the check is the double-precision sum of every element of C).
 */
double oracle_sum_f64(int M, int N, const double* X, long ldx) {
    double s = 0.0;
    for (int i = 0; i < M; ++i)
        for (int j = 0; j < N; ++j) s += X[(long)i * ldx + j];
    return s;
}

double oracle_sum_f32(int M, int N, const float* X, long ldx) {
    double s = 0.0;
    for (int i = 0; i < M; ++i)
        for (int j = 0; j < N; ++j) s += (double)X[(long)i * ldx + j];
    return s;
}

/*
 * Closed form of the sum of every element of alpha*A*B + beta*C0:
 *   sum_ij = alpha * sum_k (sum_i A[i][k]) * (sum_j B[k][j]) + beta * sum_ij C0[i][j].
 * Also returns in *bound the sum over k of (sum_i |A[i][k]|)(sum_j |B[k][j]|),
 * the natural scale for an error bound on the sum.  O(MK + KN) work.
 */
double oracle_checksum_closed_form(int M, int N, int K, double alpha,
                                   const float* A, long lda, const float* B, long ldb,
                                   double beta, const float* C0, long ldc, double* bound) {
    double total = 0.0, scale = 0.0;
    if (alpha != 0.0 && K > 0) {
        for (int k = 0; k < K; ++k) {
            double ca = 0.0, cb = 0.0, ca_abs = 0.0, cb_abs = 0.0;
            for (int i = 0; i < M; ++i) {
                const double a = (double)A[(long)i * lda + k];
                ca += a;
                ca_abs += fabs(a);
            }
            for (int j = 0; j < N; ++j) {
                const double b = (double)B[(long)k * ldb + j];
                cb += b;
                cb_abs += fabs(b);
            }
            total += ca * cb;
            scale += ca_abs * cb_abs;
        }
        total *= alpha;
        scale *= fabs(alpha);
    }
    if (beta != 0.0) {
        double s = 0.0, s_abs = 0.0;
        for (int i = 0; i < M; ++i)
            for (int j = 0; j < N; ++j) {
                const double c = (double)C0[(long)i * ldc + j];
                s += c;
                s_abs += fabs(c);
            }
        total += beta * s;
        scale += fabs(beta) * s_abs;
    }
    if (bound) *bound = scale;
    return total;
}

/*
 * Freivalds' product check, right-hand side:  y = alpha * A (B x) + beta * C0 x,
 * for a given vector x of length N (entries +-1 in the tests).  Also returns
 * yabs = |alpha| |A| (|B| |x|) + |beta| |C0| |x|, the scale for its error bound.
 */
void oracle_freivalds_rhs(int M, int N, int K, double alpha,
                          const float* A, long lda, const float* B, long ldb,
                          double beta, const float* C0, long ldc,
                          const double* x, double* y, double* yabs) {
    double* bx = (double*)calloc((size_t)(K > 0 ? K : 1), sizeof(double));
    double* bx_abs = (double*)calloc((size_t)(K > 0 ? K : 1), sizeof(double));
    if (!bx || !bx_abs) { free(bx); free(bx_abs); return; }
    const int read_ab = (alpha != 0.0) && (K > 0);
    if (read_ab) {
        for (int k = 0; k < K; ++k) {
            double s = 0.0, sa = 0.0;
            for (int j = 0; j < N; ++j) {
                const double b = (double)B[(long)k * ldb + j];
                s += b * x[j];
                sa += fabs(b) * fabs(x[j]);
            }
            bx[k] = s;
            bx_abs[k] = sa;
        }
    }
#pragma omp parallel for schedule(static)
    for (int i = 0; i < M; ++i) {
        double s = 0.0, sa = 0.0;
        if (read_ab) {
            for (int k = 0; k < K; ++k) {
                const double a = (double)A[(long)i * lda + k];
                s += a * bx[k];
                sa += fabs(a) * bx_abs[k];
            }
            s *= alpha;
            sa *= fabs(alpha);
        }
        if (beta != 0.0) {
            double c = 0.0, ca = 0.0;
            for (int j = 0; j < N; ++j) {
                const double v = (double)C0[(long)i * ldc + j];
                c += v * x[j];
                ca += fabs(v) * fabs(x[j]);
            }
            s += beta * c;
            sa += fabs(beta) * ca;
        }
        y[i] = s;
        yabs[i] = sa;
    }
    free(bx);
    free(bx_abs);
}
