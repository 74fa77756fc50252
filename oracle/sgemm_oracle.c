/*
 * FP64 CPU oracle for single-precision GEMM  C = alpha * A * B + beta * C0.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Definition followed (hatrix.site "GEMM优化原理", section 问题定义, first
 * equation; restated by aerisun.top "GPU 访存与计算优化", section "Naive GEMM
 * 的重复读取"):  C_ij = sum_{t=0}^{k-1} A_it * B_tj, with A m x k, B k x n,
 * C m x n.  The alpha/beta scaling is the usual BLAS one:
 *     r_ij = alpha * acc_ij + beta * C0_ij,   C0 not read when beta == 0,
 *     A and B not read when alpha == 0 or k == 0.
 * Storage is row-major with leading dimensions (aerisun.top, section
 * "Shared Tiling 与 block 内复用", which loads along the row-major layout):
 * A(i,t) = A[i*lda + t], B(t,j) = B[t*ldb + j], C(i,j) = C[i*ldc + j].
 *
 * Every product and every partial sum is formed in FP64 and summed in
 * increasing t for each (i, j) (the loop order i-t-j keeps that order per
 * output).  Alongside r the oracle returns the error scale
 * E_ij = sum_t |A_it| * |B_tj|, which the FP32 tolerance is stated in.
 *
 * Also the array sum s = sum_i x_i of aerisun.top "GPU 访存与计算优化"
 * (section "Reduce 的分层归约", first formula), in FP64 in increasing i, with
 * the scale sum_i |x_i| its FP32 error bound is stated in.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (contraction is
 * off so x86 and Arm builds give the same FP64 bits).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of threads OpenMP will use for the next parallel region. */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full oracle.  R and E are m x n row-major FP64 outputs (leading dimension
 * n); Rf (may be NULL) receives R rounded to FP32 (round to nearest even).
 * rows [row_begin, row_end) only are computed (the CPU-baseline leg times a
 * bounded slab of rows); pass 0, m for the whole result.
 * nthreads <= 0 uses the OpenMP default.
 */
void oracle_sgemm_f64(int64_t m, int64_t n, int64_t k, double alpha,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      double beta, const float *C0, int64_t ldc,
                      double *R, double *E, float *Rf,
                      int64_t row_begin, int64_t row_end, int nthreads) {
    (void)m;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const int use_ab = (alpha != 0.0) && (k > 0);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = row_begin; i < row_end; ++i) {
        double *r = R + (i - row_begin) * n;
        double *e = E + (i - row_begin) * n;
        for (int64_t j = 0; j < n; ++j) { r[j] = 0.0; e[j] = 0.0; }
        if (use_ab) {
            for (int64_t t = 0; t < k; ++t) {
                const double a = (double)A[i * lda + t];
                const double abs_a = fabs(a);
                const float *brow = B + t * ldb;
                for (int64_t j = 0; j < n; ++j) {
                    const double b = (double)brow[j];
                    r[j] += a * b;
                    e[j] += abs_a * fabs(b);
                }
            }
        }
        for (int64_t j = 0; j < n; ++j) {
            double v = use_ab ? alpha * r[j] : 0.0;
            if (beta != 0.0) v += beta * (double)C0[i * ldc + j];
            r[j] = v;
            if (Rf) Rf[(i - row_begin) * n + j] = (float)v;
        }
    }
}

/*
 * Sampled oracle: the same definition evaluated only at the `count`
 * coordinates (rows[s], cols[s]), k products each, summed in increasing t.
 */
void oracle_sgemm_f64_sampled(int64_t k, double alpha,
                              const float *A, int64_t lda, const float *B, int64_t ldb,
                              double beta, const float *C0, int64_t ldc,
                              int64_t count, const int64_t *rows, const int64_t *cols,
                              double *R, double *E, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const int use_ab = (alpha != 0.0) && (k > 0);
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < count; ++s) {
        const int64_t i = rows[s], j = cols[s];
        double acc = 0.0, err = 0.0;
        if (use_ab) {
            for (int64_t t = 0; t < k; ++t) {
                const double a = (double)A[i * lda + t];
                const double b = (double)B[t * ldb + j];
                acc += a * b;
                err += fabs(a) * fabs(b);
            }
        }
        double v = use_ab ? alpha * acc : 0.0;
        if (beta != 0.0) v += beta * (double)C0[i * ldc + j];
        R[s] = v;
        E[s] = err;
    }
}

/* s = sum_{i<n} x_i and a = sum_{i<n} |x_i|, FP64, increasing i. */
void oracle_sum_f64(const float *x, int64_t n, double *s, double *a) {
    double acc = 0.0, abs_acc = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double v = (double)x[i];
        acc += v;
        abs_acc += fabs(v);
    }
    *s = acc;
    *a = abs_acc;
}
