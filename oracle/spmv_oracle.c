/*
 * Oracle for y = A x with A in compressed sparse row (CSR) form.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file; only the tests, the smoke check and the bench's CPU-baseline leg do.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes is the plain definition of the sparse matrix-vector product
 * that every page states the problem with ("Sparse matrix-vector multiplication
 * (spMVM) ..." in the GPGPU spMVM paper, arXiv 1112.5588, introduction; the CSR
 * arrays Ap/Aj/Ax of "Development of Krylov and AMG linear solvers for large-scale
 * sparse matrices on GPUs", matrix-format section, Figure 3):
 *
 *     y_i = sum_{k = row_ptr[i]}^{row_ptr[i+1]-1} vals[k] * x[col_idx[k]]
 *
 * evaluated single-threaded in long double, starting from +0 and adding the
 * terms in stored order.  Inputs are converted exactly to long double.  The
 * result is reported three ways: the long double value split into two doubles
 * (hi + lo), the value rounded once to the matrix value type, and the scale
 * sum_k |vals[k] * x[col_idx[k]]| that the per-row tolerance is relative to.
 *
 * ORACLE_MUTATION (compile-time, tests only) plants one deliberate mistake so a
 * test can show that the pins catch it; the shipped oracle is built without it.
 */
#include <float.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

/* Number of mantissa bits of long double on this host (64 on x86-64, 113 on aarch64). */
int oracle_ldbl_mant_dig(void) { return LDBL_MANT_DIG; }

static long double load_value(const void *p, int dtype, int64_t k) {
    if (dtype == 0) return (long double)((const double *)p)[k];
    return (long double)((const float *)p)[k];
}

/*
 * Rows to evaluate: rows[t] for t < nrows, or every row 0..n-1 when rows == NULL
 * (then nrows must equal n).  Outputs are indexed by t.
 *
 * dtype: 0 = float64 values and vectors, 1 = float32.
 * y_round is a double* (dtype 0) or float* (dtype 1).
 * Returns 0, or -1 when an index is out of range or row_ptr is not monotone.
 */
int oracle_spmv_csr(int64_t n, const int32_t *row_ptr, const int32_t *col_idx, const void *vals,
                    int dtype, const void *x, const int64_t *rows, int64_t nrows, double *y_hi,
                    double *y_lo, double *abs_sum, void *y_round) {
    if (rows == NULL && nrows != n) return -1;
    for (int64_t t = 0; t < nrows; ++t) {
        int64_t i = rows ? rows[t] : t;
        if (i < 0 || i >= n) return -1;
        int64_t begin = row_ptr[i], end = row_ptr[i + 1];
        if (end < begin) return -1;
        long double acc = +0.0L;
        long double scale = +0.0L;
        for (int64_t k = begin; k < end; ++k) {
            int64_t j = col_idx[k];
            if (j < 0 || j >= n) return -1;
#if ORACLE_MUTATION == 1 /* transposed operand: uses x[i] instead of x[j] */
            long double term = load_value(vals, dtype, k) * load_value(x, dtype, i);
#elif ORACLE_MUTATION == 2 /* wrong sign on the product */
            long double term = -load_value(vals, dtype, k) * load_value(x, dtype, j);
#else
            long double term = load_value(vals, dtype, k) * load_value(x, dtype, j);
#endif
#if ORACLE_MUTATION == 3 /* dropped term: skips the last entry of every row */
            if (k == end - 1) continue;
#endif
#if ORACLE_MUTATION == 4 /* off-by-one index into the column array */
            if (k + 1 < end) term = load_value(vals, dtype, k) * load_value(x, dtype, col_idx[k + 1]);
#endif
            acc += term;
            scale += fabsl(term);
        }
        double hi = (double)acc;
        y_hi[t] = hi;
        y_lo[t] = (double)(acc - (long double)hi);
        abs_sum[t] = (double)scale;
        if (dtype == 0)
            ((double *)y_round)[t] = (double)acc;
        else
            ((float *)y_round)[t] = (float)acc;
    }
    return 0;
}
