/*
 * Multi-core CPU baseline: a plain CSR sparse matrix-vector product, y = A x, with
 * OpenMP threads over rows and each row summed in the value type, in stored order.
 * Test and measurement infrastructure, like the rest of this directory: only the
 * bench's CPU-baseline leg and the tests call it; the product never does.  It is NOT
 * the oracle (the oracle sums in long double); it is the straightforward multi-core
 * program the GPU library is set beside.
 *
 * dtype 0 = double, 1 = float.  schedule 0 = static (even row blocks), 1 = dynamic
 * (blocks of 256 rows handed out as threads free up: rows of very different lengths).
 * Returns the number of threads used.
 */
#include <omp.h>
#include <stdint.h>

int csr_omp_spmv(int64_t n, const int32_t *row_ptr, const int32_t *col_idx, const void *vals, int dtype,
                 const void *x, void *y, int schedule, int threads) {
    if (threads > 0) omp_set_num_threads(threads);
    int used = 1;
    if (dtype == 0) {
        const double *v = (const double *)vals, *xv = (const double *)x;
        double *yv = (double *)y;
        if (schedule == 1) {
#pragma omp parallel
            {
#pragma omp single
                used = omp_get_num_threads();
#pragma omp for schedule(dynamic, 256)
                for (int64_t i = 0; i < n; ++i) {
                    double s = 0.0;
                    for (int32_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) s += v[k] * xv[col_idx[k]];
                    yv[i] = s;
                }
            }
        } else {
#pragma omp parallel
            {
#pragma omp single
                used = omp_get_num_threads();
#pragma omp for schedule(static)
                for (int64_t i = 0; i < n; ++i) {
                    double s = 0.0;
                    for (int32_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) s += v[k] * xv[col_idx[k]];
                    yv[i] = s;
                }
            }
        }
    } else {
        const float *v = (const float *)vals, *xv = (const float *)x;
        float *yv = (float *)y;
        if (schedule == 1) {
#pragma omp parallel
            {
#pragma omp single
                used = omp_get_num_threads();
#pragma omp for schedule(dynamic, 256)
                for (int64_t i = 0; i < n; ++i) {
                    float s = 0.0f;
                    for (int32_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) s += v[k] * xv[col_idx[k]];
                    yv[i] = s;
                }
            }
        } else {
#pragma omp parallel
            {
#pragma omp single
                used = omp_get_num_threads();
#pragma omp for schedule(static)
                for (int64_t i = 0; i < n; ++i) {
                    float s = 0.0f;
                    for (int32_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) s += v[k] * xv[col_idx[k]];
                    yv[i] = s;
                }
            }
        }
    }
    return used;
}
