// Vector helpers of the scaled and multi-vector applies when a format has no fused
// epilogue: copy one column of a row-major block into a contiguous vector, and
// combine a product into a (possibly strided) output column with alpha and beta.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_util.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

using namespace dev;

template <typename T>
__global__ void k_gather_col(int64_t n, const T *__restrict__ X, int64_t ldx, T *__restrict__ out) {
    for (int64_t i = gtid(); i < n; i += static_cast<int64_t>(gridDim.x) * blockDim.x) out[i] = X[i * ldx];
}

// Y[i * ldy] = alpha * t[i] + beta * Y[i * ldy]; Y is not read when beta == 0.
template <typename T>
__global__ void k_axpby_col(int64_t n, double alpha, const T *__restrict__ t, double beta, T *__restrict__ Y,
                            int64_t ldy) {
    const T a = static_cast<T>(alpha), b = static_cast<T>(beta);
    for (int64_t i = gtid(); i < n; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        T *yp = Y + i * ldy;
        *yp = beta != 0.0 ? fma(a, t[i], b * *yp) : a * t[i];
    }
}

unsigned grid_of(int64_t n) {
    int64_t g = ceil_div(n, 256);
    if (g < 1) g = 1;
    if (g > 65536) g = 65536;
    return static_cast<unsigned>(g);
}

}  // namespace

cudaError_t launch_gather_col(int dtype, int64_t n, const void *X, int64_t ldx, void *out, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    if (dtype == SPMV_F64)
        k_gather_col<double><<<grid_of(n), 256, 0, s>>>(n, static_cast<const double *>(X), ldx,
                                                        static_cast<double *>(out));
    else
        k_gather_col<float><<<grid_of(n), 256, 0, s>>>(n, static_cast<const float *>(X), ldx,
                                                       static_cast<float *>(out));
    return cudaGetLastError();
}

cudaError_t launch_axpby_col(int dtype, int64_t n, double alpha, const void *t, double beta, void *Y, int64_t ldy,
                             cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    if (dtype == SPMV_F64)
        k_axpby_col<double><<<grid_of(n), 256, 0, s>>>(n, alpha, static_cast<const double *>(t), beta,
                                                       static_cast<double *>(Y), ldy);
    else
        k_axpby_col<float><<<grid_of(n), 256, 0, s>>>(n, alpha, static_cast<const float *>(t), beta,
                                                      static_cast<float *>(Y), ldy);
    return cudaGetLastError();
}

}  // namespace spmv
