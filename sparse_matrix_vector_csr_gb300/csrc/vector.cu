// CSR-vector apply: g lanes per row, partial sums combined with __shfl_xor_sync
// (the "subwarp" per row the scite report quotes from "Sparse Linear Algebra on
// AMD and NVIDIA GPUs"; row-length classes after the Trilinos issue on
// unpackAndCombine).
#include <cuda_runtime.h>

#include <cstdint>

#include "device_util.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

using namespace dev;

// ---------------------------------------------------------------------------
// CSR, G lanes per row
// ---------------------------------------------------------------------------
template <typename T, int G>
__global__ void __launch_bounds__(256) k_csr_vector(int64_t count, const int32_t *__restrict__ rows,
                                                   const int32_t *__restrict__ row_ptr,
                                                   const int32_t *__restrict__ col, const T *__restrict__ val,
                                                   const T *__restrict__ x, T *__restrict__ y) {
    const int64_t sub = gtid() / G;
    const int lane = threadIdx.x & (G - 1);
    if (sub >= count) return;  // the G lanes of a group leave together
    const int32_t r = rows ? __ldg(rows + sub) : static_cast<int32_t>(sub);
    const int32_t b = __ldg(row_ptr + r), e = __ldg(row_ptr + r + 1);
    T acc = T(0);
    int32_t k = b + lane;
    for (; k + G < e; k += 2 * G) {
        const int32_t c0 = ld_stream(col + k), c1 = ld_stream(col + k + G);
        const T v0 = ld_stream(val + k), v1 = ld_stream(val + k + G);
        acc = fma(v0, ld_x(x + c0), acc);
        acc = fma(v1, ld_x(x + c1), acc);
    }
    if (k < e) acc = fma(ld_stream(val + k), ld_x(x + ld_stream(col + k)), acc);
    const unsigned mask =
        (G == 32) ? 0xffffffffu : (((1u << G) - 1u) << ((threadIdx.x & 31) & ~(G - 1)));
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(mask, acc, off, G);
    if (lane == 0) y[r] = acc;
}

template <typename T>
cudaError_t csr_vector_dispatch(int g, int64_t count, const int32_t *rows, const int32_t *row_ptr,
                                const int32_t *col, const T *val, const T *x, T *y, cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    const int64_t threads = count * g;
    const unsigned grid = static_cast<unsigned>(ceil_div(threads, 256));
    switch (g) {
        case 2: k_csr_vector<T, 2><<<grid, 256, 0, s>>>(count, rows, row_ptr, col, val, x, y); break;
        case 4: k_csr_vector<T, 4><<<grid, 256, 0, s>>>(count, rows, row_ptr, col, val, x, y); break;
        case 8: k_csr_vector<T, 8><<<grid, 256, 0, s>>>(count, rows, row_ptr, col, val, x, y); break;
        case 16: k_csr_vector<T, 16><<<grid, 256, 0, s>>>(count, rows, row_ptr, col, val, x, y); break;
        case 32: k_csr_vector<T, 32><<<grid, 256, 0, s>>>(count, rows, row_ptr, col, val, x, y); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_csr_vector(int dtype, int g, int64_t count, const int32_t *rows, const int32_t *row_ptr,
                              const int32_t *col, const void *val, const void *x, void *y, cudaStream_t s) {
    if (dtype == SPMV_F64)
        return csr_vector_dispatch<double>(g, count, rows, row_ptr, col, static_cast<const double *>(val),
                                           static_cast<const double *>(x), static_cast<double *>(y), s);
    return csr_vector_dispatch<float>(g, count, rows, row_ptr, col, static_cast<const float *>(val),
                                      static_cast<const float *>(x), static_cast<float *>(y), s);
}

}  // namespace spmv
