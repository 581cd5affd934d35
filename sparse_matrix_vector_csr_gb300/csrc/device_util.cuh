// Device helpers shared by the apply kernels (each translation unit gets its own copy).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace spmv {
namespace dev {

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ int64_t gtid() {
    return static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
}

// Streaming loads for the matrix (read once per apply): evict-first in L1/L2.
__device__ __forceinline__ int32_t ld_stream(const int32_t *p) { return __ldcs(p); }
__device__ __forceinline__ double ld_stream(const double *p) { return __ldcs(p); }
__device__ __forceinline__ float ld_stream(const float *p) { return __ldcs(p); }
// x is gathered through the read-only path and kept in cache.
template <typename T>
__device__ __forceinline__ T ld_x(const T *p) { return __ldg(p); }

}  // namespace dev
}  // namespace spmv
