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
// x is gathered through the read-only path.
template <typename T>
__device__ __forceinline__ T ld_x(const T *p) { return __ldg(p); }

// The same gather with an L2 evict-last policy, so the matrix stream (loaded
// evict-first) does not push x out of L2 between gathers.  Worth its register
// when x is small against L2, or when gathers come in bursts (shared-memory
// staged kernels).
__device__ __forceinline__ uint64_t x_policy() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ double ld_x_keep(const double *p) {
    double v;
    asm("ld.global.nc.L2::cache_hint.f64 %0, [%1], %2;" : "=d"(v) : "l"(p), "l"(x_policy()));
    return v;
}
__device__ __forceinline__ float ld_x_keep(const float *p) {
    float v;
    asm("ld.global.nc.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(x_policy()));
    return v;
}
template <bool kKeep, typename T>
__device__ __forceinline__ T gather_x(const T *p) {
    if constexpr (kKeep)
        return ld_x_keep(p);
    else
        return __ldg(p);
}

// Programmatic dependent launch (kernels launched with programmatic stream
// serialization): grid_wait() blocks until the previous kernel of the stream has
// finished and its writes are visible; allow_dependents() lets the next kernel of the
// stream be scheduled before this one ends.
__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace dev
}  // namespace spmv
