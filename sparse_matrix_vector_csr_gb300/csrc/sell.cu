// Sliced-ELL apply (SELL-C-sigma, ELLPACK-R, HYB's ELL part): one thread per sorted
// row position; each thread stops at its own row's length, so padding is never
// loaded or multiplied (ELLPACK-R of the GPGPU spMVM paper, arXiv 1112.5588,
// ELLPACK-R section; the "early stopping" quoted in the scite report
// "Load-balancing Sparse Matrix Vector Product Kernels on GPUs").
#include <cuda_runtime.h>

#include <cstdint>

#include "device_util.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

using namespace dev;

// ---------------------------------------------------------------------------
// sliced layout
// ---------------------------------------------------------------------------
// Entries of a row are processed U at a time: the U column indices and values
// (predicated on the row length, so padding is never touched) are loaded first,
// then the U gathers of x, then U fused multiply-adds.  This keeps 2U independent
// streaming loads in flight per thread before the dependent gathers.  U = 4 for
// fp64 and 8 for fp32 (4 with a runtime stride) fills the load queue at 32
// registers per thread, which keeps all 64 warps of an SM resident.
template <typename T, int CS>
struct SellChunk {
    // runtime-stride addressing needs a 64-bit address per load: keep 4 in flight
    static constexpr int U = (sizeof(T) == 8 || CS == 0) ? 4 : 8;
};

// CS > 0: SELL with a compile-time slice height CS (stride = CS).
// CS == 0: runtime addressing (slice p >> log2C, row p & cmask, stride `stride`),
//          used by the single-slice ELLPACK-R / HYB-ELL layout and other slice heights.
template <typename T, int CS>
__global__ void __launch_bounds__(kSellBlock, CS > 0 ? 8 : 6) k_sell(int64_t n_pos, int log2C, uint32_t cmask, int64_t stride,
                                                        const int64_t *__restrict__ slice_ptr,
                                                        const int32_t *__restrict__ len,
                                                        const int32_t *__restrict__ perm,
                                                        const int32_t *__restrict__ col, const T *__restrict__ val,
                                                        const T *__restrict__ x, T *__restrict__ y, int64_t n) {
    constexpr int U = SellChunk<T, CS>::U;
    const int64_t p = gtid();
    if (p >= n_pos) return;
    const int w = __ldg(len + p);
    const uint64_t up = static_cast<uint64_t>(p);
    const int64_t slot = CS > 0 ? __ldg(slice_ptr + (up / CS)) + static_cast<int64_t>(up % CS)
                                : __ldg(slice_ptr + (p >> log2C)) + static_cast<int64_t>(p & cmask);
    const int32_t *cp = col + slot;
    const T *vp = val + slot;
    T acc = T(0);
    if constexpr (CS > 0) {
        for (int j = 0; j < w; j += U) {
            int32_t c[U];
            T a[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool on = j + u < w;
                c[u] = on ? ld_stream(cp + u * CS) : 0;
                a[u] = on ? ld_stream(vp + u * CS) : T(0);
            }
            T xv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) xv[u] = (j + u < w) ? ld_x(x + c[u]) : T(0);
#pragma unroll
            for (int u = 0; u < U; ++u) acc = fma(a[u], xv[u], acc);  // inactive slots add +0 * +0
            cp += U * CS;
            vp += U * CS;
        }
    } else {
        // the leading dimension of an ELL part is below 2^31: 32-bit offsets inside a chunk
        const int ld = static_cast<int>(stride);
        for (int j = 0; j < w; j += U) {
            int32_t c[U];
            T a[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool on = j + u < w;
                c[u] = on ? ld_stream(cp + u * ld) : 0;
                a[u] = on ? ld_stream(vp + u * ld) : T(0);
            }
            T xv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) xv[u] = (j + u < w) ? ld_x(x + c[u]) : T(0);
#pragma unroll
            for (int u = 0; u < U; ++u) acc = fma(a[u], xv[u], acc);
            cp += static_cast<int64_t>(U) * ld;
            vp += static_cast<int64_t>(U) * ld;
        }
    }
    const int64_t r = perm ? static_cast<int64_t>(__ldg(perm + p)) : p;
    if (r >= 0 && r < n) y[r] = acc;
}

}  // namespace

template <typename T>
cudaError_t sell_dispatch(const Sliced &sl, int64_t n, const T *x, T *y, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>(ceil_div(sl.n_pos, kSellBlock));
    const T *val = static_cast<const T *>(sl.val);
    const bool sliced = sl.log2C < 31;
    if (sliced && sl.C == 32)
        k_sell<T, 32><<<grid, kSellBlock, 0, s>>>(sl.n_pos, sl.log2C, sl.cmask, sl.stride, sl.slice_ptr, sl.len,
                                                  sl.perm, sl.col, val, x, y, n);
    else if (sliced && sl.C == 64)
        k_sell<T, 64><<<grid, kSellBlock, 0, s>>>(sl.n_pos, sl.log2C, sl.cmask, sl.stride, sl.slice_ptr, sl.len,
                                                  sl.perm, sl.col, val, x, y, n);
    else
        k_sell<T, 0><<<grid, kSellBlock, 0, s>>>(sl.n_pos, sl.log2C, sl.cmask, sl.stride, sl.slice_ptr, sl.len,
                                                 sl.perm, sl.col, val, x, y, n);
    return cudaGetLastError();
}

cudaError_t launch_sell_apply(int dtype, const Sliced &sl, int64_t n, const void *x, void *y, cudaStream_t s) {
    if (!sl.present || sl.n_pos <= 0) return cudaSuccess;
    if (dtype == SPMV_F64)
        return sell_dispatch<double>(sl, n, static_cast<const double *>(x), static_cast<double *>(y), s);
    return sell_dispatch<float>(sl, n, static_cast<const float *>(x), static_cast<float *>(y), s);
}

}  // namespace spmv
