// Sliced-ELL apply with G threads per row (G = 2 .. 32): the multi-thread-per-row
// ELL variants for wide slices ("Load-balancing Sparse Matrix Vector Product Kernels
// on GPUs", ELL kernel section).
//
// * Row-grouped (mode 0; the scheme that paper takes from its reference [2]): the
//   usual column-major slots, G adjacent threads per row taking entries j = sub,
//   sub + G, ..., each stopping at the row's length.  A warp reads G runs of 32 / G
//   consecutive slots per step.
// * Interleaved (mode 1): the same thread mapping on a rearranged layout whose slots
//   hold a row's entries in groups of G side by side (slot_of()), so the G threads of
//   a row read G adjacent values and a warp reads 32 consecutive ones.
// * Column-grouped (mode 2; the AMD rearrangement of that paper): column-major slots,
//   a warp per 32 consecutive rows and residue class of entries, G warps per row set,
//   partial sums combined in shared memory (k_sellcg).
//
// Each thread keeps U entries of its share in flight (predicated on the row length, so
// padding is never read), the G partial sums meet in a shuffle tree, and the group's
// first thread writes y through the same epilogue as the one-thread-per-row kernel.
// Launched with programmatic dependent launch: matrix data loads before grid_wait(),
// x and y after it.  Rows marked long (len = -1) are left to the row-split pass.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_util.cuh"
#include "sell_common.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

using namespace dev;
using namespace sellk;

template <typename T, int G, bool IL, bool K>
__global__ void __launch_bounds__(kSellBlock, 6)
    k_sellg(SellArgs a, const T *__restrict__ val, const T *__restrict__ x, T *__restrict__ y, Epi ep) {
    constexpr int U = 4;
    constexpr int LOG2G = G == 2 ? 1 : G == 4 ? 2 : G == 8 ? 3 : G == 16 ? 4 : 5;
    allow_dependents();
    const int64_t t = gtid();
    const int64_t p = t >> LOG2G;
    const int sub = static_cast<int>(t & (G - 1));
    const bool active = p < a.n_pos;
    const int w = active ? __ldg(a.len + p) : 0;  // -1: a long row, no entries here
    const int64_t base = active ? __ldg(a.slice_ptr + (p >> a.log2C)) : 0;
    const int64_t q = p & a.cmask;
    // slot of entry j = sub + k * G: column-major base + j * stride + q,
    // interleaved base + (k * stride + q) * G + sub; both advance G * stride per k
    const int64_t first = IL ? base + q * G + sub : base + static_cast<int64_t>(sub) * a.stride + q;
    const int64_t step = G * a.stride;
    const int32_t *__restrict__ cp = a.col + first;
    const T *__restrict__ vp = val + first;
    int32_t c[U];
    T v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const bool on = sub + u * G < w;
        c[u] = on ? ld_stream(cp + u * step) : 0;
        v[u] = on ? ld_stream(vp + u * step) : T(0);
    }
    grid_wait();
    T acc = T(0);
    for (int j = sub; j < w;) {
        T xv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) xv[u] = (j + u * G < w) ? gather_x<K>(x + c[u]) : T(0);
#pragma unroll
        for (int u = 0; u < U; ++u) acc = fma(v[u], xv[u], acc);  // inactive slots add +0 * +0
        j += U * G;
        if (j >= w) break;
        cp += U * step;
        vp += U * step;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool on = j + u * G < w;
            c[u] = on ? ld_stream(cp + u * step) : 0;
            v[u] = on ? ld_stream(vp + u * step) : T(0);
        }
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub == 0 && w >= 0 && active) {
        const int64_t r = a.perm ? static_cast<int64_t>(__ldg(a.perm + p)) : p;
        if (r >= 0 && r < a.n) store_y(y, r, acc, ep);
    }
}

// Column-grouped, column-major slots (the AMD rearrangement): a warp takes 32
// consecutive row positions and one residue class k of entries (j = k, k + G, ...), so
// at every step it reads one contiguous run of 32 slots of column j.  The G warps that
// share a set of 32 rows add their partial sums in shared memory, in warp order.
template <typename T, int G, bool K>
__global__ void __launch_bounds__(kSellBlock, (G == 8 && sizeof(T) == 8) ? 5 : 6)  // no spills at G = 8, float64
    k_sellcg(SellArgs a, const T *__restrict__ val, const T *__restrict__ x, T *__restrict__ y, Epi ep) {
    constexpr int U = 4;
    constexpr int kSets = kSellBlock / 32 / G;  // sets of 32 rows per block
    __shared__ T part[G][kSets * 32];
    allow_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int set = warp / G, k = warp % G;
    const int64_t p = (static_cast<int64_t>(blockIdx.x) * kSets + set) * 32 + lane;
    const bool active = p < a.n_pos;
    const int w = active ? __ldg(a.len + p) : 0;  // -1: a long row, no entries here
    const int64_t base = active ? __ldg(a.slice_ptr + (p >> a.log2C)) : 0;
    const int64_t q = p & a.cmask;
    const int64_t step = G * a.stride;
    const int32_t *__restrict__ cp = a.col + base + k * a.stride + q;
    const T *__restrict__ vp = val + base + k * a.stride + q;
    int32_t c[U];
    T v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const bool on = k + u * G < w;
        c[u] = on ? ld_stream(cp + u * step) : 0;
        v[u] = on ? ld_stream(vp + u * step) : T(0);
    }
    grid_wait();
    T acc = T(0);
    for (int j = k; j < w;) {
        T xv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) xv[u] = (j + u * G < w) ? gather_x<K>(x + c[u]) : T(0);
#pragma unroll
        for (int u = 0; u < U; ++u) acc = fma(v[u], xv[u], acc);
        j += U * G;
        if (j >= w) break;
        cp += U * step;
        vp += U * step;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool on = j + u * G < w;
            c[u] = on ? ld_stream(cp + u * step) : 0;
            v[u] = on ? ld_stream(vp + u * step) : T(0);
        }
    }
    part[k][set * 32 + lane] = acc;
    __syncthreads();
    if (k == 0 && active && w >= 0) {
        T sum = part[0][set * 32 + lane];
#pragma unroll
        for (int kk = 1; kk < G; ++kk) sum += part[kk][set * 32 + lane];
        const int64_t r = a.perm ? static_cast<int64_t>(__ldg(a.perm + p)) : p;
        if (r >= 0 && r < a.n) store_y(y, r, sum, ep);
    }
}

template <typename T, int G>
cudaError_t sellcg_launch(const Sliced &sl, int64_t n, const T *x, T *y, cudaStream_t s, const Epi &ep) {
    const SellArgs args = sell_args(sl, n);
    const T *val = static_cast<const T *>(sl.val);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    constexpr int64_t rows_per_block = kSellBlock / G;
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(sl.n_pos, rows_per_block)));
    cfg.blockDim = dim3(kSellBlock);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return sl.keep_x ? cudaLaunchKernelEx(&cfg, k_sellcg<T, G, true>, args, val, x, y, ep)
                     : cudaLaunchKernelEx(&cfg, k_sellcg<T, G, false>, args, val, x, y, ep);
}

template <typename T, int G, bool IL>
cudaError_t sellg_launch(const Sliced &sl, int64_t n, const T *x, T *y, cudaStream_t s, const Epi &ep) {
    const SellArgs args = sell_args(sl, n);
    const T *val = static_cast<const T *>(sl.val);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(sl.n_pos * G, kSellBlock)));
    cfg.blockDim = dim3(kSellBlock);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return sl.keep_x ? cudaLaunchKernelEx(&cfg, k_sellg<T, G, IL, true>, args, val, x, y, ep)
                     : cudaLaunchKernelEx(&cfg, k_sellg<T, G, IL, false>, args, val, x, y, ep);
}

template <typename T, bool IL>
cudaError_t sellg_dispatch_g(const Sliced &sl, int64_t n, const T *x, T *y, cudaStream_t s, const Epi &ep) {
    switch (sl.group) {
        case 2: return sellg_launch<T, 2, IL>(sl, n, x, y, s, ep);
        case 4: return sellg_launch<T, 4, IL>(sl, n, x, y, s, ep);
        case 8: return sellg_launch<T, 8, IL>(sl, n, x, y, s, ep);
        case 16: return sellg_launch<T, 16, IL>(sl, n, x, y, s, ep);
        case 32: return sellg_launch<T, 32, IL>(sl, n, x, y, s, ep);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t sellg_dispatch(const Sliced &sl, int64_t n, const T *x, T *y, cudaStream_t s, const Epi &ep) {
    if (sl.group_mode == 2) {
        switch (sl.group) {
            case 2: return sellcg_launch<T, 2>(sl, n, x, y, s, ep);
            case 4: return sellcg_launch<T, 4>(sl, n, x, y, s, ep);
            case 8: return sellcg_launch<T, 8>(sl, n, x, y, s, ep);
            default: return cudaErrorInvalidValue;
        }
    }
    return sl.interleaved ? sellg_dispatch_g<T, true>(sl, n, x, y, s, ep)
                          : sellg_dispatch_g<T, false>(sl, n, x, y, s, ep);
}

}  // namespace

cudaError_t launch_sellg_apply(int dtype, const Sliced &sl, int64_t n, const void *x, void *y, cudaStream_t s,
                               const Scale *scale) {
    if (!sl.present || sl.n_pos <= 0) return cudaSuccess;
    const Epi ep = scale ? Epi{scale->alpha, scale->beta, 1} : Epi{1.0, 0.0, 0};
    if (dtype == SPMV_F64)
        return sellg_dispatch<double>(sl, n, static_cast<const double *>(x), static_cast<double *>(y), s, ep);
    return sellg_dispatch<float>(sl, n, static_cast<const float *>(x), static_cast<float *>(y), s, ep);
}

}  // namespace spmv
