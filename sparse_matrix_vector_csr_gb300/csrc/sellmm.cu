// Multi-vector apply on the sliced layout: Y = alpha * A X + beta * Y for NV
// right-hand sides at once (NV = 2, 4 or 8), X and Y row-major (row j of X holds
// the NV values that column j of A multiplies).  The matrix entries are streamed
// once for all NV vectors, and each gather of a row of X moves NV contiguous
// values with 8- or 16-byte loads, so on matrices whose random x gathers bound the
// single-vector apply the gather cost is shared by NV products.  Long rows use the
// row-split pass in the same launch, as in sell.cu.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_util.cuh"
#include "sell_common.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

using namespace dev;
using namespace sellk;

// NV contiguous values at p with the widest aligned vector loads (the caller has
// checked that p is aligned to min(16, NV * sizeof(T)) bytes).
template <typename T, int NV>
__device__ __forceinline__ void load_row(const T *__restrict__ p, T (&o)[NV]) {
    if constexpr (sizeof(T) == 8) {
#pragma unroll
        for (int i = 0; i < NV; i += 2) {
            const double2 v = __ldg(reinterpret_cast<const double2 *>(p + i));
            o[i] = v.x;
            o[i + 1] = v.y;
        }
    } else if constexpr (NV % 4 == 0) {
#pragma unroll
        for (int i = 0; i < NV; i += 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p + i));
            o[i] = v.x;
            o[i + 1] = v.y;
            o[i + 2] = v.z;
            o[i + 3] = v.w;
        }
    } else {
        const float2 v = __ldg(reinterpret_cast<const float2 *>(p));
        o[0] = v.x;
        o[1] = v.y;
    }
}

template <typename T, int CS, int NV>
__device__ __forceinline__ void sellmm_row(int64_t p, const SellArgs &a, const T *__restrict__ val,
                                           const T *__restrict__ X, int64_t ldx, T *__restrict__ Y, int64_t ldy,
                                           const Epi &ep) {
    // entries of the row loaded ahead of their gathers: enough bytes in flight to stream
    // the matrix, within the registers the NV accumulators and gathered values leave
    constexpr int U = NV >= 8 ? 1 : sizeof(T) == 4 ? 4 : 2;
    const int w = __ldg(a.len + p);
    const uint64_t up = static_cast<uint64_t>(p);
    const int64_t slot = __ldg(a.slice_ptr + (up / CS)) + static_cast<int64_t>(up % CS);
    const int32_t *__restrict__ cp = a.col + slot;
    const T *__restrict__ vp = val + slot;
    const int64_t r = a.perm ? static_cast<int64_t>(__ldg(a.perm + p)) : p;
    int32_t c[U];
    T v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        c[u] = u < w ? ld_stream(cp + u * CS) : 0;
        v[u] = u < w ? ld_stream(vp + u * CS) : T(0);
    }
    grid_wait();  // matrix data above, X and Y below (programmatic dependent launch)
    T acc[NV];
#pragma unroll
    for (int q = 0; q < NV; ++q) acc[q] = T(0);
    for (int j = 0; j < w;) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (j + u < w) {
                T xr[NV];
                load_row<T, NV>(X + static_cast<int64_t>(c[u]) * ldx, xr);
#pragma unroll
                for (int q = 0; q < NV; ++q) acc[q] = fma(v[u], xr[q], acc[q]);
            }
        }
        j += U;
        if (j >= w) break;
        cp += U * CS;
        vp += U * CS;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            c[u] = j + u < w ? ld_stream(cp + u * CS) : 0;
            v[u] = j + u < w ? ld_stream(vp + u * CS) : T(0);
        }
    }
    if (w >= 0 && r >= 0 && r < a.n) {
#pragma unroll
        for (int q = 0; q < NV; ++q) store_y(Y + r * ldy, q, acc[q], ep);
    }
}

// One warp reduces chunk c of a long row for NV vectors; partials are kept per
// (chunk, vector), and the warp finishing a row's last chunk adds them up.
template <typename T, int NV>
__device__ __forceinline__ void splitmm_chunk(int64_t c, int lane, const SplitArgs &a, const T *__restrict__ val,
                                              const T *__restrict__ X, int64_t ldx, T *__restrict__ Y, int64_t ldy,
                                              const Epi &ep) {
    // U entries a lane loaded ahead of their gathers, as in the single-vector chunk loop;
    // each lane still adds its entries in index order
    constexpr int U = NV >= 8 ? 2 : 4;
    const int32_t b = __ldg(a.chunk_begin + c), e = __ldg(a.chunk_end + c);
    T acc[NV];
#pragma unroll
    for (int q = 0; q < NV; ++q) acc[q] = T(0);
    bool first = true;
    for (int32_t k = b + lane; k < e; k += 32 * U) {
        int32_t cc[U];
        T v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool on = k + 32 * u < e;
            cc[u] = on ? ld_stream(a.col + k + 32 * u) : 0;
            v[u] = on ? ld_stream(val + k + 32 * u) : T(0);
        }
        if (first) {
            grid_wait();  // matrix data above, X and Y below
            first = false;
        }
        T xr[U][NV];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (k + 32 * u < e)
                load_row<T, NV>(X + static_cast<int64_t>(cc[u]) * ldx, xr[u]);
            else
#pragma unroll
                for (int q = 0; q < NV; ++q) xr[u][q] = T(0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int q = 0; q < NV; ++q) acc[q] = fma(v[u], xr[u][q], acc[q]);  // past the end: +0 * +0
    }
    if (first) grid_wait();  // a lane with no entry of its own still writes after the wait
    double s[NV];
#pragma unroll
    for (int q = 0; q < NV; ++q) {
        s[q] = static_cast<double>(acc[q]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s[q] += __shfl_xor_sync(0xffffffffu, s[q], off);
    }
    const int32_t cr = __ldg(a.chunk_row + c);
    if (cr < 0) {
        if (lane == 0) {
            const int64_t r = __ldg(a.rows + ~cr);
#pragma unroll
            for (int q = 0; q < NV; ++q) store_y(Y + r * ldy, q, static_cast<T>(s[q]), ep);
        }
        return;
    }
    const int32_t c0 = __ldg(a.row_chunk_ptr + cr), c1 = __ldg(a.row_chunk_ptr + cr + 1);
    int last = 0;
    if (lane == 0) {
#pragma unroll
        for (int q = 0; q < NV; ++q) a.partial[c * NV + q] = s[q];
        __threadfence();
        last = atomicAdd(a.done + cr, 1) == (c1 - c0) - 1;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    double t[NV];
#pragma unroll
    for (int q = 0; q < NV; ++q) t[q] = 0.0;
    for (int32_t g = c0 + lane; g < c1; g += 32) {
#pragma unroll
        for (int q = 0; q < NV; ++q) t[q] += __ldcg(a.partial + static_cast<int64_t>(g) * NV + q);
    }
#pragma unroll
    for (int q = 0; q < NV; ++q) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t[q] += __shfl_xor_sync(0xffffffffu, t[q], off);
    }
    if (lane == 0) {
        const int64_t r = __ldg(a.rows + cr);
#pragma unroll
        for (int q = 0; q < NV; ++q) store_y(Y + r * ldy, q, static_cast<T>(t[q]), ep);
        a.done[cr] = 0;
    }
}

template <typename T, int CS, int NV>
__global__ void __launch_bounds__(kSellBlock) k_sellmm(SellArgs a, const T *__restrict__ val, const T *__restrict__ X,
                                                      int64_t ldx, T *__restrict__ Y, int64_t ldy, Epi ep) {
    allow_dependents();
    const int64_t p = gtid();
    if (p < a.n_pos) sellmm_row<T, CS, NV>(p, a, val, X, ldx, Y, ldy, ep);
}

template <typename T, int CS, int NV>
__global__ void __launch_bounds__(kSellBlock)
    k_sellmm_split(SellArgs a, const T *__restrict__ val, SplitArgs b, const T *__restrict__ split_val,
                   int64_t split_ctas, const T *__restrict__ X, int64_t ldx, T *__restrict__ Y, int64_t ldy, Epi ep) {
    allow_dependents();
    if (blockIdx.x < split_ctas) {
        const int64_t c = (static_cast<int64_t>(blockIdx.x) * kSellBlock + threadIdx.x) >> 5;
        if (c < b.n_chunks) splitmm_chunk<T, NV>(c, threadIdx.x & 31, b, split_val, X, ldx, Y, ldy, ep);
        return;
    }
    const int64_t p = (static_cast<int64_t>(blockIdx.x) - split_ctas) * kSellBlock + threadIdx.x;
    if (p < a.n_pos) sellmm_row<T, CS, NV>(p, a, val, X, ldx, Y, ldy, ep);
}

template <typename T, int CS, int NV>
cudaError_t mm_launch(const Sliced &sl, int64_t n, const Segmented *sg, const T *X, int64_t ldx, T *Y, int64_t ldy,
                      cudaStream_t s, const Epi &ep) {
    const T *val = static_cast<const T *>(sl.val);
    const int64_t sell_ctas = ceil_div(sl.n_pos, kSellBlock);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kSellBlock);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (sg && sg->kind == 3 && sg->n_chunks > 0) {
        const int64_t split_ctas = ceil_div(sg->n_chunks * 32, kSellBlock);
        cfg.gridDim = dim3(static_cast<unsigned>(split_ctas + sell_ctas));
        return cudaLaunchKernelEx(&cfg, k_sellmm_split<T, CS, NV>, sell_args(sl, n), val, split_args(*sg),
                                  static_cast<const T *>(sg->val), split_ctas, X, ldx, Y, ldy, ep);
    }
    cfg.gridDim = dim3(static_cast<unsigned>(sell_ctas));
    return cudaLaunchKernelEx(&cfg, k_sellmm<T, CS, NV>, sell_args(sl, n), val, X, ldx, Y, ldy, ep);
}

template <typename T, int CS>
cudaError_t mm_nv(int nv, const Sliced &sl, int64_t n, const Segmented *sg, const T *X, int64_t ldx, T *Y,
                  int64_t ldy, cudaStream_t s, const Epi &ep) {
    switch (nv) {
        case 2: return mm_launch<T, CS, 2>(sl, n, sg, X, ldx, Y, ldy, s, ep);
        case 4: return mm_launch<T, CS, 4>(sl, n, sg, X, ldx, Y, ldy, s, ep);
        case 8: return mm_launch<T, CS, 8>(sl, n, sg, X, ldx, Y, ldy, s, ep);
        default: return cudaErrorNotSupported;
    }
}

template <typename T>
cudaError_t mm_dispatch(int nv, const Sliced &sl, int64_t n, const Segmented *sg, const T *X, int64_t ldx, T *Y,
                        int64_t ldy, cudaStream_t s, const Epi &ep) {
    const bool sliced = sl.log2C < 31;
    if (sliced && sl.C == 32) return mm_nv<T, 32>(nv, sl, n, sg, X, ldx, Y, ldy, s, ep);
    if (sliced && sl.C == 64) return mm_nv<T, 64>(nv, sl, n, sg, X, ldx, Y, ldy, s, ep);
    return cudaErrorNotSupported;
}

}  // namespace

bool sell_multi_supported(const Sliced &sl) {
    return sl.present && sl.group == 1 && !sl.interleaved && sl.log2C < 31 && (sl.C == 32 || sl.C == 64);
}

cudaError_t launch_sell_multi(int dtype, int nv, const Sliced &sl, int64_t n, const Segmented *split, const void *X,
                              int64_t ldx, void *Y, int64_t ldy, cudaStream_t s, const Scale &scale) {
    if (!sl.present || sl.n_pos <= 0) return cudaSuccess;
    // Y = A X (alpha 1, beta 0) stores the sums as they are: the scaling multiply would
    // cost about a seventh of the FP64 work on short rows, and 1 * v is v
    const Epi ep{scale.alpha, scale.beta, (scale.alpha == 1.0 && scale.beta == 0.0) ? 0 : 1};
    if (dtype == SPMV_F64)
        return mm_dispatch<double>(nv, sl, n, split, static_cast<const double *>(X), ldx, static_cast<double *>(Y),
                                   ldy, s, ep);
    return mm_dispatch<float>(nv, sl, n, split, static_cast<const float *>(X), ldx, static_cast<float *>(Y), ldy, s,
                              ep);
}

}  // namespace spmv
