// Sliced-ELL apply with 16-byte vector loads: one thread per row, the row's slots
// stored in groups that one 128-bit load fetches -- four column indices at a time
// and 16 bytes of values (two doubles or four floats), the slot variant for vector
// loads of the sliced layout (slot_of() with groups of 4 indices / 16 bytes of values).
// A warp's load of one group reads 512 contiguous bytes.  Each thread still stops at
// its own row's length: a vector may carry padding slots past the row's end, which
// are never gathered or multiplied.  Same epilogue and programmatic dependent launch
// as the element-wise kernel; rows marked long (len = -1) are left to the row-split
// pass.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_util.cuh"
#include "sell_common.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

using namespace dev;
using namespace sellk;

// 4 entries of a row: their columns and values (streamed, evict-first)
template <typename T>
struct Group4 {
    int4 c;
    T v[4];
};

template <typename T>
__device__ __forceinline__ void load_group(const int32_t *__restrict__ col, const T *__restrict__ val, int64_t base,
                                           int64_t q, int64_t stride, int g, Group4<T> &out);

template <>
__device__ __forceinline__ void load_group<double>(const int32_t *__restrict__ col, const double *__restrict__ val,
                                                   int64_t base, int64_t q, int64_t stride, int g,
                                                   Group4<double> &out) {
    out.c = __ldcs(reinterpret_cast<const int4 *>(col + base + ((static_cast<int64_t>(g) * stride + q) << 2)));
    const double *v0 = val + base + ((static_cast<int64_t>(2 * g) * stride + q) << 1);
    const double *v1 = val + base + ((static_cast<int64_t>(2 * g + 1) * stride + q) << 1);
    const double2 a = __ldcs(reinterpret_cast<const double2 *>(v0));
    const double2 b = __ldcs(reinterpret_cast<const double2 *>(v1));
    out.v[0] = a.x, out.v[1] = a.y, out.v[2] = b.x, out.v[3] = b.y;
}

template <>
__device__ __forceinline__ void load_group<float>(const int32_t *__restrict__ col, const float *__restrict__ val,
                                                  int64_t base, int64_t q, int64_t stride, int g, Group4<float> &out) {
    out.c = __ldcs(reinterpret_cast<const int4 *>(col + base + ((static_cast<int64_t>(g) * stride + q) << 2)));
    const float *v0 = val + base + ((static_cast<int64_t>(g) * stride + q) << 2);
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(v0));
    out.v[0] = a.x, out.v[1] = a.y, out.v[2] = a.z, out.v[3] = a.w;
}

// A group past the row's end is not loaded: zeros, so its FMAs add +0 * +0.
template <typename T>
__device__ __forceinline__ void zero_group(Group4<T> &g) {
    g.c = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u) g.v[u] = T(0);
}

// G4: groups of 4 entries in flight per thread (1 for float64, 2 for float32)
template <typename T, int CS, bool K>
__global__ void __launch_bounds__(kSellBlock, CS > 0 ? 8 : 6)
    k_sellv(SellArgs a, const T *__restrict__ val, const T *__restrict__ x, T *__restrict__ y, Epi ep) {
    constexpr int G4 = sizeof(T) == 8 ? 1 : 2;
    allow_dependents();
    const int64_t p = gtid();
    if (p >= a.n_pos) return;
    const int w = __ldg(a.len + p);
    const uint64_t up = static_cast<uint64_t>(p);
    const int64_t base = CS > 0 ? __ldg(a.slice_ptr + (up / CS)) : __ldg(a.slice_ptr + (p >> a.log2C));
    const int64_t q = CS > 0 ? static_cast<int64_t>(up % CS) : static_cast<int64_t>(p & a.cmask);
    const int64_t stride = CS > 0 ? CS : a.stride;
    const int64_t r = a.perm ? static_cast<int64_t>(__ldg(a.perm + p)) : p;
    Group4<T> grp[G4];
#pragma unroll
    for (int k = 0; k < G4; ++k) {
        if (4 * k < w)
            load_group<T>(a.col, val, base, q, stride, k, grp[k]);
        else
            zero_group(grp[k]);
    }
    grid_wait();  // matrix data above, x and y below
    T acc = T(0);
    for (int j = 0; j < w;) {
#pragma unroll
        for (int k = 0; k < G4; ++k) {
            const int c[4] = {grp[k].c.x, grp[k].c.y, grp[k].c.z, grp[k].c.w};
            T xv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) xv[u] = (j + 4 * k + u < w) ? gather_x<K>(x + c[u]) : T(0);
#pragma unroll
            for (int u = 0; u < 4; ++u) acc = fma(grp[k].v[u], xv[u], acc);  // past the row's end: +0 * +0
        }
        j += 4 * G4;
        if (j >= w) break;
#pragma unroll
        for (int k = 0; k < G4; ++k) {
            if (j + 4 * k < w)
                load_group<T>(a.col, val, base, q, stride, (j >> 2) + k, grp[k]);
            else
                zero_group(grp[k]);
        }
    }
    if (w >= 0 && r >= 0 && r < a.n) store_y(y, r, acc, ep);
}

template <typename T, int CS, bool K>
cudaError_t sellv_launch(const Sliced &sl, int64_t n, const T *x, T *y, cudaStream_t s, const Epi &ep) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(sl.n_pos, kSellBlock)));
    cfg.blockDim = dim3(kSellBlock);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_sellv<T, CS, K>, sell_args(sl, n), static_cast<const T *>(sl.val), x, y, ep);
}

template <typename T, int CS>
cudaError_t sellv_launch_k(const Sliced &sl, int64_t n, const T *x, T *y, cudaStream_t s, const Epi &ep) {
    return sl.keep_x ? sellv_launch<T, CS, true>(sl, n, x, y, s, ep) : sellv_launch<T, CS, false>(sl, n, x, y, s, ep);
}

template <typename T>
cudaError_t sellv_dispatch(const Sliced &sl, int64_t n, const T *x, T *y, cudaStream_t s, const Epi &ep) {
    const bool sliced = sl.log2C < 31;
    if (sliced && sl.C == 32) return sellv_launch_k<T, 32>(sl, n, x, y, s, ep);
    if (sliced && sl.C == 64) return sellv_launch_k<T, 64>(sl, n, x, y, s, ep);
    return sellv_launch_k<T, 0>(sl, n, x, y, s, ep);
}

}  // namespace

cudaError_t launch_sellv_apply(int dtype, const Sliced &sl, int64_t n, const void *x, void *y, cudaStream_t s,
                               const Scale *scale) {
    if (!sl.present || sl.n_pos <= 0) return cudaSuccess;
    const Epi ep = scale ? Epi{scale->alpha, scale->beta, 1} : Epi{1.0, 0.0, 0};
    if (dtype == SPMV_F64)
        return sellv_dispatch<double>(sl, n, static_cast<const double *>(x), static_cast<double *>(y), s, ep);
    return sellv_dispatch<float>(sl, n, static_cast<const float *>(x), static_cast<float *>(y), s, ep);
}

}  // namespace spmv
