// Apply kernels of the sm_103a SpMV library.
//
//  k_sell        one thread per sorted row position of a column-major sliced layout
//                (SELL-C-sigma, ELLPACK-R, HYB's ELL part); each thread stops at its
//                own row's length, so padding is never loaded or multiplied
//                (ELLPACK-R, GPGPU spMVM paper arXiv 1112.5588, ELLPACK-R section;
//                the scite report's "early stopping").
//  k_csr_vector  g lanes per CSR row, partial sums combined with __shfl_xor_sync
//                ("subwarp" per row, scite report quoting "Sparse Linear Algebra on
//                AMD and NVIDIA GPUs").
//  k_merge_path  equal shares of the merged (row ends, entries) sequence per CTA for
//                the few very long rows (Trilinos issue on unpackAndCombine: very
//                long rows, merge-path load balancing).
//  k_coo         equal shares of COO entries per CTA with a segmented sum by row
//                (load-balanced COO kernel of the scite report's abstract).
//  k_carry_fixup adds the partial sums of rows that cross CTA boundaries; no atomics.
#include <cuda_runtime.h>

#include <cstdint>

#include "spmv_internal.cuh"

namespace spmv {
namespace {

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

// ---------------------------------------------------------------------------
// sliced layout
// ---------------------------------------------------------------------------
// Entries of a row are processed U at a time: the U column indices and values
// (predicated on the row length, so padding is never touched) are loaded first,
// then the U gathers of x, then U fused multiply-adds.  This keeps 2U independent
// streaming loads in flight per thread before the dependent gathers.  U = 4 for
// fp64 and 8 for fp32 fills the load queue without raising register use above
// 32, which keeps all 64 warps of an SM resident.
template <typename T>
struct SellChunk {
    static constexpr int U = sizeof(T) == 8 ? 4 : 8;
};

// CS > 0: SELL with a compile-time slice height CS (stride = CS).
// CS == 0: runtime addressing (slice p >> log2C, row p & cmask, stride `stride`),
//          used by the single-slice ELLPACK-R / HYB-ELL layout and other slice heights.
template <typename T, int CS>
__global__ void __launch_bounds__(kSellBlock, 8) k_sell(int64_t n_pos, int log2C, uint32_t cmask, int64_t stride,
                                                        const int64_t *__restrict__ slice_ptr,
                                                        const int32_t *__restrict__ len,
                                                        const int32_t *__restrict__ perm,
                                                        const int32_t *__restrict__ col, const T *__restrict__ val,
                                                        const T *__restrict__ x, T *__restrict__ y, int64_t n) {
    constexpr int U = SellChunk<T>::U;
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
        for (int j = 0; j < w; j += U) {
            int32_t c[U];
            T a[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool on = j + u < w;
                c[u] = on ? ld_stream(cp) : 0;
                a[u] = on ? ld_stream(vp) : T(0);
                cp += stride;
                vp += stride;
            }
            T xv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) xv[u] = (j + u < w) ? ld_x(x + c[u]) : T(0);
#pragma unroll
            for (int u = 0; u < U; ++u) acc = fma(a[u], xv[u], acc);
        }
    }
    const int64_t r = perm ? static_cast<int64_t>(__ldg(perm + p)) : p;
    if (r >= 0 && r < n) y[r] = acc;
}

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

// ---------------------------------------------------------------------------
// CTA-wide segmented scan of (flag, value) pairs, one per thread, in thread order.
// The pair of a thread is (it ended a row, sum of its still-open last segment).
// Combining an earlier pair a with a later pair b gives
//     (a.f | b.f, b.f ? b.v : a.v + b.v),
// so the exclusive result of a thread is what the rows still open at its start
// have collected from earlier threads of the CTA.
// ---------------------------------------------------------------------------
template <typename T, int THREADS>
struct SegScan {
    static constexpr int W = THREADS / 32;
    int flag[W];
    T val[W];
    int pflag[W];
    T pval[W];
};

template <typename T, int THREADS>
__device__ __forceinline__ T seg_scan_exclusive(int f, T v, SegScan<T, THREADS> &sm) {
    constexpr int W = THREADS / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int fu = __shfl_up_sync(0xffffffffu, f, off);
        const T vu = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) {
            if (!f) v = vu + v;
            f |= fu;
        }
    }
    if (lane == 31) {
        sm.flag[warp] = f;
        sm.val[warp] = v;
    }
    __syncthreads();
    if (warp == 0) {
        int wf = lane < W ? sm.flag[lane] : 0;
        T wv = lane < W ? sm.val[lane] : T(0);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int fu = __shfl_up_sync(0xffffffffu, wf, off);
            const T vu = __shfl_up_sync(0xffffffffu, wv, off);
            if (lane >= off) {
                if (!wf) wv = vu + wv;
                wf |= fu;
            }
        }
        int ef = __shfl_up_sync(0xffffffffu, wf, 1);
        T ev = __shfl_up_sync(0xffffffffu, wv, 1);
        if (lane == 0) {
            ef = 0;
            ev = T(0);
        }
        if (lane < W) {
            sm.pflag[lane] = ef;
            sm.pval[lane] = ev;
        }
    }
    __syncthreads();
    const T pv = sm.pval[warp];
    const int lf = __shfl_up_sync(0xffffffffu, f, 1);
    const T lv = __shfl_up_sync(0xffffffffu, v, 1);
    if (lane == 0) return pv;
    return lf ? lv : pv + lv;
}

// ---------------------------------------------------------------------------
// merge-path over a compact CSR (long rows, or the HEC spill)
// ---------------------------------------------------------------------------
// Stage the CTA's entries as products a_k * x[col_k] in shared memory: every
// thread issues its (at most kMergeIpt) column/value loads first, then the gathers.
template <typename T>
__device__ __forceinline__ void stage_products(const int32_t *__restrict__ col, const T *__restrict__ val,
                                               const T *__restrict__ x, int64_t k0, int nk, T *s_prod) {
    int32_t c[kMergeIpt];
    T a[kMergeIpt];
#pragma unroll
    for (int q = 0; q < kMergeIpt; ++q) {
        const int t = threadIdx.x + q * kMergeThreads;
        const bool on = t < nk;
        c[q] = on ? ld_stream(col + k0 + t) : 0;
        a[q] = on ? ld_stream(val + k0 + t) : T(0);
    }
#pragma unroll
    for (int q = 0; q < kMergeIpt; ++q) {
        const int t = threadIdx.x + q * kMergeThreads;
        if (t < nk) s_prod[t] = a[q] * ld_x(x + c[q]);
    }
}

// merge-path split: number of row ends among the first d items of the path that
// merges the row ends ptr[1..n_rows] with the entry indices 0..nnz-1
__device__ __forceinline__ int64_t merge_split(int64_t d, int64_t n_rows, int64_t nnz, const int32_t *ptr) {
    int64_t lo = max64(0, d - nnz), hi = min64(d, n_rows);
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(ptr[mid + 1]) <= d - 1 - mid)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// kIdentityRows: compact row i is matrix row i (rows may be NULL).
// part: the split of every CTA boundary, precomputed when the matrix was built
// (part[c] = row ends among the first c * kMergeItems path items), or NULL to
// search it here.
template <typename T, bool kIdentityRows = false>
__global__ void __launch_bounds__(kMergeThreads) k_merge_path(
    int64_t n_rows, int64_t nnz, const int32_t *__restrict__ ptr, const int32_t *__restrict__ rows,
    const int32_t *__restrict__ col, const T *__restrict__ val, const T *__restrict__ x, T *__restrict__ y,
    int32_t *__restrict__ carry_row, double *__restrict__ carry_val, int accumulate,
    const int32_t *__restrict__ part) {
    __shared__ T s_prod[kMergeItems];
    __shared__ int32_t s_end[kMergeItems];
    __shared__ int64_t s_coord[2];
    __shared__ SegScan<T, kMergeThreads> s_scan;

    const int64_t total = n_rows + nnz;
    const int64_t d0 = static_cast<int64_t>(blockIdx.x) * kMergeItems;
    const int64_t d1 = min(d0 + kMergeItems, total);
    int64_t i0, i1;
    if (part) {
        i0 = __ldg(part + blockIdx.x);
        i1 = __ldg(part + blockIdx.x + 1);
    } else {
        if (threadIdx.x < 2) s_coord[threadIdx.x] = merge_split(threadIdx.x ? d1 : d0, n_rows, nnz, ptr);
        __syncthreads();
        i0 = s_coord[0];
        i1 = s_coord[1];
    }
    const int64_t k0 = d0 - i0;
    const int ni = static_cast<int>(i1 - i0);
    const int nk = static_cast<int>((d1 - i1) - k0);
    stage_products(col, val, x, k0, nk, s_prod);
#pragma unroll
    for (int q = 0; q < kMergeIpt; ++q) {
        const int t = threadIdx.x + q * kMergeThreads;
        if (t < ni) s_end[t] = static_cast<int32_t>(__ldg(ptr + i0 + t + 1) - k0);
    }
    __syncthreads();

    const int npath = ni + nk;
    const int dl = min(static_cast<int>(threadIdx.x) * kMergeIpt, npath);
    const int dl_end = min(dl + kMergeIpt, npath);
    int lo = max(0, dl - nk), hi = min(dl, ni);
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_end[mid] <= dl - 1 - mid)
            lo = mid + 1;
        else
            hi = mid;
    }
    const int il0 = lo, kl0 = dl - lo;

    int il = il0, kl = kl0, flag = 0;
    T run = T(0);
    for (int it = dl; it < dl_end; ++it) {
        if (il < ni && s_end[il] <= kl) {
            flag = 1;
            run = T(0);
            ++il;
        } else {
            run += s_prod[kl];
            ++kl;
        }
    }
    const int open_row = il;
    const T carry_in = seg_scan_exclusive<T, kMergeThreads>(flag, run, s_scan);

    il = il0;
    kl = kl0;
    T acc = carry_in;
    for (int it = dl; it < dl_end; ++it) {
        if (il < ni && s_end[il] <= kl) {
            const int32_t r = kIdentityRows ? static_cast<int32_t>(i0 + il) : __ldg(rows + i0 + il);
            y[r] = accumulate ? y[r] + acc : acc;
            acc = T(0);
            ++il;
        } else {
            acc += s_prod[kl];
            ++kl;
        }
    }
    if (threadIdx.x == kMergeThreads - 1) {
        const T inclusive = flag ? run : carry_in + run;
        const int64_t i = i0 + open_row;
        if (i < n_rows) {
            carry_row[blockIdx.x] = kIdentityRows ? static_cast<int32_t>(i) : __ldg(rows + i);
            carry_val[blockIdx.x] = static_cast<double>(inclusive);
        } else {
            carry_row[blockIdx.x] = -1;
            carry_val[blockIdx.x] = 0.0;
        }
    }
}

// ---------------------------------------------------------------------------
// load-balanced COO (HYB spill): equal entry shares, segmented by row
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kMergeThreads) k_coo(int64_t nnz, const int32_t *__restrict__ crow,
                                                       const int32_t *__restrict__ col, const T *__restrict__ val,
                                                       const T *__restrict__ x, T *__restrict__ y,
                                                       int32_t *__restrict__ carry_row,
                                                       double *__restrict__ carry_val, int accumulate) {
    __shared__ T s_prod[kMergeItems];
    __shared__ int32_t s_row[kMergeItems + 1];
    __shared__ SegScan<T, kMergeThreads> s_scan;
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * kMergeItems;
    const int nk = static_cast<int>(min64(kMergeItems, nnz - k0));
    stage_products(col, val, x, k0, nk, s_prod);
#pragma unroll
    for (int q = 0; q < kMergeIpt; ++q) {
        const int t = threadIdx.x + q * kMergeThreads;
        if (t < nk) s_row[t] = ld_stream(crow + k0 + t);
    }
    if (threadIdx.x == 0) s_row[nk] = (k0 + nk < nnz) ? crow[k0 + nk] : -1;
    __syncthreads();
    const int b = min(static_cast<int>(threadIdx.x) * kMergeIpt, nk);
    const int e = min(b + kMergeIpt, nk);
    int flag = 0;
    T run = T(0);
    for (int k = b; k < e; ++k) {
        run += s_prod[k];
        if (s_row[k] != s_row[k + 1]) {
            flag = 1;
            run = T(0);
        }
    }
    const T carry_in = seg_scan_exclusive<T, kMergeThreads>(flag, run, s_scan);
    T acc = carry_in;
    for (int k = b; k < e; ++k) {
        acc += s_prod[k];
        if (s_row[k] != s_row[k + 1]) {
            const int32_t r = s_row[k];
            y[r] = accumulate ? y[r] + acc : acc;
            acc = T(0);
        }
    }
    if (threadIdx.x == kMergeThreads - 1) {
        const T inclusive = flag ? run : carry_in + run;
        if (nk > 0 && s_row[nk - 1] == s_row[nk]) {
            carry_row[blockIdx.x] = s_row[nk - 1];
            carry_val[blockIdx.x] = static_cast<double>(inclusive);
        } else {
            carry_row[blockIdx.x] = -1;
            carry_val[blockIdx.x] = 0.0;
        }
    }
}

// Rows crossing CTA boundaries: carries of one row are contiguous (rows only grow
// along the path).  One warp per carry slot; the warp whose slot starts a run sums
// the run (lanes stride through it, then a shuffle tree, all in double) and adds
// it to y once.  No atomics.
template <typename T>
__global__ void k_carry_fixup(int64_t n_cta, const int32_t *__restrict__ carry_row,
                              const double *__restrict__ carry_val, T *__restrict__ y) {
    const int64_t c = gtid() >> 5;
    const int lane = threadIdx.x & 31;
    if (c >= n_cta) return;  // whole warp
    const int32_t r = carry_row[c];
    if (r < 0 || (c > 0 && carry_row[c - 1] == r)) return;
    double s = 0.0;
    for (int64_t c2 = c + lane; c2 < n_cta; c2 += 32) {
        if (carry_row[c2] != r) break;
        s += carry_val[c2];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) y[r] = static_cast<T>(static_cast<double>(y[r]) + s);
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

int64_t merge_ctas(int64_t n_rows, int64_t nnz) { return ceil_div(n_rows + nnz, kMergeItems); }
int64_t coo_ctas(int64_t nnz) { return ceil_div(nnz, kMergeItems); }

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

cudaError_t launch_csr_vector(int dtype, int g, int64_t count, const int32_t *rows, const int32_t *row_ptr,
                              const int32_t *col, const void *val, const void *x, void *y, cudaStream_t s) {
    if (dtype == SPMV_F64)
        return csr_vector_dispatch<double>(g, count, rows, row_ptr, col, static_cast<const double *>(val),
                                           static_cast<const double *>(x), static_cast<double *>(y), s);
    return csr_vector_dispatch<float>(g, count, rows, row_ptr, col, static_cast<const float *>(val),
                                      static_cast<const float *>(x), static_cast<float *>(y), s);
}

cudaError_t launch_segmented(int dtype, const Segmented &sg, const void *x, void *y, cudaStream_t s) {
    if (sg.kind == 0 || sg.n_cta <= 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>(sg.n_cta);
    if (sg.kind == 1 && sg.rows == nullptr)
        return launch_merge_path_identity(dtype, sg.n_rows, sg.nnz, sg.ptr, sg.col, sg.val, x, y, sg.carry_row,
                                          sg.carry_val, sg.n_cta, s, sg.part);
    if (sg.kind == 1) {
        if (dtype == SPMV_F64)
            k_merge_path<double><<<grid, kMergeThreads, 0, s>>>(sg.n_rows, sg.nnz, sg.ptr, sg.rows, sg.col,
                                                                static_cast<const double *>(sg.val),
                                                                static_cast<const double *>(x),
                                                                static_cast<double *>(y), sg.carry_row,
                                                                sg.carry_val, sg.accumulate, sg.part);
        else
            k_merge_path<float><<<grid, kMergeThreads, 0, s>>>(sg.n_rows, sg.nnz, sg.ptr, sg.rows, sg.col,
                                                               static_cast<const float *>(sg.val),
                                                               static_cast<const float *>(x),
                                                               static_cast<float *>(y), sg.carry_row,
                                                               sg.carry_val, sg.accumulate, sg.part);
    } else {
        if (dtype == SPMV_F64)
            k_coo<double><<<grid, kMergeThreads, 0, s>>>(sg.nnz, sg.coo_row, sg.col,
                                                         static_cast<const double *>(sg.val),
                                                         static_cast<const double *>(x), static_cast<double *>(y),
                                                         sg.carry_row, sg.carry_val, sg.accumulate);
        else
            k_coo<float><<<grid, kMergeThreads, 0, s>>>(sg.nnz, sg.coo_row, sg.col,
                                                        static_cast<const float *>(sg.val),
                                                        static_cast<const float *>(x), static_cast<float *>(y),
                                                        sg.carry_row, sg.carry_val, sg.accumulate);
    }
    return cudaGetLastError();
}

cudaError_t launch_merge_path_identity(int dtype, int64_t n_rows, int64_t nnz, const int32_t *ptr,
                                       const int32_t *col, const void *val, const void *x, void *y,
                                       int32_t *carry_row, double *carry_val, int64_t n_cta, cudaStream_t s,
                                       const int32_t *part) {
    if (n_cta <= 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>(n_cta);
    if (dtype == SPMV_F64)
        k_merge_path<double, true><<<grid, kMergeThreads, 0, s>>>(n_rows, nnz, ptr, nullptr, col,
                                                                  static_cast<const double *>(val),
                                                                  static_cast<const double *>(x),
                                                                  static_cast<double *>(y), carry_row, carry_val, 0,
                                                                  part);
    else
        k_merge_path<float, true><<<grid, kMergeThreads, 0, s>>>(n_rows, nnz, ptr, nullptr, col,
                                                                 static_cast<const float *>(val),
                                                                 static_cast<const float *>(x),
                                                                 static_cast<float *>(y), carry_row, carry_val, 0,
                                                                 part);
    return cudaGetLastError();
}

cudaError_t launch_carry_fixup(int dtype, const Segmented &sg, void *y, cudaStream_t s) {
    if (sg.kind == 0 || sg.n_cta <= 1) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>(ceil_div(sg.n_cta * 32, 256));
    if (dtype == SPMV_F64)
        k_carry_fixup<double><<<grid, 256, 0, s>>>(sg.n_cta, sg.carry_row, sg.carry_val, static_cast<double *>(y));
    else
        k_carry_fixup<float><<<grid, 256, 0, s>>>(sg.n_cta, sg.carry_row, sg.carry_val, static_cast<float *>(y));
    return cudaGetLastError();
}

}  // namespace spmv
