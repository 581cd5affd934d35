// Load-balanced passes: merge-path over a compact CSR (the HEC spill of HYB, or every
// row of the merge format and of the allocation-free entry point), load-balanced COO
// (the HYB spill), and the carry fix-up for rows that cross CTA boundaries.  Equal work shares per CTA regardless of row lengths
// (merge-path split named in the Trilinos issue on unpackAndCombine; load-balanced
// COO of the scite report's abstract).  No atomics.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_util.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

using namespace dev;

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
// merge-path over a compact CSR (the HEC spill, or every row)
// ---------------------------------------------------------------------------
// Shared-memory slot of path item i.  Thread t walks items t*kMergeIpt .. +kMergeIpt-1,
// so a plain layout puts the 32 lanes of a warp kMergeIpt words apart (an 8- or
// 16-way bank conflict).  One pad slot after every 32 (4-byte) / 16 (8-byte) items
// spreads the lanes over all banks; the staging writes stay conflict-free.
template <typename T>
__device__ __forceinline__ int skew(int i) {
    return i + (i >> (sizeof(T) == 8 ? 4 : 5));
}
template <typename T>
__host__ __device__ constexpr int skewed_size(int n) {
    return n + (n >> (sizeof(T) == 8 ? 4 : 5)) + 1;
}

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
        if (t < nk) s_prod[skew<T>(t)] = a[q] * ld_x_keep(x + c[q]);
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
    __shared__ T s_prod[skewed_size<T>(kMergeItems)];
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
    // One walk over the thread's path items.  A row that starts and ends inside
    // the thread is written at once; the first row the thread ends may have begun
    // in earlier threads, so its value waits for the CTA scan.
    int il = lo, kl = dl - lo;
    int first = -1;
    T first_val = T(0), run = T(0);
    for (int it = dl; it < dl_end; ++it) {
        if (il < ni && s_end[il] <= kl) {
            if (first < 0) {
                first = il;
                first_val = run;
            } else {
                const int32_t r = kIdentityRows ? static_cast<int32_t>(i0 + il) : __ldg(rows + i0 + il);
                y[r] = accumulate ? y[r] + run : run;
            }
            run = T(0);
            ++il;
        } else {
            run += s_prod[skew<T>(kl)];
            ++kl;
        }
    }
    const int flag = first >= 0;
    const T carry_in = seg_scan_exclusive<T, kMergeThreads>(flag, run, s_scan);
    if (flag) {
        const int32_t r = kIdentityRows ? static_cast<int32_t>(i0 + first) : __ldg(rows + i0 + first);
        const T v = carry_in + first_val;
        y[r] = accumulate ? y[r] + v : v;
    }
    if (threadIdx.x == kMergeThreads - 1) {
        const T inclusive = flag ? run : carry_in + run;
        const int64_t i = i0 + il;
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
    __shared__ T s_prod[skewed_size<T>(kMergeItems)];
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
    int first = -1;
    T first_val = T(0), run = T(0);
    for (int k = b; k < e; ++k) {
        run += s_prod[skew<T>(k)];
        if (s_row[k] != s_row[k + 1]) {
            if (first < 0) {
                first = k;
                first_val = run;
            } else {
                const int32_t r = s_row[k];
                y[r] = accumulate ? y[r] + run : run;
            }
            run = T(0);
        }
    }
    const int flag = first >= 0;
    const T carry_in = seg_scan_exclusive<T, kMergeThreads>(flag, run, s_scan);
    if (flag) {
        const int32_t r = s_row[first];
        const T v = carry_in + first_val;
        y[r] = accumulate ? y[r] + v : v;
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

}  // namespace

int64_t merge_ctas(int64_t n_rows, int64_t nnz) { return ceil_div(n_rows + nnz, kMergeItems); }
int64_t coo_ctas(int64_t nnz) { return ceil_div(nnz, kMergeItems); }

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
