// Device-side format builder: CSR validation, row-length histogram, stable
// radix partition / sort, exclusive scans, and the slot fills of the sliced
// (SELL-C-sigma / ELLPACK-R / HYB-ELL) and compact (long rows, HYB spill) parts.
//
// The "sort" and "pad" steps follow the pJDS construction of the GPGPU spMVM
// paper (arXiv 1112.5588, pJDS section, Fig. 1): rows ordered by length, longest
// first, then each block of rows padded to its longest row and stored column by
// column.  Everything runs on the GPU; only a handful of scalars go to the host.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "spmv_internal.cuh"

namespace spmv {
namespace {

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ int64_t ceil_div_dev(int64_t a, int64_t b) { return (a + b - 1) / b; }

__device__ __forceinline__ int64_t gtid() {
    return static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
}
__device__ __forceinline__ int64_t gstride() {
    return static_cast<int64_t>(gridDim.x) * blockDim.x;
}

inline unsigned grid_for(int64_t work, int block, int64_t cap = 1 << 20) {
    int64_t g = ceil_div(work, block);
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return static_cast<unsigned>(g);
}

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
__global__ void k_validate_rows(int64_t n, int64_t nnz, const int32_t *__restrict__ row_ptr,
                                int32_t *__restrict__ len, int32_t *status) {
    bool bad = false;
    int32_t my_max = 0;
    for (int64_t i = gtid(); i <= n; i += gstride()) {
        int32_t a = row_ptr[i];
        if (i == 0 && a != 0) bad = true;
        if (i == n && static_cast<int64_t>(a) != nnz) bad = true;
        if (i < n) {
            int32_t b = row_ptr[i + 1];
            int32_t l = b - a;
            if (b < a || a < 0 || static_cast<int64_t>(b) > nnz) {
                bad = true;
                l = 0;
            }
            len[i] = l;
            my_max = max(my_max, l);
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    my_max = __reduce_max_sync(0xffffffffu, my_max);
    if ((threadIdx.x & 31) == 0) {
        if (bad) atomicOr(&status[0], 1);
        if (my_max > 0) atomicMax(&status[2], my_max);
    }
}

__global__ void k_validate_cols(int64_t n, int64_t nnz, const int32_t *__restrict__ col,
                                int32_t *status) {
    bool bad = false;
    for (int64_t k = gtid(); k < nnz; k += gstride()) {
        int32_t c = col[k];
        if (c < 0 || static_cast<int64_t>(c) >= n) bad = true;
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&status[1], 1);
}

// ---------------------------------------------------------------------------
// histogram of row lengths (block-private in shared memory)
// ---------------------------------------------------------------------------
__global__ void k_histogram(int64_t n, const int32_t *__restrict__ len, int32_t threshold,
                            int64_t *__restrict__ hist, int64_t *__restrict__ stats) {
    __shared__ int s_hist[kHistCap + 1];
    __shared__ unsigned long long s_long, s_long_nnz;
    __shared__ int s_max_short;
    for (int t = threadIdx.x; t <= kHistCap; t += blockDim.x) s_hist[t] = 0;
    if (threadIdx.x == 0) {
        s_long = 0;
        s_long_nnz = 0;
        s_max_short = 0;
    }
    __syncthreads();
    unsigned long long my_long = 0, my_long_nnz = 0;
    int my_max = 0;
    for (int64_t i = gtid(); i < n; i += gstride()) {
        int l = len[i];
        int b = l < kHistCap ? l : kHistCap;
        unsigned peers = __match_any_sync(__activemask(), b);
        if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&s_hist[b], __popc(peers));
        if (threshold >= 0 && l > threshold) {
            ++my_long;
            my_long_nnz += static_cast<unsigned long long>(l);
        } else if (l > my_max) {
            my_max = l;
        }
    }
    if (my_long) {
        atomicAdd(&s_long, my_long);
        atomicAdd(&s_long_nnz, my_long_nnz);
    }
    if (my_max) atomicMax(&s_max_short, my_max);
    __syncthreads();
    for (int t = threadIdx.x; t <= kHistCap; t += blockDim.x)
        if (s_hist[t]) atomicAdd(reinterpret_cast<unsigned long long *>(&hist[t]),
                                 static_cast<unsigned long long>(s_hist[t]));
    if (threadIdx.x == 0) {
        if (s_long) {
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats[0]), s_long);
            atomicAdd(reinterpret_cast<unsigned long long *>(&stats[1]), s_long_nnz);
        }
        atomicMax(reinterpret_cast<unsigned long long *>(&stats[2]),
                  static_cast<unsigned long long>(s_max_short));
    }
}

__global__ void k_clip_long(int64_t n, const int32_t *__restrict__ len, int32_t threshold,
                            int32_t *__restrict__ out) {
    for (int64_t i = gtid(); i < n; i += gstride()) {
        int32_t l = len[i];
        out[i] = (threshold >= 0 && l > threshold) ? 0 : l;
    }
}

__global__ void k_mark_long(int64_t n_pos, const int32_t *__restrict__ perm, const int32_t *__restrict__ len,
                            int64_t n, int32_t threshold, int32_t *__restrict__ len_sorted) {
    for (int64_t p = gtid(); p < n_pos && p < n; p += gstride()) {
        const int32_t r = perm ? perm[p] : static_cast<int32_t>(p);
        if (len[r] > threshold) len_sorted[p] = -1;
    }
}

__global__ void k_min_len(int64_t n, const int32_t *__restrict__ len, int32_t K,
                          int32_t *__restrict__ out) {
    for (int64_t i = gtid(); i < n; i += gstride()) out[i] = min(len[i], K);
}

// ---------------------------------------------------------------------------
// exclusive scan of int64 (tiles of 4096: tile sums, one-CTA scan of the sums,
// tile-local scan plus offset)
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 512;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;

// Exclusive scan of one value per thread across the CTA; returns the CTA total.
template <int THREADS>
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t *warp_sums, int64_t &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int64_t up = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += up;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        constexpr int W = THREADS / 32;
        int64_t ws = lane < W ? warp_sums[lane] : 0;
        int64_t wi = ws;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int64_t up = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += up;
        }
        if (lane < W) warp_sums[lane] = wi - ws;  // exclusive prefix of each warp
        if (lane == W - 1) warp_sums[32] = wi;
    }
    __syncthreads();
    int64_t excl = warp_sums[warp] + inc - v;
    total = warp_sums[32];
    __syncthreads();
    return excl;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_tile_sums(const int64_t *__restrict__ in, int64_t n,
                                                                 int64_t *__restrict__ tile_sums) {
    __shared__ int64_t ws[33];
    int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile + static_cast<int64_t>(threadIdx.x) * kScanItems;
    int64_t s = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k)
        if (base + k < n) s += in[base + k];
    int64_t total;
    block_exclusive_scan<kScanThreads>(s, ws, total);
    if (threadIdx.x == 0) tile_sums[blockIdx.x] = total;
}

// one CTA: in-place exclusive scan of m values, chunked with a running carry
__global__ void __launch_bounds__(kScanThreads) k_scan_single(int64_t *__restrict__ data, int64_t m) {
    __shared__ int64_t ws[33];
    int64_t carry = 0;
    for (int64_t c0 = 0; c0 < m; c0 += kScanThreads) {
        int64_t i = c0 + threadIdx.x;
        int64_t v = i < m ? data[i] : 0;
        int64_t total;
        int64_t ex = block_exclusive_scan<kScanThreads>(v, ws, total);
        if (i < m) data[i] = carry + ex;
        carry += total;
    }
}

__global__ void __launch_bounds__(kScanThreads) k_scan_apply(const int64_t *__restrict__ in, int64_t n,
                                                             const int64_t *__restrict__ tile_off,
                                                             int64_t *__restrict__ out) {
    __shared__ int64_t ws[33];
    int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile + static_cast<int64_t>(threadIdx.x) * kScanItems;
    int64_t v[kScanItems];
    int64_t s = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        v[k] = (base + k < n) ? in[base + k] : 0;
        s += v[k];
    }
    int64_t total;
    int64_t run = block_exclusive_scan<kScanThreads>(s, ws, total) + tile_off[blockIdx.x];
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        if (base + k < n) out[base + k] = run;
        run += v[k];
    }
    // the final total goes to out[n]
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == kScanThreads - 1) out[n] = run;
}

__global__ void k_set_zero_total(int64_t *out) { out[0] = 0; }

// ---------------------------------------------------------------------------
// stable 8-bit counting pass (LSD radix step / bucket partition)
// A CTA owns a tile of 8 warps x 8 rounds x 32 items, in order; within a warp
// equal digits are ranked with __match_any_sync so the scatter keeps input order.
// ---------------------------------------------------------------------------
constexpr int kRadixThreads = 256;
constexpr int kRadixWarps = kRadixThreads / 32;
constexpr int kRadixRounds = 8;
constexpr int kRadixTile = kRadixThreads * kRadixRounds;

__global__ void __launch_bounds__(kRadixThreads) k_radix_count(const uint32_t *__restrict__ keys, int64_t n,
                                                               int shift, int64_t *__restrict__ counts,
                                                               int64_t nblocks) {
    __shared__ int hist[256];
    for (int t = threadIdx.x; t < 256; t += kRadixThreads) hist[t] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t base = static_cast<int64_t>(blockIdx.x) * kRadixTile + warp * (32 * kRadixRounds);
#pragma unroll
    for (int r = 0; r < kRadixRounds; ++r) {
        int64_t i = base + r * 32 + lane;
        bool valid = i < n;
        unsigned d = valid ? ((keys[i] >> shift) & 0xFFu) : 0x100u;
        unsigned peers = __match_any_sync(0xffffffffu, d);
        if (valid && lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
    }
    __syncthreads();
    for (int d = threadIdx.x; d < 256; d += kRadixThreads) counts[static_cast<int64_t>(d) * nblocks + blockIdx.x] = hist[d];
}

__global__ void __launch_bounds__(kRadixThreads) k_radix_scatter(
    const uint32_t *__restrict__ keys_in, const int32_t *__restrict__ vals_in, int64_t n, int shift,
    const int64_t *__restrict__ offsets, uint32_t *__restrict__ keys_out, int32_t *__restrict__ vals_out,
    int64_t nblocks) {
    __shared__ int wcount[kRadixWarps][256];
    __shared__ long long wpos[kRadixWarps][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int t = threadIdx.x; t < kRadixWarps * 256; t += kRadixThreads) (&wcount[0][0])[t] = 0;
    __syncthreads();
    int64_t base = static_cast<int64_t>(blockIdx.x) * kRadixTile + warp * (32 * kRadixRounds);
    uint32_t key[kRadixRounds];
    unsigned dig[kRadixRounds];
#pragma unroll
    for (int r = 0; r < kRadixRounds; ++r) {
        int64_t i = base + r * 32 + lane;
        bool valid = i < n;
        key[r] = valid ? keys_in[i] : 0u;
        dig[r] = valid ? ((key[r] >> shift) & 0xFFu) : 0x100u;
        unsigned peers = __match_any_sync(0xffffffffu, dig[r]);
        if (valid && lane == __ffs(peers) - 1) wcount[warp][dig[r]] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int d = threadIdx.x; d < 256; d += kRadixThreads) {
        long long run = offsets[static_cast<int64_t>(d) * nblocks + blockIdx.x];
        for (int w = 0; w < kRadixWarps; ++w) {
            wpos[w][d] = run;
            run += wcount[w][d];
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int r = 0; r < kRadixRounds; ++r) {
        int64_t i = base + r * 32 + lane;
        bool valid = i < n;
        unsigned peers = __match_any_sync(0xffffffffu, dig[r]);
        long long pos = 0;
        if (valid) pos = wpos[warp][dig[r]] + __popc(peers & lt);
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) wpos[warp][dig[r]] += __popc(peers);
        __syncwarp();
        if (valid) {
            keys_out[pos] = key[r];
            vals_out[pos] = vals_in ? vals_in[i] : static_cast<int32_t>(i);
        }
    }
}

// ---------------------------------------------------------------------------
// SELL ordering
// ---------------------------------------------------------------------------

// One CTA per window of sigma rows: rank = #longer rows + #equal rows before me.
__global__ void k_window_sort(const int32_t *__restrict__ len, int64_t n, int64_t sigma,
                              int32_t *__restrict__ perm) {
    extern __shared__ int s_len[];
    int64_t w0 = static_cast<int64_t>(blockIdx.x) * sigma;
    int cnt = static_cast<int>(min64(sigma, n - w0));
    for (int t = threadIdx.x; t < cnt; t += blockDim.x) s_len[t] = len[w0 + t];
    __syncthreads();
    for (int t = threadIdx.x; t < cnt; t += blockDim.x) {
        int lt = s_len[t];
        int rank = 0;
        for (int u = 0; u < cnt; ++u) {
            int lu = s_len[u];
            rank += (lu > lt) | ((lu == lt) & (u < t));
        }
        perm[w0 + rank] = static_cast<int32_t>(w0 + t);
    }
}

__global__ void k_sort_keys(const int32_t *__restrict__ len, int64_t n, int64_t sigma, int len_bits,
                            int32_t max_len, uint32_t *__restrict__ keys, int32_t *__restrict__ vals) {
    for (int64_t i = gtid(); i < n; i += gstride()) {
        uint32_t window = static_cast<uint32_t>(i / sigma);
        keys[i] = (window << len_bits) | static_cast<uint32_t>(max_len - len[i]);
        vals[i] = static_cast<int32_t>(i);
    }
}

__global__ void k_gather_sorted(const int32_t *__restrict__ len, const int32_t *__restrict__ perm,
                                int64_t n, int64_t n_pos, int32_t *__restrict__ len_sorted,
                                int32_t *__restrict__ perm_out) {
    for (int64_t p = gtid(); p < n_pos; p += gstride()) {
        if (p < n) {
            int32_t r = perm ? perm[p] : static_cast<int32_t>(p);
            len_sorted[p] = len[r];
            if (perm_out) perm_out[p] = r;
        } else {
            len_sorted[p] = 0;
            if (perm_out) perm_out[p] = -1;
        }
    }
}

// one warp per slice: width = max over its C rows
__global__ void k_slice_widths(const int32_t *__restrict__ len_sorted, int64_t n_slices, int32_t C, int32_t round_to,
                               int32_t *__restrict__ width, int64_t *__restrict__ size) {
    const int lane = threadIdx.x & 31;
    int64_t warp = gtid() >> 5;
    int64_t nwarps = gstride() >> 5;
    for (int64_t s = warp; s < n_slices; s += nwarps) {
        int m = 0;
        for (int r = lane; r < C; r += 32) m = max(m, len_sorted[s * C + r]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) {
            m = (m + round_to - 1) / round_to * round_to;  // whole groups for the interleaved layout
            width[s] = m;
            size[s] = static_cast<int64_t>(m) * C;
        }
    }
}

template <typename T>
__global__ void k_fill_sliced(int64_t n_pos, int log2C, uint32_t cmask, int64_t stride, int log2k_col, int log2k_val,
                              bool interleaved,
                              const int64_t *__restrict__ slice_ptr, const int32_t *__restrict__ width,
                              const int32_t *__restrict__ len_sorted, const int32_t *__restrict__ perm,
                              const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_in,
                              const T *__restrict__ val_in, int32_t *__restrict__ col_out,
                              T *__restrict__ val_out) {
    for (int64_t p = gtid(); p < n_pos; p += gstride()) {
        int64_t s = p >> log2C;
        int32_t w = width[s];
        const int64_t base = slice_ptr[s], q = static_cast<int64_t>(p & cmask);
        int32_t L = len_sorted[p];
        int64_t src = 0;
        if (L > 0) src = row_ptr[perm ? perm[p] : p];
        for (int32_t j = 0; j < w; ++j) {
            const int64_t sc = slot_of(base, q, j, stride, log2k_col, interleaved);
            const int64_t sv = slot_of(base, q, j, stride, log2k_val, interleaved);
            if (j < L) {
                col_out[sc] = col_in[src + j];
                val_out[sv] = val_in[src + j];
            } else {
                col_out[sc] = 0;
                val_out[sv] = T(0);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// partitions and compact copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t vector_bin(int32_t l, int32_t forced_g) {
    // bins 0..4 = 2, 4, 8, 16, 32 lanes per row: about eight entries a lane (one entry a
    // lane spent most of the time on per-lane overhead: 3.5x slower on the HMEp-shaped matrix)
    if (forced_g > 0) return static_cast<uint32_t>(__ffs(forced_g) - 2);
    if (l <= 16) return 0;
    if (l <= 32) return 1;
    if (l <= 64) return 2;
    if (l <= 128) return 3;
    return 4;
}

__global__ void k_bucket_keys(int64_t n, const int32_t *__restrict__ len, int mode, int32_t a,
                              int32_t forced_g, uint32_t *__restrict__ keys, int32_t *__restrict__ vals) {
    for (int64_t i = gtid(); i < n; i += gstride()) {
        int32_t l = len[i];
        uint32_t k;
        if (mode == 2) {
            k = (a >= 0 && l > a) ? 6u : vector_bin(l, forced_g);
        } else {
            k = (a >= 0 && l > a) ? 1u : 0u;
        }
        keys[i] = k;
        vals[i] = static_cast<int32_t>(i);
    }
}

__global__ void k_compact_sizes(int64_t m, const int32_t *__restrict__ rows, const int32_t *__restrict__ len,
                                int32_t offset, int64_t *__restrict__ size) {
    for (int64_t i = gtid(); i < m; i += gstride()) size[i] = static_cast<int64_t>(len[rows[i]]) - offset;
}

__global__ void k_int64_to_int32(const int64_t *__restrict__ in, int64_t n, int32_t *__restrict__ out) {
    for (int64_t i = gtid(); i < n; i += gstride()) out[i] = static_cast<int32_t>(in[i]);
}

// one warp per compact row
template <typename T>
__global__ void k_compact_copy(int64_t m, const int32_t *__restrict__ rows, const int32_t *__restrict__ row_ptr,
                               int32_t offset, const int32_t *__restrict__ col_in, const T *__restrict__ val_in,
                               const int64_t *__restrict__ cptr, int32_t *__restrict__ col_out,
                               T *__restrict__ val_out, int32_t *__restrict__ coo_row) {
    const int lane = threadIdx.x & 31;
    int64_t warp = gtid() >> 5;
    int64_t nwarps = gstride() >> 5;
    for (int64_t i = warp; i < m; i += nwarps) {
        int32_t r = rows[i];
        int64_t src = static_cast<int64_t>(row_ptr[r]) + offset;
        int64_t dst = cptr[i], cnt = cptr[i + 1] - cptr[i];
        for (int64_t k = lane; k < cnt; k += 32) {
            col_out[dst + k] = col_in[src + k];
            val_out[dst + k] = val_in[src + k];
            if (coo_row) coo_row[dst + k] = r;
        }
    }
}

// merge-path split of every CTA boundary (the same search the apply kernel would do)
__global__ void k_merge_partition(int64_t n_rows, int64_t nnz, const int32_t *__restrict__ ptr, int64_t n_cta,
                                  int32_t *__restrict__ part) {
    for (int64_t c = gtid(); c <= n_cta; c += gstride()) {
        const int64_t d = min64(c * kMergeItems, n_rows + nnz);
        int64_t lo = d - nnz > 0 ? d - nnz : 0, hi = min64(d, n_rows);
        while (lo < hi) {
            const int64_t mid = (lo + hi) >> 1;
            if (static_cast<int64_t>(ptr[mid + 1]) <= d - 1 - mid)
                lo = mid + 1;
            else
                hi = mid;
        }
        part[c] = static_cast<int32_t>(lo);
    }
}

__global__ void k_chunk_counts(int64_t m, const int32_t *__restrict__ ptr, int32_t chunk, int64_t *__restrict__ count) {
    for (int64_t i = gtid(); i < m; i += gstride()) {
        const int64_t len = static_cast<int64_t>(ptr[i + 1]) - ptr[i];
        count[i] = len > 0 ? ceil_div_dev(len, chunk) : 1;
    }
}

__global__ void k_chunk_fill(int64_t m, const int32_t *__restrict__ ptr, int32_t chunk, const int64_t *__restrict__ cptr,
                             int32_t *__restrict__ row_chunk_ptr, int32_t *__restrict__ chunk_begin,
                             int32_t *__restrict__ chunk_end, int32_t *__restrict__ chunk_row) {
    for (int64_t i = gtid(); i < m; i += gstride()) {
        const int32_t a = ptr[i], b = ptr[i + 1];
        int64_t c = cptr[i];
        const bool single = cptr[i + 1] - c == 1;
        row_chunk_ptr[i] = static_cast<int32_t>(c);
        if (i == m - 1) row_chunk_ptr[m] = static_cast<int32_t>(cptr[m]);
        int32_t k = a;
        do {
            const int32_t e = (b - k > chunk) ? k + chunk : b;
            chunk_begin[c] = k;
            chunk_end[c] = e;
            chunk_row[c] = single ? ~static_cast<int32_t>(i) : static_cast<int32_t>(i);
            ++c;
            k = e;
        } while (k < b);
    }
}

// ---------------------------------------------------------------------------
// to_csr
// ---------------------------------------------------------------------------
template <typename T>
__global__ void k_sliced_to_csr(int64_t n, int64_t n_pos, int log2C, uint32_t cmask, int64_t stride, int log2k_col,
                                int log2k_val, bool interleaved, const int64_t *__restrict__ slice_ptr, const int32_t *__restrict__ len_sorted,
                                const int32_t *__restrict__ perm, const int32_t *__restrict__ col,
                                const T *__restrict__ val, const int32_t *__restrict__ out_ptr,
                                int32_t *__restrict__ out_col, T *__restrict__ out_val) {
    for (int64_t p = gtid(); p < n_pos; p += gstride()) {
        int64_t r = perm ? perm[p] : p;
        if (r < 0 || r >= n) continue;
        int32_t L = len_sorted[p];
        const int64_t base = slice_ptr[p >> log2C], q = static_cast<int64_t>(p & cmask);
        int64_t dst = out_ptr[r];
        for (int32_t j = 0; j < L; ++j) {
            out_col[dst + j] = col[slot_of(base, q, j, stride, log2k_col, interleaved)];
            out_val[dst + j] = val[slot_of(base, q, j, stride, log2k_val, interleaved)];
        }
    }
}

template <typename T>
__global__ void k_segment_to_csr(int64_t m, const int32_t *__restrict__ rows, const int32_t *__restrict__ ptr,
                                 const int32_t *__restrict__ col, const T *__restrict__ val, int32_t dst_offset,
                                 const int32_t *__restrict__ out_ptr, int32_t *__restrict__ out_col,
                                 T *__restrict__ out_val) {
    const int lane = threadIdx.x & 31;
    int64_t warp = gtid() >> 5;
    int64_t nwarps = gstride() >> 5;
    for (int64_t i = warp; i < m; i += nwarps) {
        int64_t dst = static_cast<int64_t>(out_ptr[rows[i]]) + dst_offset;
        int64_t a = ptr[i], b = ptr[i + 1];
        for (int64_t k = a + lane; k < b; k += 32) {
            out_col[dst + (k - a)] = col[k];
            out_val[dst + (k - a)] = val[k];
        }
    }
}

// ---------------------------------------------------------------------------
// column reach of blocks of rows (the spmv_apply_host pipeline)
// ---------------------------------------------------------------------------
// One thread per sorted position walks its row's column-major slots; a warp's 32
// positions lie in one block (block is a multiple of 32), so a warp maximum and one
// atomic per warp give the block's largest column.
__global__ void k_block_max_col(int64_t n_pos, int log2C, uint32_t cmask, int64_t stride,
                                const int64_t *__restrict__ slice_ptr, const int32_t *__restrict__ len,
                                const int32_t *__restrict__ col, int64_t block, int32_t *__restrict__ out) {
    const int64_t p = gtid();
    int32_t m = -1;
    if (p < n_pos) {
        const int32_t w = len[p];
        const int64_t base = slice_ptr[p >> log2C] + (p & cmask);
        for (int32_t j = 0; j < w; ++j) m = max(m, col[base + j * stride]);
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0 && m >= 0 && p < n_pos) atomicMax(out + p / block, m);
}


}  // namespace

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_validate(int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col_idx,
                            int32_t *len, int32_t *status, cudaStream_t s) {
    k_validate_rows<<<grid_for(n + 1, kBlock, 65536), kBlock, 0, s>>>(n, nnz, row_ptr, len, status);
    if (nnz > 0)
        k_validate_cols<<<grid_for(nnz, kBlock, 65536), kBlock, 0, s>>>(n, nnz, col_idx, status);
    return cudaGetLastError();
}

cudaError_t launch_histogram(int64_t n, const int32_t *len, int32_t threshold, int64_t *hist,
                             int64_t *stats, cudaStream_t s) {
    cudaMemsetAsync(hist, 0, sizeof(int64_t) * (kHistCap + 1), s);
    cudaMemsetAsync(stats, 0, sizeof(int64_t) * 3, s);
    if (n > 0) k_histogram<<<grid_for(n, kBlock, 1024), kBlock, 0, s>>>(n, len, threshold, hist, stats);
    return cudaGetLastError();
}

cudaError_t launch_clip_long(int64_t n, const int32_t *len, int32_t threshold, int32_t *out, cudaStream_t s) {
    if (n > 0) k_clip_long<<<grid_for(n, kBlock, 65536), kBlock, 0, s>>>(n, len, threshold, out);
    return cudaGetLastError();
}

cudaError_t launch_mark_long(int64_t n_pos, const int32_t *perm, const int32_t *len, int64_t n, int32_t threshold,
                             int32_t *len_sorted, cudaStream_t s) {
    if (n_pos > 0 && n > 0)
        k_mark_long<<<grid_for(n_pos, kBlock, 65536), kBlock, 0, s>>>(n_pos, perm, len, n, threshold, len_sorted);
    return cudaGetLastError();
}

cudaError_t launch_min_len(int64_t n, const int32_t *len, int32_t K, int32_t *out, cudaStream_t s) {
    if (n > 0) k_min_len<<<grid_for(n, kBlock, 65536), kBlock, 0, s>>>(n, len, K, out);
    return cudaGetLastError();
}

int64_t scan_temp_elems(int64_t n) { return ceil_div(n, kScanTile) + 1; }

cudaError_t launch_exclusive_scan(const int64_t *in, int64_t n, int64_t *out, int64_t *temp, cudaStream_t s) {
    if (n <= 0) {
        k_set_zero_total<<<1, 1, 0, s>>>(out);
        return cudaGetLastError();
    }
    int64_t tiles = ceil_div(n, kScanTile);
    k_scan_tile_sums<<<static_cast<unsigned>(tiles), kScanThreads, 0, s>>>(in, n, temp);
    k_scan_single<<<1, kScanThreads, 0, s>>>(temp, tiles);
    k_scan_apply<<<static_cast<unsigned>(tiles), kScanThreads, 0, s>>>(in, n, temp, out);
    return cudaGetLastError();
}

int64_t radix_blocks(int64_t n) { return n > 0 ? ceil_div(n, kRadixTile) : 1; }

cudaError_t launch_radix_pass(const uint32_t *keys_in, const int32_t *vals_in, int64_t n, int shift,
                              uint32_t *keys_out, int32_t *vals_out, int64_t *counts, int64_t *offsets,
                              int64_t *scan_temp, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    int64_t nb = radix_blocks(n);
    k_radix_count<<<static_cast<unsigned>(nb), kRadixThreads, 0, s>>>(keys_in, n, shift, counts, nb);
    cudaError_t e = launch_exclusive_scan(counts, 256 * nb, offsets, scan_temp, s);
    if (e != cudaSuccess) return e;
    k_radix_scatter<<<static_cast<unsigned>(nb), kRadixThreads, 0, s>>>(keys_in, vals_in, n, shift, offsets,
                                                                        keys_out, vals_out, nb);
    return cudaGetLastError();
}

cudaError_t launch_window_sort(const int32_t *len, int64_t n, int64_t sigma, int32_t *perm, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    int64_t windows = ceil_div(n, sigma);
    int threads = static_cast<int>(sigma < 1024 ? ((sigma + 31) / 32) * 32 : 1024);
    k_window_sort<<<static_cast<unsigned>(windows), threads, sizeof(int) * sigma, s>>>(len, n, sigma, perm);
    return cudaGetLastError();
}

cudaError_t launch_sort_keys(const int32_t *len, int64_t n, int64_t sigma, int len_bits, int32_t max_len,
                             uint32_t *keys, int32_t *vals, cudaStream_t s) {
    if (n > 0) k_sort_keys<<<grid_for(n, kBlock, 65536), kBlock, 0, s>>>(len, n, sigma, len_bits, max_len, keys, vals);
    return cudaGetLastError();
}

cudaError_t launch_gather_sorted(const int32_t *len, const int32_t *perm, int64_t n, int64_t n_pos,
                                 int32_t *len_sorted, int32_t *perm_out, cudaStream_t s) {
    if (n_pos > 0)
        k_gather_sorted<<<grid_for(n_pos, kBlock, 65536), kBlock, 0, s>>>(len, perm, n, n_pos, len_sorted, perm_out);
    return cudaGetLastError();
}

cudaError_t launch_slice_widths(const int32_t *len_sorted, int64_t n_slices, int32_t C, int32_t *width,
                                int64_t *size, cudaStream_t s, int32_t round_to) {
    if (n_slices > 0)
        k_slice_widths<<<grid_for(n_slices * 32, kBlock, 65536), kBlock, 0, s>>>(len_sorted, n_slices, C, round_to,
                                                                                width, size);
    return cudaGetLastError();
}

cudaError_t launch_fill_sliced(int dtype, const Sliced &sl, const int32_t *row_ptr, const int32_t *col_in,
                               const void *val_in, cudaStream_t s) {
    if (sl.n_pos <= 0 || sl.slots <= 0) return cudaSuccess;
    unsigned g = grid_for(sl.n_pos, kBlock, 1 << 20);
    if (dtype == SPMV_F64)
        k_fill_sliced<double><<<g, kBlock, 0, s>>>(sl.n_pos, sl.log2C, sl.cmask, sl.stride, sl.log2k_col, sl.log2k_val,
                                                   sl.interleaved,
                                                   sl.slice_ptr, sl.width,
                                                   sl.len, sl.perm, row_ptr, col_in,
                                                   static_cast<const double *>(val_in), sl.col,
                                                   static_cast<double *>(sl.val));
    else
        k_fill_sliced<float><<<g, kBlock, 0, s>>>(sl.n_pos, sl.log2C, sl.cmask, sl.stride, sl.log2k_col, sl.log2k_val,
                                                  sl.interleaved,
                                                  sl.slice_ptr, sl.width,
                                                  sl.len, sl.perm, row_ptr, col_in,
                                                  static_cast<const float *>(val_in), sl.col,
                                                  static_cast<float *>(sl.val));
    return cudaGetLastError();
}

cudaError_t launch_bucket_keys(int64_t n, const int32_t *len, int mode, int32_t a, int32_t forced_g,
                               uint32_t *keys, int32_t *vals, cudaStream_t s) {
    if (n > 0) k_bucket_keys<<<grid_for(n, kBlock, 65536), kBlock, 0, s>>>(n, len, mode, a, forced_g, keys, vals);
    return cudaGetLastError();
}

cudaError_t launch_compact_sizes(int64_t m, const int32_t *rows, const int32_t *len, int32_t offset,
                                 int64_t *size, cudaStream_t s) {
    if (m > 0) k_compact_sizes<<<grid_for(m, kBlock, 65536), kBlock, 0, s>>>(m, rows, len, offset, size);
    return cudaGetLastError();
}

cudaError_t launch_int64_to_int32(const int64_t *in, int64_t n, int32_t *out, cudaStream_t s) {
    if (n > 0) k_int64_to_int32<<<grid_for(n, kBlock, 65536), kBlock, 0, s>>>(in, n, out);
    return cudaGetLastError();
}

cudaError_t launch_compact_copy(int dtype, int64_t m, const int32_t *rows, const int32_t *row_ptr, int32_t offset,
                                const int32_t *col_in, const void *val_in, const int64_t *cptr, int32_t *col_out,
                                void *val_out, int32_t *coo_row, cudaStream_t s) {
    if (m <= 0) return cudaSuccess;
    unsigned g = grid_for(m * 32, kBlock, 1 << 20);
    if (dtype == SPMV_F64)
        k_compact_copy<double><<<g, kBlock, 0, s>>>(m, rows, row_ptr, offset, col_in,
                                                    static_cast<const double *>(val_in), cptr, col_out,
                                                    static_cast<double *>(val_out), coo_row);
    else
        k_compact_copy<float><<<g, kBlock, 0, s>>>(m, rows, row_ptr, offset, col_in,
                                                   static_cast<const float *>(val_in), cptr, col_out,
                                                   static_cast<float *>(val_out), coo_row);
    return cudaGetLastError();
}

cudaError_t launch_merge_partition(int64_t n_rows, int64_t nnz, const int32_t *ptr, int64_t n_cta, int32_t *part,
                                   cudaStream_t s) {
    k_merge_partition<<<grid_for(n_cta + 1, kBlock, 65536), kBlock, 0, s>>>(n_rows, nnz, ptr, n_cta, part);
    return cudaGetLastError();
}

cudaError_t launch_chunk_counts(int64_t m, const int32_t *ptr, int32_t chunk, int64_t *count, cudaStream_t s) {
    if (m > 0) k_chunk_counts<<<grid_for(m, kBlock, 65536), kBlock, 0, s>>>(m, ptr, chunk, count);
    return cudaGetLastError();
}

cudaError_t launch_chunk_fill(int64_t m, const int32_t *ptr, int32_t chunk, const int64_t *cptr,
                              int32_t *row_chunk_ptr, int32_t *chunk_begin, int32_t *chunk_end, int32_t *chunk_row,
                              cudaStream_t s) {
    if (m > 0)
        k_chunk_fill<<<grid_for(m, kBlock, 65536), kBlock, 0, s>>>(m, ptr, chunk, cptr, row_chunk_ptr, chunk_begin,
                                                                  chunk_end, chunk_row);
    return cudaGetLastError();
}

cudaError_t launch_sliced_to_csr(int dtype, int64_t n, const Sliced &sl, const int32_t *out_ptr, int32_t *out_col,
                                 void *out_val, cudaStream_t s) {
    if (!sl.present || sl.n_pos <= 0) return cudaSuccess;
    unsigned g = grid_for(sl.n_pos, kBlock, 1 << 20);
    if (dtype == SPMV_F64)
        k_sliced_to_csr<double><<<g, kBlock, 0, s>>>(n, sl.n_pos, sl.log2C, sl.cmask, sl.stride, sl.log2k_col,
                                                     sl.log2k_val, sl.interleaved, sl.slice_ptr,
                                                     sl.len, sl.perm, sl.col, static_cast<const double *>(sl.val),
                                                     out_ptr, out_col, static_cast<double *>(out_val));
    else
        k_sliced_to_csr<float><<<g, kBlock, 0, s>>>(n, sl.n_pos, sl.log2C, sl.cmask, sl.stride, sl.log2k_col,
                                                    sl.log2k_val, sl.interleaved, sl.slice_ptr,
                                                    sl.len, sl.perm, sl.col, static_cast<const float *>(sl.val),
                                                    out_ptr, out_col, static_cast<float *>(out_val));
    return cudaGetLastError();
}

cudaError_t launch_segment_to_csr(int dtype, const Segmented &sg, const int32_t *out_ptr, int32_t *out_col,
                                  void *out_val, cudaStream_t s) {
    if (sg.kind == 0 || sg.n_rows <= 0) return cudaSuccess;  // kinds 1-3 all hold a compact CSR
    unsigned g = grid_for(sg.n_rows * 32, kBlock, 1 << 20);
    if (dtype == SPMV_F64)
        k_segment_to_csr<double><<<g, kBlock, 0, s>>>(sg.n_rows, sg.rows, sg.ptr, sg.col,
                                                      static_cast<const double *>(sg.val), sg.dst_offset, out_ptr,
                                                      out_col, static_cast<double *>(out_val));
    else
        k_segment_to_csr<float><<<g, kBlock, 0, s>>>(sg.n_rows, sg.rows, sg.ptr, sg.col,
                                                     static_cast<const float *>(sg.val), sg.dst_offset, out_ptr,
                                                     out_col, static_cast<float *>(out_val));
    return cudaGetLastError();
}

cudaError_t launch_block_max_col(const Sliced &sl, int64_t block, int32_t *out, cudaStream_t s) {
    if (!sl.present || sl.n_pos <= 0) return cudaSuccess;
    if (block <= 0 || block % 32 != 0 || sl.group != 1 || sl.interleaved || sl.vec) return cudaErrorInvalidValue;
    k_block_max_col<<<grid_for(sl.n_pos, kBlock, INT_MAX), kBlock, 0, s>>>(sl.n_pos, sl.log2C, sl.cmask, sl.stride,
                                                                          sl.slice_ptr, sl.len, sl.col, block, out);
    return cudaGetLastError();
}

}  // namespace spmv
