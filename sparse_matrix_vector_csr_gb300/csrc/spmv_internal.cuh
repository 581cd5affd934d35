// Internal declarations of the sm_103a SpMV library: handle layout, launch
// constants and the host-side launchers of the build and apply kernels.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "spmv.h"

namespace spmv {

// ----------------------------------------------------------------------------
// launch constants
// ----------------------------------------------------------------------------
constexpr int kBlock = 256;                 // generic 1-D kernels
constexpr int kSellBlock = 256;             // sliced apply
constexpr int kMergeThreads = 256;          // merge-path / COO segmented pass
constexpr int kMergeIpt = 8;                // path items per thread
constexpr int kMergeItems = kMergeThreads * kMergeIpt;
constexpr int kHistCap = 4096;              // row-length histogram: buckets 0..kHistCap-1, last = ">= kHistCap"
constexpr int kWindowSortMax = 2048;        // SELL windows up to this many rows are sorted in one CTA
constexpr int kShortRow = 8;                 // rows this short on a small matrix: whole-row loads
constexpr int64_t kShortRowsMax = 152 * 2048;  // "small": fewer row positions than one wave of threads
constexpr int kSplitChunk = 2048;           // entries per warp in the row-split pass for long rows (float32)
constexpr int kSplitChunk64 = 4096;         // float64 chunks fused with one-thread-per-row slices
constexpr int kMaxHostBlocks = 1024;         // row blocks of the spmv_apply_host pipeline, at most
constexpr int kTailMaxW = 4;                 // narrow-tail table: slice widths 0..kTailMaxW

// ----------------------------------------------------------------------------
// format parts
// ----------------------------------------------------------------------------

// Sliced column-major storage: SELL-C-sigma, ELLPACK-R, or the ELL part of HYB.
// Sorted position p lives in slice s = p >> log2C at row r = p & cmask of the
// slice; its j-th stored entry sits at slot slice_ptr[s] + j * stride + r.
// SELL: stride = C.  ELL (one slice): log2C = 31, cmask = 0x7fffffff, stride = ld.
struct Sliced {
    bool present = false;
    int64_t n_pos = 0;        // positions: n rounded up to C (SELL) or to ld (ELL)
    int log2C = 0;
    uint32_t cmask = 0;
    int64_t stride = 0;
    int32_t C = 0;
    int64_t sigma = 1;
    int64_t ld = 0;
    int64_t n_slices = 0;
    int64_t slots = 0;           // allocated slot count (sum of C * width)
    int64_t padded_entries = 0;  // sum over real rows of their slice width
    int64_t stored_entries = 0;  // entries actually held (sum of len)
    int32_t max_width = 0;
    bool keep_x = false;           // gather x with an L2 evict-last policy
    int32_t group = 1;             // threads per row in the apply (1, 2, 4, ..., 32)
    int log2g = 0;
    int group_mode = 0;            // with group > 1: 0 row-grouped, 1 interleaved, 2 column-grouped
    bool interleaved = false;      // slot layout, see slot_of() (group_mode 1 or vec)
    bool vec = false;              // one thread per row reading 16-byte vectors of its row
    int log2k_col = 0;             // interleaved slots: index groups of 2^log2k_col
    int log2k_val = 0;             //                    value groups of 2^log2k_val
    bool staged = false;           // apply by sellb.cu's bulk-staged kernel
    bool pdl = true;               // launch with programmatic dependent launch (off for views
                                   // whose start waits on an event of another stream)
    // Narrow tail of a globally sorted SELL-32 layout (sigma >= n, one thread per row,
    // column-major slots), where slice widths never increase: for w = 0..kTailMaxW the
    // slices of width <= w are those from tail_slice[w] on (n_slices if none), and the
    // first of them starts at slot tail_slot[w].  has_tail is false for other layouts.
    bool has_tail = false;
    int64_t tail_slice[kTailMaxW + 1] = {};
    int64_t tail_slot[kTailMaxW + 1] = {};
    // CTAs for the narrow tail when no long-row chunks share the launch (12 per SM): each
    // loops over the tail instead of a short-lived CTA per 512 rows
    int64_t tail_cap = 0;
    int64_t *slice_ptr = nullptr;  // [n_slices + 1]
    int32_t *width = nullptr;      // [n_slices]
    int32_t *len = nullptr;        // [n_pos] entries stored at each position
    int32_t *perm = nullptr;       // [n_pos] original row (-1 = padding); nullptr = identity
    int32_t *col = nullptr;        // [slots]
    void *val = nullptr;           // [slots]
};

// Slot of entry j of the row held at in-slice position q of a slice starting at
// `base` (stride = C for SELL, the leading dimension for ELLPACK-R / HYB-ELL).
// Column-major ("row-grouped"): base + j * stride + q, so entry j of the slice's
// rows is contiguous.  Interleaved ("column-grouped", for g threads per row): the
// entries of a row come in groups of g = 2^log2g that sit side by side,
// base + ((j >> log2g) * stride + q) * g + (j & (g - 1)), so the g threads of a row
// read g adjacent values and a warp reads 32 consecutive ones.  Slice widths are
// then whole groups.
__host__ __device__ inline int64_t slot_of(int64_t base, int64_t q, int64_t j, int64_t stride, int log2g,
                                           bool interleaved) {
    return interleaved ? base + ((((j >> log2g) * stride + q) << log2g) | (j & ((int64_t{1} << log2g) - 1)))
                       : base + j * stride + q;
}

// Rows handled by the segmented pass: the long rows taken out of a format, or
// the HYB spill.  kind 1 = compact CSR walked by merge-path, kind 2 = COO,
// kind 3 = compact CSR cut into row chunks (row-split pass).
struct Segmented {
    int kind = 0;
    int64_t n_rows = 0;
    int64_t nnz = 0;
    int32_t *rows = nullptr;     // [n_rows] original row of each compact row (increasing)
    int32_t *ptr = nullptr;      // [n_rows + 1] compact row pointer
    int32_t *coo_row = nullptr;  // [nnz] original row of every entry (kind 2)
    int32_t *col = nullptr;      // [nnz]
    void *val = nullptr;         // [nnz]
    int64_t n_cta = 0;
    int32_t *carry_row = nullptr;  // [n_cta] row left open at the end of each CTA (-1 = none)
    double *carry_val = nullptr;   // [n_cta] its partial sum
    int32_t *part = nullptr;       // [n_cta + 1] merge-path split of every CTA boundary (kind 1)
    int64_t n_chunks = 0;          // kind 3: chunks of at most `chunk` entries, none crossing a row
    int32_t chunk = 0;             // kind 3: kSplitChunk64 or kSplitChunk entries per chunk
    int32_t *chunk_begin = nullptr;    // [n_chunks] first entry of each chunk (compact CSR index)
    int32_t *chunk_end = nullptr;      // [n_chunks] one past its last entry
    int32_t *row_chunk_ptr = nullptr;  // [n_rows + 1] chunks of compact row i
    int32_t *chunk_row = nullptr;      // [n_chunks] compact row of the chunk; ~row if it is the row's only chunk
    int64_t n_multi = 0;               // compact rows cut into more than one chunk
    int32_t *done = nullptr;           // [n_rows] chunks of the row finished in the running apply
    double *partial = nullptr;         // [n_chunks * 8] partial sums, up to 8 right-hand sides
    // carry_row, carry_val, done and partial are written by the apply: the handle keeps
    // them per stream (ApplyScratch) and each apply fills in its own stream's set
    int accumulate = 1;            // 1: add into y (y written before), 0: write y
    int32_t dst_offset = 0;        // in-row position of the first held entry (K for the spill)
};

// The arrays an apply writes besides y, one set per stream a handle is applied on:
// applies of one handle on different streams may overlap on the GPU, and each works
// in its own set, while applies on one stream run in stream order and share it.
struct ApplyScratch {
    cudaStream_t stream = nullptr;
    int32_t *carry_row = nullptr;  // [seg.n_cta]   merge-path / COO carries
    double *carry_val = nullptr;   // [seg.n_cta]
    double *partial = nullptr;     // [seg.n_chunks * 8] row-split chunk partials
    int32_t *done = nullptr;       // [seg.n_rows]  row-split counters, zero between applies
    void *tmp_x = nullptr;         // [n] columns of scaled / multi-vector applies without a
    void *tmp_y = nullptr;         // [n] fused path (allocated on first need)
    void *x_stage = nullptr;       // [n] spmv_apply_host staging (allocated on first need)
    void *y_stage = nullptr;       // [n]
};

// One CSR-vector launch: g lanes per row over rows bin_rows[offset, offset + count),
// or rows [0, count) when the handle has no bin list.
struct Bin {
    int g = 0;
    int64_t count = 0;
    int64_t offset = 0;
};

}  // namespace spmv

struct spmv_handle_s {
    int64_t n = 0;
    int64_t nnz = 0;
    int dtype = SPMV_F64;
    int format = SPMV_FMT_AUTO;
    int requested_format = SPMV_FMT_AUTO;
    spmv_format_params params{};
    int device = 0;
    int32_t max_len = 0;
    double mean_len = 0.0;

    // the input CSR (row pointer always kept; columns/values for CSR-vector)
    int32_t *row_ptr = nullptr;
    int32_t *csr_col = nullptr;
    void *csr_val = nullptr;

    spmv::Sliced sliced;
    spmv::Segmented seg;
    std::vector<spmv::Bin> bins;
    int32_t *bin_rows = nullptr;

    int64_t n_long_rows = 0;
    int64_t long_nnz = 0;
    int32_t K = 0;

    // per-stream apply scratch; scratch_mutex guards the list and `allocations`
    // after the build
    std::mutex scratch_mutex;
    std::vector<std::unique_ptr<spmv::ApplyScratch>> scratch;
    // spmv_apply_host pipeline: decided by the first call (0 = not yet, 1 = pipelined,
    // -1 = not pipelined); row positions per block; for every block, the last piece of x
    // its columns reach (-1 = the block has no entries); copy streams and events.
    // host_mutex serialises the pipeline's set-up and its calls (they share the copy
    // streams and events).
    std::mutex host_mutex;
    int host_pipe = 0;
    int64_t host_block = 0;
    std::vector<int32_t> host_need;
    std::atomic<int> host_last_blocks{-1};  // blocks of the last spmv_apply_host call (0 = unpipelined)
    cudaStream_t host_in = nullptr;
    cudaStream_t host_out = nullptr;
    std::vector<cudaEvent_t> host_events;

    // permuted basis (spmv_build_permuted): position -> original index; nullptr = identity
    int32_t *basis_perm = nullptr;
    int ordering = SPMV_ORDER_NATURAL;

    int *dev_err = nullptr;  // device flag: a bounded wait of an apply kernel ran out
    std::vector<std::string> kernels;  // launch sequence of one apply
    std::vector<void *> allocations;
};

namespace spmv {

// ----------------------------------------------------------------------------
// error state (thread-local) -- api.cu
// ----------------------------------------------------------------------------
int set_error(int status, const std::string &msg);
int set_cuda_error(cudaError_t err, const char *what);

// ----------------------------------------------------------------------------
// device memory of the library -- api.cu
// ----------------------------------------------------------------------------
// Every device allocation of the library goes through these: they keep the count and
// size of what it holds (spmv_device_memory) and fail an allocation on request (the
// SPMV_FAIL_ALLOC environment variable, a host-side fault injector for tests).
cudaError_t lib_malloc(void **p, size_t bytes);
cudaError_t lib_malloc_async(void **p, size_t bytes, cudaStream_t s);
void lib_free(void *p);
void lib_free_async(void *p, cudaStream_t s);

#define SPMV_TRY_CUDA(expr)                                              \
    do {                                                                 \
        cudaError_t spmv_err__ = (expr);                                 \
        if (spmv_err__ != cudaSuccess) return ::spmv::set_cuda_error(spmv_err__, #expr); \
    } while (0)

#define SPMV_TRY(expr)                      \
    do {                                    \
        int spmv_st__ = (expr);             \
        if (spmv_st__ != SPMV_OK) return spmv_st__; \
    } while (0)

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
// [a, a + abytes) and [b, b + bbytes) share a byte
inline bool spans_overlap(const void *a, size_t abytes, const void *b, size_t bbytes) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + bbytes && pb < pa + abytes;
}
// p is device memory of the current device (or managed memory, reachable from every
// device); memory of another GPU, host memory and unknown addresses are not -- api.cu
bool device_memory_here(const void *p);
inline size_t value_bytes(int dtype) { return dtype == SPMV_F64 ? 8 : 4; }

// ----------------------------------------------------------------------------
// build launchers -- build.cu.  All enqueue on `s`; none synchronises.
// ----------------------------------------------------------------------------

// status[0]: bad row_ptr flag, status[1]: bad column flag, status[2]: max row length.
cudaError_t launch_validate(int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col_idx,
                            int32_t *len, int32_t *status, cudaStream_t s);
// hist[kHistCap + 1] of min(len, kHistCap); stats[0] = rows with len > threshold,
// stats[1] = their entries, stats[2] = longest row with len <= threshold.
cudaError_t launch_histogram(int64_t n, const int32_t *len, int32_t threshold, int64_t *hist,
                             int64_t *stats, cudaStream_t s);
// out[i] = 0 for rows longer than threshold (threshold < 0: no cut), else len[i].
cudaError_t launch_clip_long(int64_t n, const int32_t *len, int32_t threshold, int32_t *out,
                             cudaStream_t s);
// len_sorted[p] = -1 where the row at sorted position p is longer than threshold
cudaError_t launch_mark_long(int64_t n_pos, const int32_t *perm, const int32_t *len, int64_t n, int32_t threshold,
                             int32_t *len_sorted, cudaStream_t s);
cudaError_t launch_min_len(int64_t n, const int32_t *len, int32_t K, int32_t *out, cudaStream_t s);

// Exclusive scan of int64 values: out[i] = sum in[0..i), out has n+1 entries.
// Needs scan_temp_elems(n) int64 of temporary storage.
int64_t scan_temp_elems(int64_t n);
cudaError_t launch_exclusive_scan(const int64_t *in, int64_t n, int64_t *out, int64_t *temp,
                                  cudaStream_t s);

// Stable partition / radix sort machinery (8-bit digits).
int64_t radix_blocks(int64_t n);
// One stable counting pass on digit (key >> shift) & 255.  counts/offsets need
// 256 * radix_blocks(n) + 1 int64; scan_temp needs scan_temp_elems(256*blocks).
cudaError_t launch_radix_pass(const uint32_t *keys_in, const int32_t *vals_in, int64_t n, int shift,
                              uint32_t *keys_out, int32_t *vals_out, int64_t *counts,
                              int64_t *offsets, int64_t *scan_temp, cudaStream_t s);

// SELL ordering.  Window sort for sigma <= kWindowSortMax.
cudaError_t launch_window_sort(const int32_t *len, int64_t n, int64_t sigma, int32_t *perm,
                               cudaStream_t s);
// key[i] = (i / sigma) << len_bits | (max_len - len[i]); val[i] = i.
cudaError_t launch_sort_keys(const int32_t *len, int64_t n, int64_t sigma, int len_bits,
                             int32_t max_len, uint32_t *keys, int32_t *vals, cudaStream_t s);
// len_sorted[p] = len[perm[p]] for p < n, 0 beyond; perm_out[p] = perm[p] or -1.
cudaError_t launch_gather_sorted(const int32_t *len, const int32_t *perm, int64_t n, int64_t n_pos,
                                 int32_t *len_sorted, int32_t *perm_out, cudaStream_t s);
// width[s] = max len_sorted over the slice, rounded up to a multiple of round_to;
// size[s] = C * width[s].
cudaError_t launch_slice_widths(const int32_t *len_sorted, int64_t n_slices, int32_t C,
                                int32_t *width, int64_t *size, cudaStream_t s, int32_t round_to = 1);
// Slot fill from CSR (values of `dtype`), padding slots get column 0 / value 0.
cudaError_t launch_fill_sliced(int dtype, const Sliced &sl, const int32_t *row_ptr,
                               const int32_t *col_in, const void *val_in, cudaStream_t s);

// bucket[i] = pred(len[i]) for partitions.
// mode 0: long rows (len > a); mode 1: HYB spill rows (len > a);
// mode 2: CSR-vector bin id (6 = long row, beyond a) for len.
cudaError_t launch_bucket_keys(int64_t n, const int32_t *len, int mode, int32_t a, int32_t forced_g,
                               uint32_t *keys, int32_t *vals, cudaStream_t s);
// size[i] = len[rows[i]] - offset
cudaError_t launch_compact_sizes(int64_t m, const int32_t *rows, const int32_t *len, int32_t offset,
                                 int64_t *size, cudaStream_t s);
cudaError_t launch_int64_to_int32(const int64_t *in, int64_t n, int32_t *out, cudaStream_t s);
// Copy entries [row_ptr[r] + offset, row_ptr[r+1]) of each listed row into compact arrays.
cudaError_t launch_compact_copy(int dtype, int64_t m, const int32_t *rows, const int32_t *row_ptr,
                                int32_t offset, const int32_t *col_in, const void *val_in,
                                const int64_t *cptr, int32_t *col_out, void *val_out,
                                int32_t *coo_row, cudaStream_t s);

// row chunks of a compact CSR: count[i] = ceil(len_i / chunk) (at least 1)
cudaError_t launch_chunk_counts(int64_t m, const int32_t *ptr, int32_t chunk, int64_t *count, cudaStream_t s);
cudaError_t launch_chunk_fill(int64_t m, const int32_t *ptr, int32_t chunk, const int64_t *cptr, int32_t *row_chunk_ptr,
                              int32_t *chunk_begin, int32_t *chunk_end, int32_t *chunk_row, cudaStream_t s);


// to_csr
cudaError_t launch_sliced_to_csr(int dtype, int64_t n, const Sliced &sl, const int32_t *out_ptr,
                                 int32_t *out_col, void *out_val, cudaStream_t s);
cudaError_t launch_segment_to_csr(int dtype, const Segmented &sg, const int32_t *out_ptr,
                                  int32_t *out_col, void *out_val, cudaStream_t s);

// ----------------------------------------------------------------------------
// apply launchers -- sell.cu, vector.cu, merge.cu
// ----------------------------------------------------------------------------
// y = alpha * (A x) + beta * y instead of y = A x (y not read when beta == 0)
struct Scale {
    double alpha;
    double beta;
};
// split: the row-split pass of the long rows (kind 3) to run in the same launch, or nullptr;
// scale: nullptr for y = A x
cudaError_t launch_sell_apply(int dtype, const Sliced &sl, int64_t n, const Segmented *split, const void *x, void *y,
                              cudaStream_t s, const Scale *scale = nullptr);
// bulk-staged SELL-32 apply (sellb.cu): one thread per row, column-major slots; err is
// the handle's device flag, set when a bounded wait runs out
bool sell_staged_supported(const Sliced &sl);
cudaError_t launch_sell_staged(int dtype, const Sliced &sl, int64_t n, const void *x, void *y, int *err,
                               cudaStream_t s, const Scale *scale = nullptr);
// row positions the sliced apply hands to its narrow-tail path (0 = none) -- sell.cu
int64_t sell_tail_positions(const Sliced &sl);
cudaError_t launch_csr_vector(int dtype, int g, int64_t count, const int32_t *rows,
                              const int32_t *row_ptr, const int32_t *col, const void *val,
                              const void *x, void *y, cudaStream_t s);
cudaError_t launch_segmented(int dtype, const Segmented &sg, const void *x, void *y, cudaStream_t s);
cudaError_t launch_carry_fixup(int dtype, const Segmented &sg, void *y, cudaStream_t s);
// multi-vector apply on the sliced layout (NV = 2, 4, 8 right-hand sides, row-major X/Y) -- sellmm.cu
bool sell_multi_supported(const Sliced &sl);
// Orderings of the permuted basis (order.cu).  compute_ordering fills perm (new -> old)
// for an already validated CSR (max_len = its longest row); permute_csr writes
// B = P A P^T (row i of B = row perm[i] of A, columns renamed through the inverse).
int compute_ordering(int ordering, int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col,
                     int32_t max_len, const int32_t *user_perm, int32_t *perm, cudaStream_t s);
int permute_csr(int dtype, int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col, const void *val,
                const int32_t *perm, int32_t *out_ptr, int32_t *out_col, void *out_val, cudaStream_t s);
// direction 0: dst[i] = src[perm[i]]; 1: dst[perm[i]] = src[i]
cudaError_t launch_permute_vector(int dtype, int64_t n, const int32_t *perm, const void *src, void *dst,
                                  int direction, cudaStream_t s);

// One thread per row with 16-byte vector loads (sellv.cu, sl.vec); long rows are left to
// launch_rowsplit.
// out[b] = the largest column index stored in the rows at sorted positions
// [b * block, (b + 1) * block) of a one-thread-per-row, column-major sliced layout
// (out must hold -1 on entry; it stays -1 for a block without entries).  block is a
// multiple of 32 and of the slice height.
cudaError_t launch_block_max_col(const Sliced &sl, int64_t block, int32_t *out, cudaStream_t s);

cudaError_t launch_sellv_apply(int dtype, const Sliced &sl, int64_t n, const void *x, void *y, cudaStream_t s,
                               const Scale *scale = nullptr);
// G = sl.group threads per row (sellg.cu); long rows (len = -1) are left to launch_rowsplit.
cudaError_t launch_sellg_apply(int dtype, const Sliced &sl, int64_t n, const void *x, void *y, cudaStream_t s,
                               const Scale *scale = nullptr);
cudaError_t launch_sell_multi(int dtype, int nv, const Sliced &sl, int64_t n, const Segmented *split, const void *X,
                              int64_t ldx, void *Y, int64_t ldy, cudaStream_t s, const Scale &scale);
// vecops.cu: out[i] = X[i * ldx]; Y[i * ldy] = alpha * t[i] + beta * Y[i * ldy] (Y unread when beta == 0)
cudaError_t launch_gather_col(int dtype, int64_t n, const void *X, int64_t ldx, void *out, cudaStream_t s);
cudaError_t launch_axpby_col(int dtype, int64_t n, double alpha, const void *t, double beta, void *Y, int64_t ldy,
                             cudaStream_t s);
// row-split pass (kind 3) on its own (next to the CSR-vector bins)
cudaError_t launch_rowsplit(int dtype, const Segmented &sg, const void *x, void *y, cudaStream_t s);
// merge-path over a whole CSR (row i of the path is matrix row i), writing y
cudaError_t launch_merge_path_identity(int dtype, int64_t n_rows, int64_t nnz, const int32_t *ptr,
                                       const int32_t *col, const void *val, const void *x, void *y,
                                       int32_t *carry_row, double *carry_val, int64_t n_cta, cudaStream_t s,
                                       const int32_t *part);
// part[c] = merge-path split at diagonal c * kMergeItems, c = 0..n_cta (build time)
cudaError_t launch_merge_partition(int64_t n_rows, int64_t nnz, const int32_t *ptr, int64_t n_cta, int32_t *part,
                                   cudaStream_t s);
int64_t merge_ctas(int64_t n_rows, int64_t nnz);
int64_t coo_ctas(int64_t nnz);

}  // namespace spmv
