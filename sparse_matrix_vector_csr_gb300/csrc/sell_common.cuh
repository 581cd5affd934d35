// Pieces shared by the sliced-ELL kernels (sell.cu) and their multi-vector
// versions (sellmm.cu): argument blocks, the output rule, and the programmatic
// dependent launch hooks.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "device_util.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace sellk {

// Output of a row: y = v (mode 0), or y = alpha * v + beta * y (mode 1; y is not
// read when beta == 0, so whatever it held, NaN included, is overwritten).
struct Epi {
    double alpha;
    double beta;
    int mode;
};

template <typename T>
__device__ __forceinline__ void store_y(T *__restrict__ y, int64_t r, T v, const Epi &e) {
    if (e.mode == 0) {
        y[r] = v;
    } else {
        const T a = static_cast<T>(e.alpha), b = static_cast<T>(e.beta);
        y[r] = e.beta != 0.0 ? fma(a, v, b * y[r]) : a * v;
    }
}

struct SellArgs {
    int64_t n_pos;
    int log2C;
    uint32_t cmask;
    int64_t stride;
    const int64_t *slice_ptr;
    const int32_t *len;   // -1 marks a long row (handled by the row-split pass)
    const int32_t *perm;  // nullptr = natural order
    const int32_t *col;
    int64_t n;
};

struct SplitArgs {
    int64_t n_chunks;
    const int32_t *chunk_begin;
    const int32_t *chunk_end;
    const int32_t *chunk_row;      // compact row, or ~row when it is the row's only chunk
    const int32_t *rows;           // compact row -> matrix row
    const int32_t *row_chunk_ptr;  // chunks of compact row i: [row_chunk_ptr[i], row_chunk_ptr[i+1])
    const int32_t *col;
    double *partial;               // one partial sum per chunk of a row with several chunks
    int32_t *done;                 // per compact row: chunks finished in this apply (back to 0 after it)
    int accumulate;
};

// CS > 0: SELL with a compile-time slice height CS (stride = CS).
// CS == 0: runtime addressing (slice p >> log2C, row p & cmask, stride `stride`),
//          used by the single-slice ELLPACK-R / HYB-ELL layout and other slice heights.
// Programmatic dependent launch: a sliced-apply kernel may start while the previous
// kernel of the stream is still draining.  Everything read before grid_wait() is
// the handle's own matrix data, immutable after the build; x (which the previous
// kernel may produce) and y (which it may still read) are touched only after it.
using dev::allow_dependents;
using dev::grid_wait;

inline SellArgs sell_args(const Sliced &sl, int64_t n) {
    return SellArgs{sl.n_pos, sl.log2C, sl.cmask, sl.stride, sl.slice_ptr, sl.len, sl.perm, sl.col, n};
}

inline SplitArgs split_args(const Segmented &sg) {
    return SplitArgs{sg.n_chunks, sg.chunk_begin, sg.chunk_end, sg.chunk_row, sg.rows, sg.row_chunk_ptr,
                     sg.col, sg.partial, sg.done, sg.accumulate};
}

}  // namespace sellk
}  // namespace spmv
