// Sliced-ELL apply (SELL-C-sigma, ELLPACK-R, HYB's ELL part): one thread per sorted
// row position; each thread stops at its own row's length, so padding is never
// loaded or multiplied (ELLPACK-R of the GPGPU spMVM paper, arXiv 1112.5588,
// ELLPACK-R section; the "early stopping" quoted in the scite report
// "Load-balancing Sparse Matrix Vector Product Kernels on GPUs").
//
// Long rows leave the sliced layout for the row-split pass (the Trilinos issue on
// unpackAndCombine treats its longest class of rows with three levels of parallelism:
// rows, pieces of a row, and the entries of a piece): every long row is cut into
// chunks of at most 2048 entries (4096 in float64 in the fused launch below) and one
// warp reduces one chunk.  A row with a single chunk is written at once; for longer
// rows the warp that completes the last chunk sums the row's partials (in double, in
// chunk order) -- it learns it is last from a per-row integer counter.  Work per warp
// is bounded whatever the row lengths; values are never accumulated atomically, and
// the summation order is fixed.  The sliced rows and the chunks write disjoint rows of
// y, so both run in one launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "device_util.cuh"
#include "sell_common.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

using namespace dev;
using namespace sellk;

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

template <typename T, int U, int CS>
__device__ __forceinline__ void load_slots(const int32_t *__restrict__ cp, const T *__restrict__ vp, int64_t ld, int j,
                                           int w, int32_t (&c)[U], T (&v)[U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const bool on = j + u < w;
        const int64_t off = CS > 0 ? static_cast<int64_t>(u * CS) : u * ld;
        c[u] = on ? ld_stream(cp + off) : 0;
        v[u] = on ? ld_stream(vp + off) : T(0);
    }
}

// CS > 0: SELL with a compile-time slice height CS (stride = CS).
// CS == 0: runtime addressing (slice p >> log2C, row p & cmask, stride `stride`),
//          used by the single-slice ELLPACK-R / HYB-ELL layout and other slice heights.
// Entries are processed U at a time: U column indices and values (predicated on the
// row length, so padding is never touched), then the U gathers, then U FMAs.
// UW > 0 replaces U (the short-row variant below loads a whole row of up to UW entries
// before the dependency wait).
template <typename T, int CS, bool K, int UW = 0>
__device__ __forceinline__ void sell_row(int64_t p, const SellArgs &a, const T *__restrict__ val,
                                         const T *__restrict__ x, T *__restrict__ y, const Epi &ep) {
    constexpr int U = UW > 0 ? UW : SellChunk<T, CS>::U;
    const int w = __ldg(a.len + p);
    const uint64_t up = static_cast<uint64_t>(p);
    const int64_t slot = CS > 0 ? __ldg(a.slice_ptr + (up / CS)) + static_cast<int64_t>(up % CS)
                                : __ldg(a.slice_ptr + (p >> a.log2C)) + static_cast<int64_t>(p & a.cmask);
    // the ELL leading dimension is below 2^31
    const int64_t ld = CS > 0 ? CS : static_cast<int64_t>(static_cast<int>(a.stride));
    const int32_t *__restrict__ cp = a.col + slot;
    const T *__restrict__ vp = val + slot;
    const int64_t r = a.perm ? static_cast<int64_t>(__ldg(a.perm + p)) : p;
    int32_t c[U];
    T v[U];
    load_slots<T, U, CS>(cp, vp, ld, 0, w, c, v);  // first entries before the dependency wait
    grid_wait();
    T acc = T(0);
    for (int j = 0; j < w;) {
        T xv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) xv[u] = (j + u < w) ? gather_x<K>(x + c[u]) : T(0);
#pragma unroll
        for (int u = 0; u < U; ++u) acc = fma(v[u], xv[u], acc);  // inactive slots add +0 * +0
        j += U;
        if (j >= w) break;
        cp += U * ld;
        vp += U * ld;
        load_slots<T, U, CS>(cp, vp, ld, j, w, c, v);
    }
    if (w >= 0 && r >= 0 && r < a.n) store_y(y, r, acc, ep);
}

// One warp reduces chunk c of a long row.
template <typename T, bool K>
__device__ __forceinline__ void split_chunk(int64_t c, int lane, const SplitArgs &a, const T *__restrict__ val,
                                            const T *__restrict__ x, T *__restrict__ y, const Epi &ep) {
    constexpr int U = 4;
    const int32_t b = __ldg(a.chunk_begin + c), e = __ldg(a.chunk_end + c);
    T acc = T(0);
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
            grid_wait();  // see sell_row
            first = false;
        }
        T xv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) xv[u] = (k + 32 * u < e) ? gather_x<K>(x + cc[u]) : T(0);
#pragma unroll
        for (int u = 0; u < U; ++u) acc = fma(v[u], xv[u], acc);
    }
    if (first) grid_wait();  // a lane with no entry of its own still writes after the wait
    double s = static_cast<double>(acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const int32_t cr = __ldg(a.chunk_row + c);
    if (cr < 0) {  // the row's only chunk
        if (lane == 0) {
            const int32_t r = __ldg(a.rows + ~cr);
            if (a.accumulate)
                y[r] = static_cast<T>(static_cast<double>(y[r]) + s);
            else
                store_y(y, r, static_cast<T>(s), ep);
        }
        return;
    }
    // A row with several chunks: publish this chunk's partial; the warp that finishes
    // the row's last chunk adds all of them up in chunk order (same order every
    // apply) and writes y, then clears the row's counter for the next apply.
    const int32_t c0 = __ldg(a.row_chunk_ptr + cr), c1 = __ldg(a.row_chunk_ptr + cr + 1);
    int last = 0;
    if (lane == 0) {
        a.partial[c] = s;
        __threadfence();
        last = atomicAdd(a.done + cr, 1) == (c1 - c0) - 1;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    double t = 0.0;
    for (int32_t q = c0 + lane; q < c1; q += 32) t += __ldcg(a.partial + q);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    if (lane == 0) {
        const int32_t r = __ldg(a.rows + cr);
        if (a.accumulate)
            y[r] = static_cast<T>(static_cast<double>(y[r]) + t);
        else
            store_y(y, r, static_cast<T>(t), ep);
        a.done[cr] = 0;
    }
}

// K: gather x with the L2 evict-last policy (chosen per handle at build time)
template <typename T, int CS, bool K>
__global__ void __launch_bounds__(kSellBlock, CS > 0 ? 8 : 6)
    k_sell(SellArgs a, const T *__restrict__ val, const T *__restrict__ x, T *__restrict__ y, Epi ep) {
    allow_dependents();
    const int64_t p = gtid();
    if (p < a.n_pos) sell_row<T, CS, K>(p, a, val, x, y, ep);
}

// Short rows on a small matrix (fewer row positions than one wave of threads, every row
// at most kShortRow entries): each thread loads its whole row before grid_wait(), so
// between back-to-back applies the matrix read overlaps the previous apply entirely.
// With less than a wave there is no occupancy to protect, hence 64 registers.  W is the
// matrix's longest row: back to back, only the gathers, the multiply-adds and the store
// remain after the wait, and on this GPU a warp's float64 multiply-add holds the FP64 pipe
// for about 19 cycles (1.7 lanes a clock per SM), so a 5-entry stencil row compiled for 8
// multiply-adds spent 3/8 of that critical path on padding (predicated-off multiply-adds
// still take their turn in the pipe).  MINB = 4 (64 registers) below a wave; float64
// matrices whose longest row is 1-3 or 5-7 entries take the same kernel above a wave at
// MINB = 6 (40 registers): 7 multiply-adds for the 3D Laplacian's 7-entry rows instead of
// 8 measured 29.6 against 30.9 us per apply (float32, whose multiply-adds are cheap, stays
// with k_sell: 18.0 against 17.8; widths 4 and 8 are whole groups of k_sell's four).
template <typename T, int CS, bool K, int W, int MINB>
__global__ void __launch_bounds__(kSellBlock, MINB)
    k_sell_short(SellArgs a, const T *__restrict__ val, const T *__restrict__ x, T *__restrict__ y, Epi ep) {
    allow_dependents();
    const int64_t p = gtid();
    if (p < a.n_pos) sell_row<T, CS, K, W>(p, a, val, x, y, ep);
}

// Sliced rows and row-split chunks in one launch: the first split_ctas CTAs take
// eight chunks each (one per warp), the rest take kSellBlock row positions each.
// Float64 gets 40 registers (6 blocks per SM): at 32 the chunk code spills, and the
// power-law matrix measured 169.7 against 178.2 us per apply.
template <typename T, int CS, bool K>
__global__ void __launch_bounds__(kSellBlock, (CS > 0 && sizeof(T) == 4) ? 8 : 6)
    k_sell_split(SellArgs a, const T *__restrict__ val, SplitArgs b, const T *__restrict__ split_val,
                 int64_t split_ctas, const T *__restrict__ x, T *__restrict__ y, Epi ep) {
    allow_dependents();
    if (blockIdx.x < split_ctas) {
        const int64_t c = (static_cast<int64_t>(blockIdx.x) * kSellBlock + threadIdx.x) >> 5;
        if (c < b.n_chunks) split_chunk<T, K>(c, threadIdx.x & 31, b, split_val, x, y, ep);
        return;
    }
    const int64_t p = (static_cast<int64_t>(blockIdx.x) - split_ctas) * kSellBlock + threadIdx.x;
    if (p < a.n_pos) sell_row<T, CS, K>(p, a, val, x, y, ep);
}

// ---------------------------------------------------------------------------
// narrow tail of a globally sorted layout
// ---------------------------------------------------------------------------
// With all rows sorted by length (sigma >= n) the slice widths never increase, and the
// last slices hold the rows of at most kTailW entries: on the power-law matrix three
// rows in four.  There a thread's whole row is an entry or two, and sell_row spends it
// on a chain of three dependent loads (slice offset and length, then the row's slots,
// then x) with a single gather in flight.  The tail path takes each slot address from
// the table of width regions (no slice-offset load), and gives every thread kTailR rows
// (row q of kTailR consecutive slices, one warp per kTailR slices) with all their loads
// issued before the first gather: two dependent steps, and kTailR times the gathers in
// flight.  The slots are loaded up to the slice width (padding slots hold column 0 and
// value 0), and x is gathered only below the row's own length, so padding never
// touches x.
constexpr int kTailW = 2;  // slice widths the tail path takes
constexpr int kTailR = 2;  // rows per thread there
static_assert(kTailW <= kTailMaxW, "tail table too small");

struct TailArgs {
    int64_t n_slices;
    int64_t slice[kTailW + 1];  // first slice of width <= w
    int64_t slot[kTailW + 1];   // its first slot
};

template <typename T, bool K>
__device__ __forceinline__ void sell_tail(int64_t warp, int lane, const SellArgs &a, const TailArgs &t,
                                          const T *__restrict__ val, const T *__restrict__ x, T *__restrict__ y,
                                          const Epi &ep) {
    int32_t c[kTailR][kTailW];
    T v[kTailR][kTailW];
    int len[kTailR];
    int32_t row[kTailR];
#pragma unroll
    for (int r = 0; r < kTailR; ++r) {
        const int64_t s = t.slice[kTailW] + warp * kTailR + r;
        len[r] = -1;
        row[r] = -1;
        int w = 0;
        int64_t slot = 0;
        if (s < t.n_slices) {
            // width of slice s: the smallest w whose region (slices t.slice[w] on) holds s
            int64_t s0 = t.slice[kTailW], b0 = t.slot[kTailW];
            w = kTailW;
#pragma unroll
            for (int q = kTailW - 1; q >= 0; --q)
                if (s >= t.slice[q]) {
                    w = q;
                    s0 = t.slice[q];
                    b0 = t.slot[q];
                }
            slot = b0 + (s - s0) * (32 * w) + lane;
            const int64_t p = s * 32 + lane;
            len[r] = __ldg(a.len + p);
            row[r] = __ldg(a.perm + p);
        }
#pragma unroll
        for (int j = 0; j < kTailW; ++j) {
            const bool on = j < w;
            c[r][j] = on ? ld_stream(a.col + slot + 32 * j) : 0;
            v[r][j] = on ? ld_stream(val + slot + 32 * j) : T(0);
        }
    }
    grid_wait();  // see sell_row
    T xv[kTailR][kTailW];
#pragma unroll
    for (int r = 0; r < kTailR; ++r)
#pragma unroll
        for (int j = 0; j < kTailW; ++j) xv[r][j] = j < len[r] ? gather_x<K>(x + c[r][j]) : T(0);
#pragma unroll
    for (int r = 0; r < kTailR; ++r) {
        T acc = T(0);
#pragma unroll
        for (int j = 0; j < kTailW; ++j) acc = fma(v[r][j], xv[r][j], acc);  // past the row: +0 * +0
        if (len[r] >= 0 && row[r] >= 0 && row[r] < a.n) store_y(y, row[r], acc, ep);
    }
}

// A globally sorted layout with a narrow tail: the first split_ctas CTAs take the long
// rows' chunks (one per warp, as in k_sell_split; none without long rows), the next
// head_ctas the positions before the tail (one per thread), the rest the tail -- one
// group of 2 x 32 rows per warp with chunks in the launch (the tail CTAs then fill the
// slots the chunks leave), or, without chunks, at most Sliced::tail_cap CTAs that loop.
template <typename T, bool K, bool SPLIT>
__global__ void __launch_bounds__(kSellBlock, SPLIT ? 6 : 8)
    k_sell_tail(SellArgs a, const T *__restrict__ val, SplitArgs b, const T *__restrict__ split_val,
                int64_t split_ctas, int64_t head_ctas, TailArgs t, const T *__restrict__ x, T *__restrict__ y,
                Epi ep) {
    allow_dependents();
    if (SPLIT && blockIdx.x < split_ctas) {
        const int64_t c = (static_cast<int64_t>(blockIdx.x) * kSellBlock + threadIdx.x) >> 5;
        if (c < b.n_chunks) split_chunk<T, K>(c, threadIdx.x & 31, b, split_val, x, y, ep);
        return;
    }
    const int64_t hb = static_cast<int64_t>(blockIdx.x) - (SPLIT ? split_ctas : 0);
    if (hb < head_ctas) {
        const int64_t p = hb * kSellBlock + threadIdx.x;
        if (p < t.slice[kTailW] * 32) sell_row<T, 32, K>(p, a, val, x, y, ep);
        return;
    }
    const int64_t first = (hb - head_ctas) * (kSellBlock / 32) + (threadIdx.x >> 5);
    if constexpr (SPLIT) {
        sell_tail<T, K>(first, threadIdx.x & 31, a, t, val, x, y, ep);
    } else {
        // no chunks in the launch: the tail CTAs are capped and each loops over the tail
        // (a CTA of two rows a thread lives a few microseconds; launching one per 512 rows
        // left the SMs' slots idle between CTAs)
        const int64_t stride = (static_cast<int64_t>(gridDim.x) - head_ctas) * (kSellBlock / 32);
        const int64_t n_warps = (t.n_slices - t.slice[kTailW] + kTailR - 1) / kTailR;
        for (int64_t warp = first; warp < n_warps; warp += stride)
            sell_tail<T, K>(warp, threadIdx.x & 31, a, t, val, x, y, ep);
    }
}

// Row-split chunks alone (long rows next to the CSR-vector bins).
template <typename T>
__global__ void __launch_bounds__(256) k_split_chunks(SplitArgs b, const T *__restrict__ val, const T *__restrict__ x,
                                                     T *__restrict__ y) {
    const int64_t c = gtid() >> 5;
    if (c < b.n_chunks) split_chunk<T, true>(c, threadIdx.x & 31, b, val, x, y, Epi{1.0, 0.0, 0});
}

// k_sell_short compiled for the matrix's longest row (1 .. kShortRow entries)
template <typename T, int CS, bool K, int MINB>
cudaError_t short_launch(cudaLaunchConfig_t &cfg, const Sliced &sl, int64_t n, const T *x, T *y, const Epi &ep) {
    const T *val = static_cast<const T *>(sl.val);
    static_assert(kShortRow == 8, "one case per row width");
    switch (sl.max_width) {
        case 0:
        case 1: return cudaLaunchKernelEx(&cfg, k_sell_short<T, CS, K, 1, MINB>, sell_args(sl, n), val, x, y, ep);
        case 2: return cudaLaunchKernelEx(&cfg, k_sell_short<T, CS, K, 2, MINB>, sell_args(sl, n), val, x, y, ep);
        case 3: return cudaLaunchKernelEx(&cfg, k_sell_short<T, CS, K, 3, MINB>, sell_args(sl, n), val, x, y, ep);
        case 4: return cudaLaunchKernelEx(&cfg, k_sell_short<T, CS, K, 4, MINB>, sell_args(sl, n), val, x, y, ep);
        case 5: return cudaLaunchKernelEx(&cfg, k_sell_short<T, CS, K, 5, MINB>, sell_args(sl, n), val, x, y, ep);
        case 6: return cudaLaunchKernelEx(&cfg, k_sell_short<T, CS, K, 6, MINB>, sell_args(sl, n), val, x, y, ep);
        case 7: return cudaLaunchKernelEx(&cfg, k_sell_short<T, CS, K, 7, MINB>, sell_args(sl, n), val, x, y, ep);
        default: return cudaLaunchKernelEx(&cfg, k_sell_short<T, CS, K, 8, MINB>, sell_args(sl, n), val, x, y, ep);
    }
}

template <typename T, int CS, bool K>
cudaError_t sell_launch(const Sliced &sl, int64_t n, const Segmented *sg, const T *x, T *y, cudaStream_t s,
                        const Epi &ep) {
    const T *val = static_cast<const T *>(sl.val);
    const int64_t sell_ctas = ceil_div(sl.n_pos, kSellBlock);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = sl.pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kSellBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool split = sg && sg->kind == 3 && sg->n_chunks > 0;
    if (CS == 32 && sl.has_tail && sl.tail_slice[kTailW] < sl.n_slices) {
        TailArgs t;
        t.n_slices = sl.n_slices;
        for (int w = 0; w <= kTailW; ++w) {
            t.slice[w] = sl.tail_slice[w];
            t.slot[w] = sl.tail_slot[w];
        }
        const int64_t split_ctas = split ? ceil_div(sg->n_chunks * 32, kSellBlock) : 0;
        const int64_t head_ctas = ceil_div(t.slice[kTailW] * 32, kSellBlock);
        int64_t tail_ctas = ceil_div(sl.n_slices - t.slice[kTailW], (kSellBlock / 32) * kTailR);
        if (!split && sl.tail_cap > 0) tail_ctas = std::min(tail_ctas, sl.tail_cap);
        cfg.gridDim = dim3(static_cast<unsigned>(split_ctas + head_ctas + tail_ctas));
        const SplitArgs b = split ? split_args(*sg) : SplitArgs{};
        const T *split_val = split ? static_cast<const T *>(sg->val) : nullptr;
        if (split)
            return cudaLaunchKernelEx(&cfg, k_sell_tail<T, K, true>, sell_args(sl, n), val, b, split_val, split_ctas,
                                      head_ctas, t, x, y, ep);
        return cudaLaunchKernelEx(&cfg, k_sell_tail<T, K, false>, sell_args(sl, n), val, b, split_val, split_ctas,
                                  head_ctas, t, x, y, ep);
    }
    if (split) {
        const int64_t split_ctas = ceil_div(sg->n_chunks * 32, kSellBlock);
        cfg.gridDim = dim3(static_cast<unsigned>(split_ctas + sell_ctas));
        return cudaLaunchKernelEx(&cfg, k_sell_split<T, CS, K>, sell_args(sl, n), val, split_args(*sg),
                                  static_cast<const T *>(sg->val), split_ctas, x, y, ep);
    }
    cfg.gridDim = dim3(static_cast<unsigned>(sell_ctas));
    if (sl.max_width <= kShortRow && sl.n_pos <= kShortRowsMax)
        return short_launch<T, CS, K, 4>(cfg, sl, n, x, y, ep);
    if constexpr (sizeof(T) == 8) {  // widths 4 and 8 are whole groups of k_sell's four
        if (sl.max_width < kShortRow && (sl.max_width & 3)) return short_launch<T, CS, K, 6>(cfg, sl, n, x, y, ep);
    }
    return cudaLaunchKernelEx(&cfg, k_sell<T, CS, K>, sell_args(sl, n), val, x, y, ep);
}

template <typename T, int CS>
cudaError_t sell_launch_k(const Sliced &sl, int64_t n, const Segmented *sg, const T *x, T *y, cudaStream_t s,
                          const Epi &ep) {
    return sl.keep_x ? sell_launch<T, CS, true>(sl, n, sg, x, y, s, ep)
                     : sell_launch<T, CS, false>(sl, n, sg, x, y, s, ep);
}

template <typename T>
cudaError_t sell_dispatch(const Sliced &sl, int64_t n, const Segmented *sg, const T *x, T *y, cudaStream_t s,
                          const Epi &ep) {
    const bool sliced = sl.log2C < 31;
    if (sliced && sl.C == 32) return sell_launch_k<T, 32>(sl, n, sg, x, y, s, ep);
    if (sliced && sl.C == 64) return sell_launch_k<T, 64>(sl, n, sg, x, y, s, ep);
    return sell_launch_k<T, 0>(sl, n, sg, x, y, s, ep);
}

template <typename T>
cudaError_t split_dispatch(const Segmented &sg, const T *x, T *y, cudaStream_t s) {
    if (sg.kind != 3 || sg.n_chunks <= 0) return cudaSuccess;
    k_split_chunks<T><<<static_cast<unsigned>(ceil_div(sg.n_chunks * 32, 256)), 256, 0, s>>>(
        split_args(sg), static_cast<const T *>(sg.val), x, y);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sell_apply(int dtype, const Sliced &sl, int64_t n, const Segmented *split, const void *x, void *y,
                              cudaStream_t s, const Scale *scale) {
    if (!sl.present || sl.n_pos <= 0) return cudaSuccess;
    const Epi ep = scale ? Epi{scale->alpha, scale->beta, 1} : Epi{1.0, 0.0, 0};
    if (dtype == SPMV_F64)
        return sell_dispatch<double>(sl, n, split, static_cast<const double *>(x), static_cast<double *>(y), s, ep);
    return sell_dispatch<float>(sl, n, split, static_cast<const float *>(x), static_cast<float *>(y), s, ep);
}

int64_t sell_tail_positions(const Sliced &sl) {
    if (!sl.present || !sl.has_tail || sl.C != 32 || sl.tail_slice[kTailW] >= sl.n_slices) return 0;
    return (sl.n_slices - sl.tail_slice[kTailW]) * 32;
}

cudaError_t launch_rowsplit(int dtype, const Segmented &sg, const void *x, void *y, cudaStream_t s) {
    if (dtype == SPMV_F64)
        return split_dispatch<double>(sg, static_cast<const double *>(x), static_cast<double *>(y), s);
    return split_dispatch<float>(sg, static_cast<const float *>(x), static_cast<float *>(y), s);
}

}  // namespace spmv
