// Bulk-staged SELL-32 apply: the matrix slots reach shared memory through the bulk
// copy engine (cp.async.bulk, completion counted on an mbarrier), and the threads
// gather x with plain loads at the column indices they read there.  This is the staging
// the SELL layout invites: a slice of C rows is one contiguous block of C * width slots
// (GPGPU spMVM paper, pJDS section, Fig. 1), and eight consecutive slices are one
// contiguous block too.  The copies carry an L2 evict-first hint, so the once-read
// stream does not push x out of L2, and a thread that reads its indices from shared
// memory keeps eight gathers in flight without waiting on a global load.
//
// Measured on GB300, it is slower than the register kernel (sell.cu) and is only built
// on request (format parameter `staged`): the matrices it was meant for, those whose x
// gathers have no locality, are bound by the requests an SM sends to L2 (one per
// 128-byte line a warp instruction touches, about one per clock), and the bulk copies'
// requests go through that same path, so moving the stream off the load pipe frees
// none of it; each CTA also waits for its first copy with nothing else to do.
//
// Work: one CTA of 256 threads per group of 8 consecutive slices (256 row positions,
// one per thread).  A group whose slices are at most kChunkCols wide is copied whole
// (two copies: indices and values; shared memory mirrors the global layout); a wider
// group goes in chunks of kChunkCols columns per slice (a copy per slice and array),
// through two stages so that chunk k + 1 lands while chunk k is summed.  Each thread
// stops at its own row's length, so padding is never gathered.  The copies of the
// matrix are issued before the programmatic-dependent-launch wait (the matrix is the
// handle's own, immutable data); x and y are touched after it.
//
// Waits on the mbarriers are bounded by a clock deadline (about a second); on timeout
// the kernel records it in a device flag of the handle, waits (again bounded) for its
// copies to land, and returns.  Synchronising entry points report the flag as
// SPMV_ERR_TIMEOUT.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_util.cuh"
#include "sell_common.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

using namespace dev;
using namespace sellk;

constexpr int kGroupSlices = kSellBlock / 32;           // 8 slices of 32 rows per CTA
constexpr int kChunkCols = 16;                          // columns per slice in one chunk
constexpr int kStageSlots = kGroupSlices * 32 * kChunkCols;  // 4096 slots per stage
constexpr int kGatherBatch = 8;                         // gathers in flight per thread
constexpr long long kWaitCycles = 2000000000LL;         // about one second at 2 GHz

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// true once the phase with this parity has completed; false after about a second
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bytes (a multiple of 16) from global src (16-byte aligned) to shared dst (16-byte
// aligned), completion counted on bar
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

struct StagedArgs {
    int64_t n_slices;
    int nstages;          // 1: every group fits one stage whole; 2: chunked groups go through two stages
    int64_t stage_slots;  // slots per stage
    int *err;             // set to 1 when a wait ran out
};

template <typename T>
__device__ __forceinline__ T *stage_val(unsigned char *smem, const StagedArgs &st, int b) {
    return reinterpret_cast<T *>(smem + st.nstages * st.stage_slots * 4) + b * st.stage_slots;
}

// Thread 0: issue chunk k of the group into stage b.  whole: the group's slots
// [g0, g1) in one copy per array; otherwise columns [k * kChunkCols, ...) of every
// slice, slice q at q * 32 * kChunkCols.
template <typename T>
__device__ __forceinline__ void issue_chunk(unsigned char *smem, uint64_t *bar, const StagedArgs &st, int b, int k,
                                            bool whole, const int64_t *base, const int32_t *width, int nsl,
                                            const int32_t *__restrict__ col, const T *__restrict__ val, uint64_t pol) {
    int32_t *scol = reinterpret_cast<int32_t *>(smem) + b * st.stage_slots;
    T *sval = stage_val<T>(smem, st, b);
    if (whole) {
        const int64_t g0 = base[0], g1 = base[nsl - 1] + 32 * static_cast<int64_t>(width[nsl - 1]);
        const uint32_t slots = static_cast<uint32_t>(g1 - g0);
        mbar_expect_tx(bar + b, slots * static_cast<uint32_t>(4 + sizeof(T)));
        if (slots) {
            bulk_copy(scol, col + g0, slots * 4, bar + b, pol);
            bulk_copy(sval, val + g0, slots * static_cast<uint32_t>(sizeof(T)), bar + b, pol);
        }
        return;
    }
    uint32_t total = 0;
    int cols[kGroupSlices];
#pragma unroll
    for (int q = 0; q < kGroupSlices; ++q) {
        const int c = q < nsl ? min(max(width[q] - k * kChunkCols, 0), kChunkCols) : 0;
        cols[q] = c;
        total += static_cast<uint32_t>(c) * 32u * static_cast<uint32_t>(4 + sizeof(T));
    }
    mbar_expect_tx(bar + b, total);
#pragma unroll
    for (int q = 0; q < kGroupSlices; ++q) {
        if (!cols[q]) continue;
        const int64_t src = base[q] + 32 * static_cast<int64_t>(k) * kChunkCols;
        const uint32_t slots = 32u * static_cast<uint32_t>(cols[q]);
        bulk_copy(scol + q * 32 * kChunkCols, col + src, slots * 4, bar + b, pol);
        bulk_copy(sval + q * 32 * kChunkCols, val + src, slots * static_cast<uint32_t>(sizeof(T)), bar + b, pol);
    }
}

template <typename T, bool K>
__global__ void __launch_bounds__(kSellBlock) k_sell_staged(SellArgs a, const T *__restrict__ val, StagedArgs st,
                                                           const T *__restrict__ x, T *__restrict__ y, Epi ep) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t bar[2];
    __shared__ int64_t base[kGroupSlices];
    __shared__ int32_t width[kGroupSlices];
    __shared__ int armed[2];  // phases armed on each stage's mbarrier (thread 0 only)
    allow_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kGroupSlices;
    const int nsl = static_cast<int>(min(static_cast<int64_t>(kGroupSlices), st.n_slices - s0));
    const int64_t s = s0 + warp;
    const bool have = warp < nsl;
    const int64_t p = s * 32 + lane;
    // this thread's row: length and output row (matrix data: may be read before the wait)
    const int w = have ? __ldg(a.len + p) : -1;
    const int64_t r = have ? (a.perm ? static_cast<int64_t>(__ldg(a.perm + p)) : p) : -1;
    if (lane == 0) {
        const int64_t b0 = have ? __ldg(a.slice_ptr + s) : 0;
        const int64_t b1 = have ? __ldg(a.slice_ptr + s + 1) : 0;
        base[warp] = b0;
        width[warp] = static_cast<int32_t>((b1 - b0) / 32);
    }
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    int maxw = 0;
#pragma unroll
    for (int q = 0; q < kGroupSlices; ++q) maxw = max(maxw, q < nsl ? width[q] : 0);
    const bool whole = maxw <= kChunkCols;
    const int nk = whole ? 1 : (maxw + kChunkCols - 1) / kChunkCols;
    const uint64_t pol = evict_first_policy();
    if (threadIdx.x == 0) {
        issue_chunk<T>(smem, bar, st, 0, 0, whole, base, width, nsl, a.col, val, pol);
        armed[0] = 1;
        armed[1] = 0;
        if (nk > 1) {
            issue_chunk<T>(smem, bar, st, 1, 1, whole, base, width, nsl, a.col, val, pol);
            armed[1] = 1;
        }
    }
    grid_wait();  // x and y only after the previous kernel of the stream
    const int my_w = have ? width[warp] : 0;
    const int64_t off_whole = have ? base[warp] - base[0] : 0;
    T acc = T(0);
    bool ok = true;
    for (int k = 0; k < nk; ++k) {
        const int b = k & 1;
        ok = ok && mbar_wait_bounded(bar + b, static_cast<uint32_t>((k >> 1) & 1));
        if (ok) {
            const int jc = k * kChunkCols;
            const int cols = whole ? my_w : min(max(my_w - jc, 0), kChunkCols);
            const int upto = min(cols, w - jc);  // this row's entries in the chunk (w < 0: none)
            const int32_t *scol = reinterpret_cast<const int32_t *>(smem) + b * st.stage_slots +
                                  (whole ? off_whole : warp * 32 * kChunkCols) + lane;
            const T *sval = stage_val<T>(smem, st, b) + (whole ? off_whole : warp * 32 * kChunkCols) + lane;
            for (int j = 0; j < upto; j += kGatherBatch) {
                T xv[kGatherBatch], vv[kGatherBatch];
#pragma unroll
                for (int u = 0; u < kGatherBatch; ++u) {
                    const bool on = j + u < upto;
                    vv[u] = on ? sval[(j + u) * 32] : T(0);
                    xv[u] = on ? gather_x<K>(x + scol[(j + u) * 32]) : T(0);
                }
#pragma unroll
                for (int u = 0; u < kGatherBatch; ++u) acc = fma(vv[u], xv[u], acc);  // past the row: +0 * +0
            }
        }
        if (k + 2 < nk) {
            __syncthreads();  // stage b is free
            if (threadIdx.x == 0 && ok) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_chunk<T>(smem, bar, st, b, k + 2, whole, base, width, nsl, a.col, val, pol);
                ++armed[b];
            }
        }
    }
    if (!ok) {
        if (lane == 0) atomicOr(st.err, 1);
        // Let the copies already issued land before the CTA's shared memory goes away
        // (the CTA lives until its last thread returns).  Thread 0 arms a stage again
        // only after its own wait for the stage's previous phase succeeded, so at most
        // the last armed phase of each stage is in flight: wait for that one.
        if (threadIdx.x == 0)
            for (int b = 0; b < 2; ++b)
                if (armed[b] > 0) (void)mbar_wait_bounded(bar + b, static_cast<uint32_t>((armed[b] - 1) & 1));
        return;
    }
    if (w >= 0 && r >= 0 && r < a.n) store_y(y, r, acc, ep);
}

template <typename T, bool K>
cudaError_t staged_launch(const Sliced &sl, int64_t n, const T *x, T *y, int *err, cudaStream_t s, const Epi &ep) {
    StagedArgs st;
    st.n_slices = sl.n_slices;
    st.nstages = sl.max_width <= kChunkCols ? 1 : 2;
    st.stage_slots = st.nstages == 1 ? static_cast<int64_t>(kGroupSlices) * 32 * sl.max_width : kStageSlots;
    st.err = err;
    const size_t smem = static_cast<size_t>(st.nstages * st.stage_slots) * (4 + sizeof(T));
    auto kern = k_sell_staged<T, K>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = sl.pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kSellBlock);
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(sl.n_slices, kGroupSlices)));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, sell_args(sl, n), static_cast<const T *>(sl.val), st, x, y, ep);
}

}  // namespace

bool sell_staged_supported(const Sliced &sl) {
    return sl.present && sl.log2C == 5 && sl.C == 32 && sl.group == 1 && !sl.vec && !sl.interleaved;
}

cudaError_t launch_sell_staged(int dtype, const Sliced &sl, int64_t n, const void *x, void *y, int *err,
                               cudaStream_t s, const Scale *scale) {
    if (!sl.present || sl.n_pos <= 0) return cudaSuccess;
    const Epi ep = scale ? Epi{scale->alpha, scale->beta, 1} : Epi{1.0, 0.0, 0};
    if (dtype == SPMV_F64)
        return sl.keep_x ? staged_launch<double, true>(sl, n, static_cast<const double *>(x), static_cast<double *>(y),
                                                       err, s, ep)
                         : staged_launch<double, false>(sl, n, static_cast<const double *>(x),
                                                        static_cast<double *>(y), err, s, ep);
    return sl.keep_x
               ? staged_launch<float, true>(sl, n, static_cast<const float *>(x), static_cast<float *>(y), err, s, ep)
               : staged_launch<float, false>(sl, n, static_cast<const float *>(x), static_cast<float *>(y), err, s, ep);
}

}  // namespace spmv
