// Conjugate gradients (Hestenes-Stiefel) on a handle: the Krylov use of SpMV that the
// Krylov/AMG paper builds on (its solvers section combines the sparse matrix-vector
// product with the vector updates and dot products of its equations (2)-(6)).
//
// Everything stays on the device.  One iteration is four launches on the caller's
// stream: q = A p (the handle's apply), p.q, the r update fused with the r.r
// reduction and the stopping test, and the x and p updates fused (both read p), so a
// step moves ten vectors besides the product.  Dot products reduce in double
// with a fixed grid; the last block to finish adds the per-block partials in block
// order, so every sum is reproducible run to run.  The step lengths and the stopping
// decision live in device memory: once the test has passed, the update kernels return
// at once, so the host only needs to look at a flag every few iterations and the
// iteration count is exact.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "device_util.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

using namespace dev;

constexpr int kRedBlocksPerSm = 4;  // 64 registers a thread for the unrolled loads
constexpr int kRedBlocks = 152 * kRedBlocksPerSm;  // one wave on 152 SMs; fixed, so reductions are reproducible
constexpr int kRedThreads = 256;
constexpr int kCheckEvery = 8;    // iterations enqueued between two host looks at the flag

struct Control {
    int32_t stop;        // 0 running, 1 converged, 2 p.Ap <= 0 (not positive definite)
    int32_t iterations;  // completed iterations
    uint32_t arrivals;   // blocks finished in the running reduction
    int32_t pad;
};

// Scalars: rr[0], rr[1] the residual norms squared by iteration parity, pq = p.Ap, bb = b.b
struct Scalars {
    double rr[2];
    double pq;
    double bb;
};

__device__ __forceinline__ double block_sum(double v) {
    __shared__ double warp_sum[kRedThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = v;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x < 32) {
        t = threadIdx.x < kRedThreads / 32 ? warp_sum[threadIdx.x] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    }
    return t;  // valid in thread 0
}

// Store this block's sum; the last block to arrive adds all of them in block order.
// Returns true in every thread of that block, with the total valid in its thread 0.
__device__ __forceinline__ bool finish_sum(double block_total, double *partial, uint32_t *arrivals,
                                           double &total) {
    __shared__ bool is_last;
    if (threadIdx.x == 0) {
        partial[blockIdx.x] = block_total;
        __threadfence();
        is_last = atomicAdd(arrivals, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!is_last) return false;
    __threadfence();
    double s = 0.0;
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += blockDim.x) s += __ldcg(partial + i);
    total = block_sum(s);
    if (threadIdx.x == 0) *arrivals = 0;
    return true;
}

// All solver kernels are launched with programmatic stream serialization: a kernel's
// blocks may become resident while the previous kernel drains, and wait in grid_wait()
// before touching anything that kernel writes.
//
// The solver's vectors live in its workspace, 256-byte aligned and zero-padded to a
// multiple of 256 bytes, so the kernels move them as 16-byte packs with no tail: the
// padding stays zero through every update.  Each thread keeps U packs of every operand
// in flight.  Per-thread partial sums are kept in the value type's accumulator (float
// for float32 vectors, whose double multiply-adds would run at the FP64 rate) and the
// block and grid sums in double.

template <typename T>
struct alignas(16) Pack {
    static constexpr int L = 16 / sizeof(T);
    T v[L];
};

template <typename T>
struct Acc {
    using type = double;
};
template <>
struct Acc<float> {
    using type = float;
};

template <typename T, int U>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_dot(int64_t units, const Pack<T> *__restrict__ a, const Pack<T> *__restrict__ b, double *__restrict__ partial,
          Control *ctl, double *__restrict__ out) {
    allow_dependents();
    grid_wait();
    if (ctl->stop) return;
    using A = typename Acc<T>::type;
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    A s = 0;
    for (int64_t u0 = gtid(); u0 < units; u0 += U * st) {
        Pack<T> pa[U], pb[U];
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (u0 + k * st < units) pa[k] = a[u0 + k * st], pb[k] = b[u0 + k * st];
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (u0 + k * st < units)
#pragma unroll
                for (int l = 0; l < Pack<T>::L; ++l) s = fma(static_cast<A>(pa[k].v[l]), static_cast<A>(pb[k].v[l]), s);
    }
    const double bs = block_sum(static_cast<double>(s));
    double total;
    if (finish_sum(bs, partial, &ctl->arrivals, total) && threadIdx.x == 0) *out = total;
}

// r -= alpha q with alpha = rr_cur / pq, then rr_next = r.r and the stopping test
template <typename T, int U>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_cg_r(int64_t units, Scalars *sc, Control *ctl, int cur, double stop_rr, const Pack<T> *__restrict__ q,
           Pack<T> *__restrict__ r, double *__restrict__ partial) {
    allow_dependents();
    grid_wait();
    if (ctl->stop) return;
    const double pq = sc->pq;
    if (!(pq > 0.0)) {  // no positive curvature along p: CG is undefined here
        if (blockIdx.x == 0 && threadIdx.x == 0) ctl->stop = 2;
        return;
    }
    using A = typename Acc<T>::type;
    const T alpha = static_cast<T>(sc->rr[cur] / pq);
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    A s = 0;
    for (int64_t u0 = gtid(); u0 < units; u0 += U * st) {
        Pack<T> pq_[U], pr[U];
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (u0 + k * st < units) pq_[k] = q[u0 + k * st], pr[k] = r[u0 + k * st];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (u0 + k * st < units) {
#pragma unroll
                for (int l = 0; l < Pack<T>::L; ++l) {
                    pr[k].v[l] = fma(-alpha, pq_[k].v[l], pr[k].v[l]);
                    s = fma(static_cast<A>(pr[k].v[l]), static_cast<A>(pr[k].v[l]), s);
                }
                r[u0 + k * st] = pr[k];
            }
        }
    }
    const double bs = block_sum(static_cast<double>(s));
    double total;
    if (finish_sum(bs, partial, &ctl->arrivals, total) && threadIdx.x == 0) {
        sc->rr[cur ^ 1] = total;
        ctl->iterations += 1;
        if (!(total > stop_rr)) ctl->stop = 1;  // NaN stops too
    }
}

// x += alpha p (alpha = rr_cur / pq), then p = r + beta p (beta = rr_next / rr_cur).
// In the step that met the stopping test only x moves; later steps return at once.
template <typename T, int U>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_cg_xp(int64_t units, const Scalars *sc, const Control *ctl, int32_t step, const Pack<T> *__restrict__ r,
            Pack<T> *__restrict__ p, Pack<T> *__restrict__ x) {
    allow_dependents();
    grid_wait();
    const int32_t stop = ctl->stop;
    if (stop && (stop != 1 || ctl->iterations != step + 1)) return;
    const int cur = step & 1;
    const T alpha = static_cast<T>(sc->rr[cur] / sc->pq);
    const T beta = static_cast<T>(sc->rr[cur ^ 1] / sc->rr[cur]);
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t u0 = gtid(); u0 < units; u0 += U * st) {
        Pack<T> pp[U], px[U], pr[U];
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (u0 + k * st < units) {
                pp[k] = p[u0 + k * st], px[k] = x[u0 + k * st];
                if (!stop) pr[k] = r[u0 + k * st];
            }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (u0 + k * st < units) {
#pragma unroll
                for (int l = 0; l < Pack<T>::L; ++l) px[k].v[l] = fma(alpha, pp[k].v[l], px[k].v[l]);
                x[u0 + k * st] = px[k];
                if (!stop) {
#pragma unroll
                    for (int l = 0; l < Pack<T>::L; ++l) pr[k].v[l] = fma(beta, pp[k].v[l], pr[k].v[l]);
                    p[u0 + k * st] = pr[k];
                }
            }
        }
    }
}

template <typename... P, typename... A>
cudaError_t launch(void (*kernel)(P...), cudaStream_t s, A... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kRedBlocks);
    cfg.blockDim = dim3(kRedThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct StreamBuffer {
    void *ptr = nullptr;
    cudaStream_t s = nullptr;
    ~StreamBuffer() {
        if (ptr) cudaFreeAsync(ptr, s);
    }
};

template <typename T>
int cg(spmv_handle_t h, const T *b, T *x, double rtol, int32_t max_iter, cudaStream_t s, int32_t *iterations,
       double *relative_residual) {
    constexpr int kUnroll = 4;    // packs of each operand in flight per thread
    constexpr int kUnrollXp = 2;  // three operands: fits 64 registers without spilling
    using P = Pack<T>;
    const int64_t n = h->n;
    const size_t vec = static_cast<size_t>(n) * sizeof(T);
    const size_t vec_pad = (vec + 255) / 256 * 256;
    const int64_t units = static_cast<int64_t>(vec_pad / sizeof(P));
    // workspace: r, p, q, x (zero-padded) | partial sums | scalars | control
    StreamBuffer ws;
    ws.s = s;
    const size_t bytes = 4 * vec_pad + kRedBlocks * sizeof(double) + sizeof(Scalars) + sizeof(Control);
    SPMV_TRY_CUDA(cudaMallocAsync(&ws.ptr, bytes, s));
    SPMV_TRY_CUDA(cudaMemsetAsync(ws.ptr, 0, bytes, s));
    char *base = static_cast<char *>(ws.ptr);
    P *r = reinterpret_cast<P *>(base);
    P *p = reinterpret_cast<P *>(base + vec_pad);
    P *q = reinterpret_cast<P *>(base + 2 * vec_pad);
    P *xw = reinterpret_cast<P *>(base + 3 * vec_pad);
    double *partial = reinterpret_cast<double *>(base + 4 * vec_pad);
    Scalars *sc = reinterpret_cast<Scalars *>(partial + kRedBlocks);
    Control *ctl = reinterpret_cast<Control *>(sc + 1);
    const P *cr = r, *cp = p, *cq = q;

    // bb = b.b, then r = b - A x, p = r, rr = r.r
    SPMV_TRY_CUDA(cudaMemcpyAsync(r, b, vec, cudaMemcpyDeviceToDevice, s));
    SPMV_TRY_CUDA(launch(k_dot<T, kUnroll>, s, units, cr, cr, partial, ctl, &sc->bb));
    SPMV_TRY_CUDA(cudaMemcpyAsync(xw, x, vec, cudaMemcpyDeviceToDevice, s));
    SPMV_TRY(spmv_apply_ex(h, -1.0, xw, 1.0, r, s));
    SPMV_TRY_CUDA(cudaMemcpyAsync(p, r, vec, cudaMemcpyDeviceToDevice, s));
    SPMV_TRY_CUDA(launch(k_dot<T, kUnroll>, s, units, cr, cr, partial, ctl, &sc->rr[0]));
    Scalars hs{};
    SPMV_TRY_CUDA(cudaMemcpyAsync(&hs, sc, sizeof(hs), cudaMemcpyDeviceToHost, s));
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    const double denom = hs.bb > 0.0 ? hs.bb : 1.0;  // b = 0: absolute residual
    const double stop_rr = rtol * rtol * denom;

    int32_t launched = 0;
    Control hc{};
    if (max_iter > 0 && hs.rr[0] > stop_rr) {
        while (launched < max_iter) {
            const int32_t block = std::min<int32_t>(kCheckEvery, max_iter - launched);
            for (int32_t j = 0; j < block; ++j, ++launched) {
                const int cur = launched & 1;
                SPMV_TRY(spmv_apply(h, p, q, s));
                SPMV_TRY_CUDA(launch(k_dot<T, kUnroll>, s, units, cp, cq, partial, ctl, &sc->pq));
                SPMV_TRY_CUDA(launch(k_cg_r<T, kUnroll>, s, units, sc, ctl, cur, stop_rr, cq, r, partial));
                SPMV_TRY_CUDA(launch(k_cg_xp<T, kUnrollXp>, s, units, static_cast<const Scalars *>(sc),
                                     static_cast<const Control *>(ctl), launched, cr, p, xw));
            }
            SPMV_TRY_CUDA(cudaMemcpyAsync(&hc, ctl, sizeof(hc), cudaMemcpyDeviceToHost, s));
            SPMV_TRY_CUDA(cudaStreamSynchronize(s));
            if (hc.stop) break;
        }
        SPMV_TRY_CUDA(cudaMemcpyAsync(x, xw, vec, cudaMemcpyDeviceToDevice, s));
        SPMV_TRY_CUDA(cudaMemcpyAsync(&hs, sc, sizeof(hs), cudaMemcpyDeviceToHost, s));
        SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    }
    const double rr = hs.rr[hc.iterations & 1];
    if (iterations) *iterations = hc.iterations;
    if (relative_residual) *relative_residual = std::sqrt(rr / denom);
    if (hc.stop == 2)
        return set_error(SPMV_ERR_UNSUPPORTED, "conjugate gradients broke down: p.Ap <= 0 (matrix not positive definite)");
    return SPMV_OK;
}

}  // namespace
}  // namespace spmv

using namespace spmv;

extern "C" SPMV_API int spmv_cg(spmv_handle_t h, const void *b, void *x, double rtol, int32_t max_iter,
                                void *stream, int32_t *iterations, double *relative_residual) {
    if (iterations) *iterations = 0;
    if (relative_residual) *relative_residual = 0.0;
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (max_iter < 0 || !(rtol >= 0.0)) return set_error(SPMV_ERR_INVALID_ARG, "need max_iter >= 0 and rtol >= 0");
    if (h->n == 0) return SPMV_OK;
    if (!b || !x) return set_error(SPMV_ERR_INVALID_ARG, "NULL b or x");
    if (b == x) return set_error(SPMV_ERR_INVALID_ARG, "b and x must not alias");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (h->dtype == SPMV_F64)
        return cg<double>(h, static_cast<const double *>(b), static_cast<double *>(x), rtol, max_iter, s, iterations,
                          relative_residual);
    return cg<float>(h, static_cast<const float *>(b), static_cast<float *>(x), rtol, max_iter, s, iterations,
                     relative_residual);
}
