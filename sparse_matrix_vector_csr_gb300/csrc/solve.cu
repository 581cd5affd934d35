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
// at once, so the iteration count is exact however far the host has enqueued.  The host
// paces its launches on a progress record (iterations done, stop flag) that the kernels
// write into page-locked host memory, keeping two iterations queued: no copy or
// synchronisation sits in the stream between iterations.
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
constexpr int kAhead = 2;         // iterations enqueued beyond the last one whose update finished

struct Control {
    int32_t stop;        // 0 running, 1 converged, 2 p.Ap <= 0 (not positive definite)
    int32_t iterations;  // completed iterations
    uint32_t arrivals;   // blocks finished in the running reduction
    int32_t pad;
};

// The solve's progress as the host sees it: page-locked host memory that the kernels
// write through its device mapping whenever they change the iteration count or the stop
// flag, so the host paces its launches without any copy in the stream.
struct Progress {
    int32_t iterations;
    int32_t stop;
};

__device__ __forceinline__ void publish(Progress *pg, const Control *ctl) {
    volatile Progress *v = pg;
    v->iterations = ctl->iterations;
    v->stop = ctl->stop;
    __threadfence_system();
}

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
    k_cg_r(int64_t units, Scalars *sc, Control *ctl, Progress *pg, int cur, double stop_rr,
           const Pack<T> *__restrict__ q, Pack<T> *__restrict__ r, double *__restrict__ partial) {
    allow_dependents();
    grid_wait();
    if (ctl->stop) return;
    const double pq = sc->pq;
    if (!(pq > 0.0)) {  // no positive curvature along p: CG is undefined here
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            ctl->stop = 2;
            publish(pg, ctl);
        }
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
        publish(pg, ctl);
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

// ---------------------------------------------------------------------------
// BiCGSTAB (van der Vorst), unpreconditioned, shadow residual r_hat = r_0
// ---------------------------------------------------------------------------
struct BiScalars {
    double rho[2];  // (r_hat, r) for the step of matching parity
    double rv;      // (r_hat, v)
    double ts, tt;  // (t, s), (t, t)
    double rr[2];   // (r, r) after the step of matching parity
    double bb;
    double alpha, omega;
};

// Two sums at once: every block stores both of its block sums, the last block adds
// each in block order.
__device__ __forceinline__ bool finish_sum2(double a, double b, double *partial, uint32_t *arrivals, double &ta,
                                            double &tb) {
    __shared__ bool is_last;
    if (threadIdx.x == 0) {
        partial[2 * blockIdx.x] = a;
        partial[2 * blockIdx.x + 1] = b;
        __threadfence();
        is_last = atomicAdd(arrivals, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!is_last) return false;
    __threadfence();
    double sa = 0.0, sb = 0.0;
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += blockDim.x) {
        sa += __ldcg(partial + 2 * i);
        sb += __ldcg(partial + 2 * i + 1);
    }
    ta = block_sum(sa);
    __syncthreads();  // warp_sum is reused
    tb = block_sum(sb);
    if (threadIdx.x == 0) *arrivals = 0;
    return true;
}

// p = r + beta (p - omega v), beta = (rho_k / rho_{k-1}) (alpha / omega)
template <typename T, int U>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_bi_p(int64_t units, const BiScalars *sc, Control *ctl, Progress *pg, int cur, const Pack<T> *__restrict__ r,
           const Pack<T> *__restrict__ v, Pack<T> *__restrict__ p) {
    allow_dependents();
    grid_wait();
    if (ctl->stop) return;
    const double rho = sc->rho[cur];
    if (!(rho != 0.0)) {  // (r_hat, r) = 0 (or NaN): breakdown
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            ctl->stop = 2;
            publish(pg, ctl);
        }
        return;
    }
    const T beta = static_cast<T>((rho / sc->rho[cur ^ 1]) * (sc->alpha / sc->omega));
    const T omega = static_cast<T>(sc->omega);
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t u0 = gtid(); u0 < units; u0 += U * st) {
        Pack<T> pr[U], pv[U], pp[U];
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (u0 + k * st < units) pr[k] = r[u0 + k * st], pv[k] = v[u0 + k * st], pp[k] = p[u0 + k * st];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (u0 + k * st < units) {
#pragma unroll
                for (int l = 0; l < Pack<T>::L; ++l)
                    pp[k].v[l] = fma(beta, fma(-omega, pv[k].v[l], pp[k].v[l]), pr[k].v[l]);
                p[u0 + k * st] = pp[k];
            }
        }
    }
}

// alpha = rho_k / (r_hat, v); s = r - alpha v
template <typename T, int U>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_bi_s(int64_t units, BiScalars *sc, Control *ctl, Progress *pg, int cur, const Pack<T> *__restrict__ r,
           const Pack<T> *__restrict__ v, Pack<T> *__restrict__ s_out) {
    allow_dependents();
    grid_wait();
    if (ctl->stop) return;
    const double rv = sc->rv;
    if (!(rv != 0.0)) {  // (r_hat, A p) = 0: breakdown
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            ctl->stop = 2;
            publish(pg, ctl);
        }
        return;
    }
    const double alpha_d = sc->rho[cur] / rv;
    if (blockIdx.x == 0 && threadIdx.x == 0) sc->alpha = alpha_d;
    const T alpha = static_cast<T>(alpha_d);
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t u0 = gtid(); u0 < units; u0 += U * st) {
        Pack<T> pr[U], pv[U];
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (u0 + k * st < units) pr[k] = r[u0 + k * st], pv[k] = v[u0 + k * st];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (u0 + k * st < units) {
#pragma unroll
                for (int l = 0; l < Pack<T>::L; ++l) pr[k].v[l] = fma(-alpha, pv[k].v[l], pr[k].v[l]);
                s_out[u0 + k * st] = pr[k];
            }
        }
    }
}

// (t, s) and (t, t) in one pass
template <typename T, int U>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_bi_tt(int64_t units, BiScalars *sc, Control *ctl, const Pack<T> *__restrict__ t, const Pack<T> *__restrict__ s,
            double *__restrict__ partial) {
    allow_dependents();
    grid_wait();
    if (ctl->stop) return;
    using A = typename Acc<T>::type;
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    A ts = 0, tt = 0;
    for (int64_t u0 = gtid(); u0 < units; u0 += U * st) {
        Pack<T> pt[U], ps[U];
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (u0 + k * st < units) pt[k] = t[u0 + k * st], ps[k] = s[u0 + k * st];
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (u0 + k * st < units)
#pragma unroll
                for (int l = 0; l < Pack<T>::L; ++l) {
                    ts = fma(static_cast<A>(pt[k].v[l]), static_cast<A>(ps[k].v[l]), ts);
                    tt = fma(static_cast<A>(pt[k].v[l]), static_cast<A>(pt[k].v[l]), tt);
                }
    }
    const double bts = block_sum(static_cast<double>(ts));
    __syncthreads();  // warp_sum is reused
    const double btt = block_sum(static_cast<double>(tt));
    double a, b;
    if (finish_sum2(bts, btt, partial, &ctl->arrivals, a, b) && threadIdx.x == 0) {
        sc->ts = a;
        sc->tt = b;
    }
}

// omega = (t, s) / (t, t); x += alpha p + omega s; r = s - omega t; then (r, r), the next
// rho = (r_hat, r) and the stopping test
template <typename T, int U>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_bi_xr(int64_t units, BiScalars *sc, Control *ctl, Progress *pg, int cur, double stop_rr,
            const Pack<T> *__restrict__ p,
            const Pack<T> *__restrict__ s, const Pack<T> *__restrict__ t, const Pack<T> *__restrict__ r_hat,
            Pack<T> *__restrict__ x, Pack<T> *__restrict__ r, double *__restrict__ partial) {
    allow_dependents();
    grid_wait();
    if (ctl->stop) return;
    using A = typename Acc<T>::type;
    const double tt_d = sc->tt;
    const double omega_d = tt_d > 0.0 ? sc->ts / tt_d : 0.0;
    const T alpha = static_cast<T>(sc->alpha), omega = static_cast<T>(omega_d);
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    A rr = 0, rho = 0;
    for (int64_t u0 = gtid(); u0 < units; u0 += U * st) {
        Pack<T> pp[U], ps[U], pt[U], px[U], ph[U];
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (u0 + k * st < units) {
                pp[k] = p[u0 + k * st], ps[k] = s[u0 + k * st], pt[k] = t[u0 + k * st];
                px[k] = x[u0 + k * st], ph[k] = r_hat[u0 + k * st];
            }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (u0 + k * st < units) {
#pragma unroll
                for (int l = 0; l < Pack<T>::L; ++l) {
                    px[k].v[l] = fma(omega, ps[k].v[l], fma(alpha, pp[k].v[l], px[k].v[l]));
                    const T rn = fma(-omega, pt[k].v[l], ps[k].v[l]);
                    ps[k].v[l] = rn;
                    rr = fma(static_cast<A>(rn), static_cast<A>(rn), rr);
                    rho = fma(static_cast<A>(ph[k].v[l]), static_cast<A>(rn), rho);
                }
                x[u0 + k * st] = px[k];
                r[u0 + k * st] = ps[k];
            }
        }
    }
    const double brr = block_sum(static_cast<double>(rr));
    __syncthreads();  // warp_sum is reused
    const double brho = block_sum(static_cast<double>(rho));
    double a, b;
    if (finish_sum2(brr, brho, partial, &ctl->arrivals, a, b) && threadIdx.x == 0) {
        sc->rr[cur ^ 1] = a;
        sc->rho[cur ^ 1] = b;
        sc->omega = omega_d;
        ctl->iterations += 1;
        if (!(a > stop_rr))
            ctl->stop = 1;             // converged (NaN stops too)
        else if (omega_d == 0.0)
            ctl->stop = 2;             // omega = 0 before convergence: breakdown
        publish(pg, ctl);
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
        if (ptr) lib_free_async(ptr, s);
    }
};

// Paces the host's launches on the solve's Progress: before enqueuing an iteration the
// host waits until at most kAhead - 1 enqueued iterations are still unfinished, so the
// stream never drains between iterations and at most kAhead run after a stop (every
// update kernel then returns at once; only the products run).  The wait looks at the
// stream every 1024 reads and ends when the stream is idle or reports an error, so it
// cannot outlast the work it waits for.
// The record lives in page-locked memory allocated once per host thread (a solve call
// is synchronous, so a thread runs one solve at a time) and kept for the thread's life:
// allocating and freeing it per solve cost about a millisecond.
struct Pacer {
    Progress *host = nullptr;
    Progress *dev = nullptr;
    cudaStream_t s = nullptr;
    ~Pacer() {
        if (host) cudaStreamSynchronize(s);  // no kernel of this solve may still write the record
    }
    int init() {
        thread_local Progress *record = nullptr;
        if (record) {  // still page-locked? (a device reset releases it)
            cudaPointerAttributes attr;
            if (cudaPointerGetAttributes(&attr, record) != cudaSuccess || attr.type != cudaMemoryTypeHost) {
                (void)cudaGetLastError();
                record = nullptr;
            }
        }
        if (!record)
            SPMV_TRY_CUDA(cudaHostAlloc(reinterpret_cast<void **>(&record), sizeof(Progress),
                                        cudaHostAllocMapped | cudaHostAllocPortable));
        host = record;
        host->iterations = 0;
        host->stop = 0;
        SPMV_TRY_CUDA(cudaHostGetDevicePointer(reinterpret_cast<void **>(&dev), host, 0));
        return SPMV_OK;
    }
    // returns with *stop set when the solve has stopped
    int wait(int32_t launched, bool *stop) {
        const volatile Progress *v = host;
        for (uint32_t reads = 1;; ++reads) {
            if (v->stop) {
                *stop = true;
                return SPMV_OK;
            }
            if (launched - v->iterations < kAhead) return SPMV_OK;
            if ((reads & 1023u) == 0) {
                const cudaError_t e = cudaStreamQuery(s);
                if (e == cudaSuccess) return SPMV_OK;  // everything enqueued has finished
                if (e != cudaErrorNotReady) return set_cuda_error(e, "cudaStreamQuery");
            }
        }
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
    SPMV_TRY_CUDA(lib_malloc_async(&ws.ptr, bytes, s));
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
        Pacer pace;
        pace.s = s;
        SPMV_TRY(pace.init());
        for (; launched < max_iter; ++launched) {
            bool stop = false;
            SPMV_TRY(pace.wait(launched, &stop));
            if (stop) break;
            const int cur = launched & 1;
            SPMV_TRY(spmv_apply(h, p, q, s));
            SPMV_TRY_CUDA(launch(k_dot<T, kUnroll>, s, units, cp, cq, partial, ctl, &sc->pq));
            SPMV_TRY_CUDA(launch(k_cg_r<T, kUnroll>, s, units, sc, ctl, pace.dev, cur, stop_rr, cq, r, partial));
            SPMV_TRY_CUDA(launch(k_cg_xp<T, kUnrollXp>, s, units, static_cast<const Scalars *>(sc),
                                 static_cast<const Control *>(ctl), launched, cr, p, xw));
        }
        SPMV_TRY_CUDA(cudaMemcpyAsync(x, xw, vec, cudaMemcpyDeviceToDevice, s));
        SPMV_TRY_CUDA(cudaMemcpyAsync(&hs, sc, sizeof(hs), cudaMemcpyDeviceToHost, s));
        SPMV_TRY_CUDA(cudaMemcpyAsync(&hc, ctl, sizeof(hc), cudaMemcpyDeviceToHost, s));
        SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    }
    const double rr = hs.rr[hc.iterations & 1];
    if (iterations) *iterations = hc.iterations;
    if (relative_residual) *relative_residual = std::sqrt(rr / denom);
    if (hc.stop == 2)
        return set_error(SPMV_ERR_UNSUPPORTED, "conjugate gradients broke down: p.Ap <= 0 (matrix not positive definite)");
    return SPMV_OK;
}

template <typename T>
int bicgstab(spmv_handle_t h, const T *b, T *x, double rtol, int32_t max_iter, cudaStream_t s, int32_t *iterations,
             double *relative_residual) {
    constexpr int kUnroll = 2;  // up to five operands a kernel: 2 packs each in flight
    using P = Pack<T>;
    const int64_t n = h->n;
    const size_t vec = static_cast<size_t>(n) * sizeof(T);
    const size_t vec_pad = (vec + 255) / 256 * 256;
    const int64_t units = static_cast<int64_t>(vec_pad / sizeof(P));
    // workspace: r, r_hat, p, v, s, t, x (zero-padded) | 2 x block partials | scalars | control
    StreamBuffer ws;
    ws.s = s;
    const size_t bytes = 7 * vec_pad + 2 * kRedBlocks * sizeof(double) + sizeof(BiScalars) + sizeof(Control);
    SPMV_TRY_CUDA(lib_malloc_async(&ws.ptr, bytes, s));
    SPMV_TRY_CUDA(cudaMemsetAsync(ws.ptr, 0, bytes, s));
    char *base = static_cast<char *>(ws.ptr);
    P *r = reinterpret_cast<P *>(base);
    P *rh = reinterpret_cast<P *>(base + vec_pad);
    P *p = reinterpret_cast<P *>(base + 2 * vec_pad);
    P *v = reinterpret_cast<P *>(base + 3 * vec_pad);
    P *sv = reinterpret_cast<P *>(base + 4 * vec_pad);
    P *t = reinterpret_cast<P *>(base + 5 * vec_pad);
    P *xw = reinterpret_cast<P *>(base + 6 * vec_pad);
    double *partial = reinterpret_cast<double *>(base + 7 * vec_pad);
    BiScalars *sc = reinterpret_cast<BiScalars *>(partial + 2 * kRedBlocks);
    Control *ctl = reinterpret_cast<Control *>(sc + 1);
    const P *cr = r, *crh = rh, *cp = p, *cv = v, *csv = sv, *ct = t;

    // bb = b.b; r = b - A x; r_hat = r; rho_0 = (r_hat, r); rr_0 = (r, r); rho_-1 = alpha = omega = 1
    SPMV_TRY_CUDA(cudaMemcpyAsync(r, b, vec, cudaMemcpyDeviceToDevice, s));
    SPMV_TRY_CUDA(launch(k_dot<T, 4>, s, units, cr, cr, partial, ctl, &sc->bb));
    SPMV_TRY_CUDA(cudaMemcpyAsync(xw, x, vec, cudaMemcpyDeviceToDevice, s));
    SPMV_TRY(spmv_apply_ex(h, -1.0, xw, 1.0, r, s));
    SPMV_TRY_CUDA(cudaMemcpyAsync(rh, r, vec, cudaMemcpyDeviceToDevice, s));
    SPMV_TRY_CUDA(launch(k_dot<T, 4>, s, units, cr, cr, partial, ctl, &sc->rr[0]));
    SPMV_TRY_CUDA(launch(k_dot<T, 4>, s, units, crh, cr, partial, ctl, &sc->rho[0]));
    const double one = 1.0;
    SPMV_TRY_CUDA(cudaMemcpyAsync(&sc->rho[1], &one, sizeof(double), cudaMemcpyHostToDevice, s));
    SPMV_TRY_CUDA(cudaMemcpyAsync(&sc->alpha, &one, sizeof(double), cudaMemcpyHostToDevice, s));
    SPMV_TRY_CUDA(cudaMemcpyAsync(&sc->omega, &one, sizeof(double), cudaMemcpyHostToDevice, s));
    BiScalars hs{};
    SPMV_TRY_CUDA(cudaMemcpyAsync(&hs, sc, sizeof(hs), cudaMemcpyDeviceToHost, s));
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    const double denom = hs.bb > 0.0 ? hs.bb : 1.0;  // b = 0: absolute residual
    const double stop_rr = rtol * rtol * denom;

    int32_t launched = 0;
    Control hc{};
    if (max_iter > 0 && hs.rr[0] > stop_rr) {
        Pacer pace;
        pace.s = s;
        SPMV_TRY(pace.init());
        for (; launched < max_iter; ++launched) {
            bool stop = false;
            SPMV_TRY(pace.wait(launched, &stop));
            if (stop) break;
            const int cur = launched & 1;
            SPMV_TRY_CUDA(launch(k_bi_p<T, kUnroll>, s, units, static_cast<const BiScalars *>(sc), ctl, pace.dev, cur,
                                 cr, cv, p));
            SPMV_TRY(spmv_apply(h, p, v, s));
            SPMV_TRY_CUDA(launch(k_dot<T, 4>, s, units, crh, cv, partial, ctl, &sc->rv));
            SPMV_TRY_CUDA(launch(k_bi_s<T, kUnroll>, s, units, sc, ctl, pace.dev, cur, cr, cv, sv));
            SPMV_TRY(spmv_apply(h, sv, t, s));
            SPMV_TRY_CUDA(launch(k_bi_tt<T, kUnroll>, s, units, sc, ctl, ct, csv, partial));
            SPMV_TRY_CUDA(launch(k_bi_xr<T, kUnroll>, s, units, sc, ctl, pace.dev, cur, stop_rr, cp, csv, ct, crh, xw,
                                 r, partial));
        }
        SPMV_TRY_CUDA(cudaMemcpyAsync(x, xw, vec, cudaMemcpyDeviceToDevice, s));
        SPMV_TRY_CUDA(cudaMemcpyAsync(&hs, sc, sizeof(hs), cudaMemcpyDeviceToHost, s));
        SPMV_TRY_CUDA(cudaMemcpyAsync(&hc, ctl, sizeof(hc), cudaMemcpyDeviceToHost, s));
        SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    }
    const double rr = hs.rr[hc.iterations & 1];
    if (iterations) *iterations = hc.iterations;
    if (relative_residual) *relative_residual = std::sqrt(rr / denom);
    if (hc.stop == 2) return set_error(SPMV_ERR_UNSUPPORTED, "BiCGSTAB broke down (rho, (r_hat, Ap) or omega is 0)");
    return SPMV_OK;
}


// ---------------------------------------------------------------------------
// GMRES(m) (Saad and Schultz), unpreconditioned, restarted
// ---------------------------------------------------------------------------
constexpr int kGmMax = 64;  // longest restart (Krylov dimension of a cycle)
constexpr int kGmTile = 8;  // dot products a thread accumulates at once

// Small state of a GMRES solve, in device memory.  H holds the rotated Hessenberg
// matrix column by column: entry (i, j) at H[j * (kGmMax + 1) + i].
struct GmScalars {
    double tol;   // rtol * ||b|| (||b|| -> 1 when b = 0)
    double beta;  // ||b - A x|| at the last restart
    double inv;   // 1 / ||w|| (or 1 / beta) for the scale kernel
    double d1[kGmMax + 1];  // V^T w, first Gram-Schmidt pass
    double d2[kGmMax + 1];  // second pass
    double H[(kGmMax + 1) * kGmMax];
    double cs[kGmMax], sn[kGmMax];
    double g[kGmMax + 1];
    double y[kGmMax];
    int32_t steps;       // Arnoldi steps of the running cycle
    int32_t cycle_done;  // the running cycle has ended
    int32_t max_iter;
    int32_t m;
};

__device__ __forceinline__ void gm_publish(Progress *pg, const Control *ctl, const GmScalars *gs) {
    volatile Progress *v = pg;
    v->iterations = ctl->iterations;
    v->stop = ctl->stop || gs->cycle_done;
    __threadfence_system();
}

// True in every thread of the last block to finish; resets the arrival count.
__device__ __forceinline__ bool last_block(Control *ctl) {
    __shared__ bool is_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        is_last = atomicAdd(&ctl->arrivals, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (is_last) {
        __threadfence();
        if (threadIdx.x == 0) ctl->arrivals = 0;
    }
    return is_last;
}

// out[k] = V_k . w for k < nk (V_k at V + k * units), kGmTile dot products at a time;
// per-block partials, then each sum over blocks in block order by one warp of the last
// block.  which = 1 writes d1, 2 writes d2.
template <typename T>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_gm_dot(int64_t units, const Pack<T> *__restrict__ V, int nk, const Pack<T> *__restrict__ w,
             double *__restrict__ partial, Control *ctl, GmScalars *gs, int which) {
    allow_dependents();
    grid_wait();
    if (ctl->stop || gs->cycle_done) return;
    using A = typename Acc<T>::type;
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int k0 = 0; k0 < nk; k0 += kGmTile) {
        A acc[kGmTile];
#pragma unroll
        for (int t = 0; t < kGmTile; ++t) acc[t] = 0;
        for (int64_t u = gtid(); u < units; u += st) {
            const Pack<T> pw = w[u];
#pragma unroll
            for (int t = 0; t < kGmTile; ++t) {
                if (k0 + t < nk) {
                    const Pack<T> pv = V[static_cast<int64_t>(k0 + t) * units + u];
#pragma unroll
                    for (int l = 0; l < Pack<T>::L; ++l)
                        acc[t] = fma(static_cast<A>(pv.v[l]), static_cast<A>(pw.v[l]), acc[t]);
                }
            }
        }
        for (int t = 0; t < kGmTile && k0 + t < nk; ++t) {
            const double bs = block_sum(static_cast<double>(acc[t]));
            if (threadIdx.x == 0) partial[static_cast<int64_t>(k0 + t) * gridDim.x + blockIdx.x] = bs;
            __syncthreads();  // warp_sum is reused
        }
    }
    if (!last_block(ctl)) return;
    double *out = which == 1 ? gs->d1 : gs->d2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int k = warp; k < nk; k += kRedThreads / 32) {
        double s = 0.0;
        for (int i = lane; i < static_cast<int>(gridDim.x); i += 32) s += __ldcg(partial + static_cast<int64_t>(k) * gridDim.x + i);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) out[k] = s;
    }
}

// Arnoldi column j, by one thread once ||w||^2 is summed: H(:, j) = d1 + d2 with
// h_{j+1} = ||w||; the earlier rotations, the new one, the rotated right-hand side g
// and the end-of-cycle test.
__device__ void gm_column(Control *ctl, GmScalars *gs, Progress *pg, int j, double ww) {
    const double hn = sqrt(ww);
    double *col = gs->H + static_cast<int64_t>(j) * (kGmMax + 1);
    for (int i = 0; i <= j; ++i) col[i] = gs->d1[i] + gs->d2[i];
    col[j + 1] = hn;
    for (int i = 0; i < j; ++i) {
        const double a = col[i], b = col[i + 1];
        col[i] = gs->cs[i] * a + gs->sn[i] * b;
        col[i + 1] = -gs->sn[i] * a + gs->cs[i] * b;
    }
    const double rho = hypot(col[j], col[j + 1]);
    const double c = rho > 0.0 ? col[j] / rho : 1.0;
    const double s = rho > 0.0 ? col[j + 1] / rho : 0.0;
    gs->cs[j] = c;
    gs->sn[j] = s;
    col[j] = c * col[j] + s * col[j + 1];
    col[j + 1] = 0.0;
    const double gj = gs->g[j];
    gs->g[j + 1] = -s * gj;
    gs->g[j] = c * gj;
    gs->steps = j + 1;
    ctl->iterations += 1;
    const bool met = !(fabs(gs->g[j + 1]) > gs->tol);  // NaN ends the cycle too
    if (met || hn == 0.0 || ctl->iterations >= gs->max_iter || j + 1 == gs->m) gs->cycle_done = 1;
    gs->inv = hn > 0.0 ? 1.0 / hn : 0.0;
    gm_publish(pg, ctl, gs);
}

// w += sign * sum_{k < nk} coef_k V_k, coef = d1 (which 1), d2 (2) or y (3); nk < 0 takes
// the cycle's step count.  column >= 0: also ||w||^2, and the last block finishes
// Arnoldi column `column`.  During a cycle (which 1, 2) the kernel does nothing once
// the cycle has ended; the update of x (which 3) only once the solve has stopped.
template <typename T>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_gm_axpy(int64_t units, const Pack<T> *__restrict__ V, int nk, int which, double sign, Pack<T> *__restrict__ w,
              double *__restrict__ partial, Control *ctl, GmScalars *gs, Progress *pg, int column) {
    __shared__ double s_coef[kGmMax + 1];
    allow_dependents();
    grid_wait();
    if (ctl->stop || (which != 3 && gs->cycle_done)) return;
    if (nk < 0) nk = gs->steps;
    const double *coef = which == 1 ? gs->d1 : which == 2 ? gs->d2 : gs->y;
    for (int i = threadIdx.x; i < nk; i += blockDim.x) s_coef[i] = sign * coef[i];
    __syncthreads();
    using A = typename Acc<T>::type;
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    A ss = 0;
    for (int64_t u = gtid(); u < units; u += st) {
        Pack<T> pw = w[u];
#pragma unroll 4
        for (int k = 0; k < nk; ++k) {
            const Pack<T> pv = V[static_cast<int64_t>(k) * units + u];
            const T c = static_cast<T>(s_coef[k]);
#pragma unroll
            for (int l = 0; l < Pack<T>::L; ++l) pw.v[l] = fma(c, pv.v[l], pw.v[l]);
        }
        w[u] = pw;
        if (column >= 0)
#pragma unroll
            for (int l = 0; l < Pack<T>::L; ++l) ss = fma(static_cast<A>(pw.v[l]), static_cast<A>(pw.v[l]), ss);
    }
    if (column < 0) return;
    const double bs = block_sum(static_cast<double>(ss));
    if (threadIdx.x == 0) partial[blockIdx.x] = bs;
    if (!last_block(ctl)) return;
    double s = 0.0;
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += blockDim.x) s += __ldcg(partial + i);
    const double total = block_sum(s);
    if (threadIdx.x == 0) gm_column(ctl, gs, pg, column, total);
}

// v *= inv (the new basis vector, or r / beta at a restart)
template <typename T>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_gm_scale(int64_t units, Pack<T> *__restrict__ v, Control *ctl, const GmScalars *gs) {
    allow_dependents();
    grid_wait();
    if (ctl->stop || gs->cycle_done) return;
    const T inv = static_cast<T>(gs->inv);
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t u = gtid(); u < units; u += st) {
        Pack<T> p = v[u];
#pragma unroll
        for (int l = 0; l < Pack<T>::L; ++l) p.v[l] *= inv;
        v[u] = p;
    }
}

// y = R^-1 g by back-substitution over the cycle's steps (one thread); a zero pivot
// is a breakdown (stop = 2).
__global__ void k_gm_solve(Control *ctl, GmScalars *gs, Progress *pg) {
    if (threadIdx.x != 0 || ctl->stop) return;
    const int n = gs->steps;
    for (int i = n - 1; i >= 0; --i) {
        const double piv = gs->H[static_cast<int64_t>(i) * (kGmMax + 1) + i];
        if (piv == 0.0) {
            ctl->stop = 2;
            gm_publish(pg, ctl, gs);
            return;
        }
        double t = gs->g[i];
        for (int l = i + 1; l < n; ++l) t -= gs->H[static_cast<int64_t>(l) * (kGmMax + 1) + i] * gs->y[l];
        gs->y[i] = t / piv;
    }
}

// ||r|| at a restart (r = b - A x in v_0): the convergence test on the true residual,
// then g = beta e_1 and a fresh cycle.
template <typename T>
__global__ void __launch_bounds__(kRedThreads, kRedBlocksPerSm)
    k_gm_restart(int64_t units, const Pack<T> *__restrict__ r, double *__restrict__ partial, Control *ctl,
                 GmScalars *gs, Progress *pg) {
    allow_dependents();
    grid_wait();
    if (ctl->stop) return;
    using A = typename Acc<T>::type;
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    A ss = 0;
    for (int64_t u = gtid(); u < units; u += st) {
        const Pack<T> p = r[u];
#pragma unroll
        for (int l = 0; l < Pack<T>::L; ++l) ss = fma(static_cast<A>(p.v[l]), static_cast<A>(p.v[l]), ss);
    }
    const double bs = block_sum(static_cast<double>(ss));
    if (threadIdx.x == 0) partial[blockIdx.x] = bs;
    if (!last_block(ctl)) return;
    double s = 0.0;
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += blockDim.x) s += __ldcg(partial + i);
    const double total = block_sum(s);
    if (threadIdx.x == 0) {
        const double beta = sqrt(total);
        gs->beta = beta;
        if (!(beta > gs->tol)) ctl->stop = 1;  // converged (NaN stops too)
        gs->g[0] = beta;
        for (int i = 1; i <= kGmMax; ++i) gs->g[i] = 0.0;
        gs->steps = 0;
        gs->cycle_done = 0;
        gs->inv = beta > 0.0 ? 1.0 / beta : 0.0;
        gm_publish(pg, ctl, gs);
    }
}


template <typename T>
int gmres(spmv_handle_t h, const T *b, T *x, int32_t m, double rtol, int32_t max_iter, cudaStream_t s,
          int32_t *iterations, double *relative_residual) {
    using P = Pack<T>;
    const int64_t n = h->n;
    const size_t vec = static_cast<size_t>(n) * sizeof(T);
    const size_t vec_pad = (vec + 255) / 256 * 256;
    const int64_t units = static_cast<int64_t>(vec_pad / sizeof(P));
    // workspace: V (m + 1 vectors) | x (zero-padded) | partial sums ((kGmMax + 1) arrays) |
    // GMRES scalars | control
    StreamBuffer ws;
    ws.s = s;
    const size_t bytes = static_cast<size_t>(m + 2) * vec_pad + static_cast<size_t>(kGmMax + 1) * kRedBlocks * sizeof(double) +
                         sizeof(GmScalars) + sizeof(Control);
    SPMV_TRY_CUDA(lib_malloc_async(&ws.ptr, bytes, s));
    SPMV_TRY_CUDA(cudaMemsetAsync(ws.ptr, 0, bytes, s));
    char *base = static_cast<char *>(ws.ptr);
    P *V = reinterpret_cast<P *>(base);
    P *xw = reinterpret_cast<P *>(base + static_cast<size_t>(m + 1) * vec_pad);
    double *partial = reinterpret_cast<double *>(base + static_cast<size_t>(m + 2) * vec_pad);
    GmScalars *gs = reinterpret_cast<GmScalars *>(partial + static_cast<size_t>(kGmMax + 1) * kRedBlocks);
    Control *ctl = reinterpret_cast<Control *>(gs + 1);

    // ||b|| for the tolerance (v_0 holds b meanwhile)
    SPMV_TRY_CUDA(cudaMemcpyAsync(V, b, vec, cudaMemcpyDeviceToDevice, s));
    SPMV_TRY_CUDA(launch(k_dot<T, 4>, s, units, static_cast<const P *>(V), static_cast<const P *>(V), partial, ctl,
                         &gs->beta));
    double bb = 0.0;
    SPMV_TRY_CUDA(cudaMemcpyAsync(&bb, &gs->beta, sizeof(bb), cudaMemcpyDeviceToHost, s));
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    const double denom = bb > 0.0 ? std::sqrt(bb) : 1.0;  // b = 0: absolute residual
    const double tol = rtol * denom;
    SPMV_TRY_CUDA(cudaMemcpyAsync(&gs->tol, &tol, sizeof(tol), cudaMemcpyHostToDevice, s));
    SPMV_TRY_CUDA(cudaMemcpyAsync(&gs->max_iter, &max_iter, sizeof(max_iter), cudaMemcpyHostToDevice, s));
    SPMV_TRY_CUDA(cudaMemcpyAsync(&gs->m, &m, sizeof(m), cudaMemcpyHostToDevice, s));

    Pacer pace;
    pace.s = s;
    SPMV_TRY(pace.init());
    // r = b - A x into v_0, its norm (the first convergence test) and v_0 = r / beta
    SPMV_TRY_CUDA(cudaMemcpyAsync(xw, x, vec, cudaMemcpyDeviceToDevice, s));
    SPMV_TRY(spmv_apply_ex(h, -1.0, xw, 1.0, V, s));
    SPMV_TRY_CUDA(launch(k_gm_restart<T>, s, units, static_cast<const P *>(V), partial, ctl, gs, pace.dev));
    SPMV_TRY_CUDA(launch(k_gm_scale<T>, s, units, V, ctl, static_cast<const GmScalars *>(gs)));

    Control hc{};
    for (;;) {
        SPMV_TRY_CUDA(cudaMemcpyAsync(&hc, ctl, sizeof(hc), cudaMemcpyDeviceToHost, s));
        SPMV_TRY_CUDA(cudaStreamSynchronize(s));
        if (hc.stop || hc.iterations >= max_iter) break;
        // one cycle: Arnoldi steps paced on the progress record, which the step that ends
        // the cycle marks stopped
        pace.host->iterations = hc.iterations;
        pace.host->stop = 0;
        int32_t launched = hc.iterations;
        for (int j = 0; j < m && launched < max_iter; ++j, ++launched) {
            bool stop = false;
            SPMV_TRY(pace.wait(launched, &stop));
            if (stop) break;
            P *vj = V + static_cast<int64_t>(j) * units;
            P *w = V + static_cast<int64_t>(j + 1) * units;
            SPMV_TRY(spmv_apply(h, vj, w, s));
            SPMV_TRY_CUDA(launch(k_gm_dot<T>, s, units, static_cast<const P *>(V), j + 1, static_cast<const P *>(w),
                                 partial, ctl, gs, 1));
            SPMV_TRY_CUDA(launch(k_gm_axpy<T>, s, units, static_cast<const P *>(V), j + 1, 1, -1.0, w, partial, ctl,
                                 gs, pace.dev, -1));
            SPMV_TRY_CUDA(launch(k_gm_dot<T>, s, units, static_cast<const P *>(V), j + 1, static_cast<const P *>(w),
                                 partial, ctl, gs, 2));
            SPMV_TRY_CUDA(launch(k_gm_axpy<T>, s, units, static_cast<const P *>(V), j + 1, 2, -1.0, w, partial, ctl,
                                 gs, pace.dev, j));
            SPMV_TRY_CUDA(launch(k_gm_scale<T>, s, units, w, ctl, static_cast<const GmScalars *>(gs)));
        }
        // end of the cycle: y = R^-1 g, x += V y, then r = b - A x and the restart test
        k_gm_solve<<<1, 32, 0, s>>>(ctl, gs, pace.dev);
        SPMV_TRY_CUDA(cudaGetLastError());
        SPMV_TRY_CUDA(launch(k_gm_axpy<T>, s, units, static_cast<const P *>(V), -1, 3, 1.0, xw, partial, ctl, gs,
                             pace.dev, -1));
        SPMV_TRY_CUDA(cudaMemcpyAsync(V, b, vec, cudaMemcpyDeviceToDevice, s));
        SPMV_TRY(spmv_apply_ex(h, -1.0, xw, 1.0, V, s));
        SPMV_TRY_CUDA(launch(k_gm_restart<T>, s, units, static_cast<const P *>(V), partial, ctl, gs, pace.dev));
        SPMV_TRY_CUDA(launch(k_gm_scale<T>, s, units, V, ctl, static_cast<const GmScalars *>(gs)));
    }
    double beta = 0.0;
    SPMV_TRY_CUDA(cudaMemcpyAsync(x, xw, vec, cudaMemcpyDeviceToDevice, s));
    SPMV_TRY_CUDA(cudaMemcpyAsync(&beta, &gs->beta, sizeof(beta), cudaMemcpyDeviceToHost, s));
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    if (iterations) *iterations = hc.iterations;
    if (relative_residual) *relative_residual = beta / denom;
    if (hc.stop == 2)
        return set_error(SPMV_ERR_UNSUPPORTED, "GMRES broke down: zero pivot (A singular on the Krylov space)");
    return SPMV_OK;
}

}  // namespace
}  // namespace spmv

using namespace spmv;

namespace {
// b and x: device memory of the current device, which must be the handle's
int check_solve_vectors(spmv_handle_t h, const void *b, const void *x) {
    int dev = -1;
    SPMV_TRY_CUDA(cudaGetDevice(&dev));
    if (dev != h->device)
        return set_error(SPMV_ERR_INVALID_ARG, "the handle belongs to CUDA device " + std::to_string(h->device) +
                                                   " but device " + std::to_string(dev) + " is current");
    if (!device_memory_here(b) || !device_memory_here(x))
        return set_error(SPMV_ERR_INVALID_ARG, "b and x must be device memory of the current device");
    return SPMV_OK;
}

// two vectors of the handle's n values share a byte
bool overlapping(spmv_handle_t h, const void *a, const void *b) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    const uintptr_t bytes = static_cast<uintptr_t>(h->n) * value_bytes(h->dtype);
    return pa < pb + bytes && pb < pa + bytes;
}
}  // namespace

extern "C" SPMV_API int spmv_cg(spmv_handle_t h, const void *b, void *x, double rtol, int32_t max_iter,
                                void *stream, int32_t *iterations, double *relative_residual) {
    if (iterations) *iterations = 0;
    if (relative_residual) *relative_residual = 0.0;
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (max_iter < 0 || !(rtol >= 0.0)) return set_error(SPMV_ERR_INVALID_ARG, "need max_iter >= 0 and rtol >= 0");
    if (h->n == 0) return SPMV_OK;
    if (!b || !x) return set_error(SPMV_ERR_INVALID_ARG, "NULL b or x");
    if (overlapping(h, b, x)) return set_error(SPMV_ERR_INVALID_ARG, "b and x must not overlap");
    SPMV_TRY(check_solve_vectors(h, b, x));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (h->dtype == SPMV_F64)
        return cg<double>(h, static_cast<const double *>(b), static_cast<double *>(x), rtol, max_iter, s, iterations,
                          relative_residual);
    return cg<float>(h, static_cast<const float *>(b), static_cast<float *>(x), rtol, max_iter, s, iterations,
                     relative_residual);
}

extern "C" SPMV_API int spmv_bicgstab(spmv_handle_t h, const void *b, void *x, double rtol, int32_t max_iter,
                                      void *stream, int32_t *iterations, double *relative_residual) {
    if (iterations) *iterations = 0;
    if (relative_residual) *relative_residual = 0.0;
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (max_iter < 0 || !(rtol >= 0.0)) return set_error(SPMV_ERR_INVALID_ARG, "need max_iter >= 0 and rtol >= 0");
    if (h->n == 0) return SPMV_OK;
    if (!b || !x) return set_error(SPMV_ERR_INVALID_ARG, "NULL b or x");
    if (overlapping(h, b, x)) return set_error(SPMV_ERR_INVALID_ARG, "b and x must not overlap");
    SPMV_TRY(check_solve_vectors(h, b, x));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (h->dtype == SPMV_F64)
        return bicgstab<double>(h, static_cast<const double *>(b), static_cast<double *>(x), rtol, max_iter, s,
                                iterations, relative_residual);
    return bicgstab<float>(h, static_cast<const float *>(b), static_cast<float *>(x), rtol, max_iter, s, iterations,
                           relative_residual);
}

extern "C" SPMV_API int spmv_gmres(spmv_handle_t h, const void *b, void *x, int32_t restart, double rtol,
                                   int32_t max_iter, void *stream, int32_t *iterations, double *relative_residual) {
    if (iterations) *iterations = 0;
    if (relative_residual) *relative_residual = 0.0;
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (max_iter < 0 || !(rtol >= 0.0)) return set_error(SPMV_ERR_INVALID_ARG, "need max_iter >= 0 and rtol >= 0");
    if (restart < 1 || restart > kGmMax)
        return set_error(SPMV_ERR_INVALID_ARG, "restart must lie in [1, " + std::to_string(kGmMax) + "]");
    if (h->n == 0) return SPMV_OK;
    if (!b || !x) return set_error(SPMV_ERR_INVALID_ARG, "NULL b or x");
    if (overlapping(h, b, x)) return set_error(SPMV_ERR_INVALID_ARG, "b and x must not overlap");
    SPMV_TRY(check_solve_vectors(h, b, x));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (h->dtype == SPMV_F64)
        return gmres<double>(h, static_cast<const double *>(b), static_cast<double *>(x), restart, rtol, max_iter, s,
                             iterations, relative_residual);
    return gmres<float>(h, static_cast<const float *>(b), static_cast<float *>(x), restart, rtol, max_iter, s,
                        iterations, relative_residual);
}
