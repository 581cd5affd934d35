// spmv_probe_gather: the random-gather rates of the device, the ceiling of the matrices
// whose x accesses have no locality (uniformly random columns; the short rows of a
// power-law matrix).  On such a matrix every x access of a warp touches its own
// 32-byte sector, and the sliced kernels can go no faster than the device serves
// scattered accesses, whatever the bandwidth left to the streamed matrix entries.
//
// An SM sends its L1 misses to L2 as one request per 128-byte line, carrying the
// line's sectors that the warp instruction needs, and two limits apply at once: the
// requests an SM can send per clock, and the sectors the L2 can return.  Lanes whose
// columns fall into one line (a long row's sorted columns) share a request.  So the
// probe has two shapes:
//   sectors_per_line = 1  every lane gathers its own random element: one request per
//                         gather (the request rate);
//   sectors_per_line = 2, 4  groups of that many consecutive lanes read distinct
//                         sectors of one random line (the sector rate, with fewer
//                         requests).
// Each thread draws its positions from a 32-bit linear congruential sequence mapped
// onto [0, n) (or onto the whole lines of x) by a multiply-high, so there is no index
// stream, and gathers eight at a time (eight independent loads in flight, as the sliced
// kernels keep), through the same read-only load path.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_util.cuh"
#include "spmv_internal.cuh"

namespace spmv {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeInFlight = 8;

template <typename T, int SPL>
__global__ void __launch_bounds__(kProbeThreads) k_probe_gather(const T *__restrict__ x, uint32_t n, int64_t rounds,
                                                              uint32_t seed, double *__restrict__ out) {
    constexpr uint32_t kPerSector = 32 / sizeof(T), kPerLine = 128 / sizeof(T);
    const uint32_t lig = threadIdx.x % SPL;  // lane within its group of SPL
    // distinct starting states per group of SPL lanes (a multiplicative hash of the
    // group's first thread index), so that the lanes of a group draw the same lines
    const uint32_t tid = blockIdx.x * kProbeThreads + threadIdx.x - lig;
    uint32_t state = (tid + 1u) * 2654435761u ^ seed;
    const uint32_t lines = n / kPerLine;  // whole lines of x (SPL > 1 only)
    T acc = T(0);
    for (int64_t r = 0; r < rounds; ++r) {
        uint32_t idx[kProbeInFlight];
#pragma unroll
        for (int u = 0; u < kProbeInFlight; ++u) {
            state = state * 1664525u + 1013904223u;
            if (SPL == 1)
                idx[u] = __umulhi(state, n);  // in [0, n)
            else  // sector lig of a line in [0, lines): below lines * kPerLine <= n
                idx[u] = __umulhi(state, lines) * kPerLine + lig * kPerSector;
        }
        T v[kProbeInFlight];
#pragma unroll
        for (int u = 0; u < kProbeInFlight; ++u) v[u] = __ldg(x + idx[u]);
#pragma unroll
        for (int u = 0; u < kProbeInFlight; ++u) acc += v[u];
    }
    // keep the loads: one sum per block into *out
    double s = static_cast<double>(acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    __shared__ double warp_sum[kProbeThreads / 32];
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < kProbeThreads / 32; ++w) t += warp_sum[w];
        atomicAdd(out, t);
    }
}

template <typename T>
cudaError_t probe_launch(int spl, unsigned blocks, cudaStream_t s, const void *x, uint32_t n, int64_t rounds,
                         void *out) {
    const T *xp = static_cast<const T *>(x);
    double *o = static_cast<double *>(out);
    const uint32_t seed = 0x9e3779b9u;
    if (spl == 1)
        k_probe_gather<T, 1><<<blocks, kProbeThreads, 0, s>>>(xp, n, rounds, seed, o);
    else if (spl == 2)
        k_probe_gather<T, 2><<<blocks, kProbeThreads, 0, s>>>(xp, n, rounds, seed, o);
    else
        k_probe_gather<T, 4><<<blocks, kProbeThreads, 0, s>>>(xp, n, rounds, seed, o);
    return cudaGetLastError();
}

}  // namespace
}  // namespace spmv

using namespace spmv;

extern "C" SPMV_API int spmv_probe_gather(const void *x, int64_t n, int dtype, int sectors_per_line, int64_t gathers,
                                          void *out_sum, void *stream, int64_t *gathers_done) {
    if (!x || !out_sum || n <= 0 || n >= (int64_t(1) << 31) || gathers < 0)
        return set_error(SPMV_ERR_INVALID_ARG, "need x, out_sum, 0 < n < 2^31 and gathers >= 0");
    if (dtype != SPMV_F64 && dtype != SPMV_F32)
        return set_error(SPMV_ERR_INVALID_ARG, "dtype must be SPMV_F64 or SPMV_F32");
    if (sectors_per_line != 1 && sectors_per_line != 2 && sectors_per_line != 4)
        return set_error(SPMV_ERR_INVALID_ARG, "sectors_per_line must be 1, 2 or 4");
    const int64_t per_line = dtype == SPMV_F64 ? 16 : 32;
    if (sectors_per_line > 1 && n < per_line)
        return set_error(SPMV_ERR_INVALID_ARG, "sectors_per_line > 1 needs x to hold one 128-byte line");
    if (!device_memory_here(x) || !device_memory_here(out_sum))
        return set_error(SPMV_ERR_INVALID_ARG, "x and out_sum must be device memory of the current device");
    int dev = 0, sms = 0;
    SPMV_TRY_CUDA(cudaGetDevice(&dev));
    SPMV_TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    // a full wave: 2048 resident threads on every SM
    const int64_t blocks = static_cast<int64_t>(sms) * (2048 / kProbeThreads);
    const int64_t per_round = blocks * kProbeThreads * kProbeInFlight;
    const int64_t rounds = (gathers + per_round - 1) / per_round;
    if (gathers_done) *gathers_done = rounds * per_round;
    if (rounds == 0) return SPMV_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint32_t nn = static_cast<uint32_t>(n);
    const unsigned nb = static_cast<unsigned>(blocks);
    SPMV_TRY_CUDA(dtype == SPMV_F64 ? probe_launch<double>(sectors_per_line, nb, s, x, nn, rounds, out_sum)
                                    : probe_launch<float>(sectors_per_line, nb, s, x, nn, rounds, out_sum));
    return SPMV_OK;
}
