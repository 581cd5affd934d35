// spmv_csr_apply_noalloc: y = A x straight from a caller's CSR without any device
// allocation.  The only scratch the computation needs -- one carry (row, partial
// sum) per CTA of the merge-path pass -- lives in a fixed array of this library's
// own device memory, declared below.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

#include "spmv_internal.cuh"

namespace spmv {
namespace {

// Largest number of merge-path CTAs (2048 path items each) the fixed scratch serves:
// n + nnz <= kNoAllocMaxCtas * kMergeItems = 134,217,728.
constexpr int64_t kNoAllocMaxCtas = 65536;
// carry values (double) first, then carry rows (int32): 768 KiB in total.
constexpr size_t kNoAllocScratchBytes = kNoAllocMaxCtas * (sizeof(double) + sizeof(int32_t));

// Every device that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_address[kMaxDevices] = {};

// The cached address is still this device's array: a cudaDeviceReset ends the context
// that held it, and the reloaded module may place the array elsewhere.
bool still_valid(void *p, int dev) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return attr.type == cudaMemoryTypeDevice && attr.device == dev;
}

// Device address of the scratch array on the current device.  In host code the
// name g_noalloc_scratch is only a host-side stand-in, so the address is looked up
// with the device current, on the first call on each device, and cached; every call
// checks the cached address before use and looks it up again if the device was reset.
int scratch_address(void **out) {
    int dev = -1;
    SPMV_TRY_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(SPMV_ERR_UNSUPPORTED, "device ordinal beyond the scratch table");
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_address[dev] && !still_valid(g_scratch_address[dev], dev)) g_scratch_address[dev] = nullptr;
    if (!g_scratch_address[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaGetSymbolAddress(no-alloc scratch)");
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return SPMV_OK;
}

}  // namespace
}  // namespace spmv

using namespace spmv;

extern "C" SPMV_API int spmv_csr_apply_noalloc(int64_t n, int64_t nnz, const int32_t *row_ptr,
                                               const int32_t *col_idx, const void *vals, int dtype,
                                               const void *x, void *y, void *stream) {
    if (n < 0 || nnz < 0 || n >= (int64_t(1) << 31) || nnz >= (int64_t(1) << 31))
        return set_error(SPMV_ERR_INVALID_ARG, "n and nnz must lie in [0, 2^31)");
    if (dtype != SPMV_F64 && dtype != SPMV_F32)
        return set_error(SPMV_ERR_INVALID_ARG, "dtype must be SPMV_F64 or SPMV_F32");
    const int64_t n_cta = merge_ctas(n, nnz);
    if (n_cta > kNoAllocMaxCtas)
        return set_error(SPMV_ERR_TOO_LARGE,
                         "n + nnz = " + std::to_string(n + nnz) + " exceeds the allocation-free limit of " +
                             std::to_string(kNoAllocMaxCtas * kMergeItems));
    if (n == 0) return SPMV_OK;
    if (!row_ptr || !x || !y || (nnz > 0 && (!col_idx || !vals)))
        return set_error(SPMV_ERR_INVALID_ARG, "NULL array");
    if (!device_memory_here(row_ptr) || !device_memory_here(x) || !device_memory_here(y) ||
        (nnz > 0 && (!device_memory_here(col_idx) || !device_memory_here(vals))))
        return set_error(SPMV_ERR_INVALID_ARG, "every array must be device memory of the current device");
    // y is written while other CTAs still read x and the matrix
    const size_t vb = value_bytes(dtype), ybytes = static_cast<size_t>(n) * vb;
    if (spans_overlap(y, ybytes, x, ybytes)) return set_error(SPMV_ERR_INVALID_ARG, "x and y overlap");
    if (spans_overlap(y, ybytes, row_ptr, static_cast<size_t>(n + 1) * sizeof(int32_t)) ||
        (nnz > 0 && (spans_overlap(y, ybytes, col_idx, static_cast<size_t>(nnz) * sizeof(int32_t)) ||
                     spans_overlap(y, ybytes, vals, static_cast<size_t>(nnz) * vb))))
        return set_error(SPMV_ERR_INVALID_ARG, "y overlaps the matrix arrays");
    void *scratch = nullptr;
    SPMV_TRY(scratch_address(&scratch));
    Segmented sg;
    sg.kind = 1;
    sg.n_rows = n;
    sg.nnz = nnz;
    sg.n_cta = n_cta;
    sg.carry_val = static_cast<double *>(scratch);
    sg.carry_row = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(scratch) + kNoAllocMaxCtas * sizeof(double));
    sg.accumulate = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Every CTA writes its own carry slot, so nothing in the scratch needs clearing.
    SPMV_TRY_CUDA(launch_merge_path_identity(dtype, n, nnz, row_ptr, col_idx, vals, x, y, sg.carry_row, sg.carry_val,
                                             n_cta, s, nullptr));
    SPMV_TRY_CUDA(launch_carry_fixup(dtype, sg, y, s));
    return SPMV_OK;
}
