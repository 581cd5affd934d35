// C-ABI entry points of the sm_103a SpMV library (declared in include/spmv.h):
// argument checks, format selection, the build sequence, apply dispatch, and the
// inspection helpers used by tests and the bench.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "spmv_internal.cuh"

namespace spmv {

namespace {
thread_local int g_last_error = SPMV_OK;
thread_local char g_last_msg[1024] = "";
}  // namespace

int set_error(int status, const std::string &msg) {
    g_last_error = status;
    std::snprintf(g_last_msg, sizeof(g_last_msg), "%s", msg.c_str());
    return status;
}

int set_cuda_error(cudaError_t err, const char *what) {
    const int st = (err == cudaErrorMemoryAllocation) ? SPMV_ERR_OOM : SPMV_ERR_CUDA;
    (void)cudaGetLastError();  // clear a non-sticky error so later calls start clean
    return set_error(st, std::string(what) + ": " + cudaGetErrorString(err));
}

// ---------------------------------------------------------------------------
// device memory of the library
// ---------------------------------------------------------------------------
namespace {
std::mutex g_mem_mutex;
std::unordered_map<void *, size_t> g_mem_live;  // every device allocation held, with its size
int64_t g_mem_bytes = 0;
std::string g_fail_value;  // SPMV_FAIL_ALLOC as last seen
long g_fail_seen = 0;      // allocations since it took that value

// SPMV_FAIL_ALLOC=k: the k-th device allocation after the variable took its current
// value fails as if the device were out of memory (once; the count restarts whenever
// the value changes, unset included).  Called with g_mem_mutex held.
bool injected_failure() {
    const char *v = std::getenv("SPMV_FAIL_ALLOC");
    const std::string cur = v ? v : "";
    if (cur != g_fail_value) {
        g_fail_value = cur;
        g_fail_seen = 0;
    }
    if (cur.empty()) return false;
    char *end = nullptr;
    const long k = std::strtol(cur.c_str(), &end, 10);
    if (end == cur.c_str() || k <= 0) return false;
    return ++g_fail_seen == k;
}

void track(void *p, size_t bytes) {
    g_mem_live[p] = bytes;
    g_mem_bytes += static_cast<int64_t>(bytes);
}

void untrack(void *p) {
    auto it = g_mem_live.find(p);
    if (it == g_mem_live.end()) return;
    g_mem_bytes -= static_cast<int64_t>(it->second);
    g_mem_live.erase(it);
}
}  // namespace

cudaError_t lib_malloc(void **p, size_t bytes) {
    std::lock_guard<std::mutex> lock(g_mem_mutex);
    *p = nullptr;
    if (injected_failure()) return cudaErrorMemoryAllocation;
    const cudaError_t e = cudaMalloc(p, bytes);
    if (e == cudaSuccess) track(*p, bytes);
    return e;
}

cudaError_t lib_malloc_async(void **p, size_t bytes, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_mem_mutex);
    *p = nullptr;
    if (injected_failure()) return cudaErrorMemoryAllocation;
    const cudaError_t e = cudaMallocAsync(p, bytes, s);
    if (e == cudaSuccess) track(*p, bytes);
    return e;
}

void lib_free(void *p) {
    if (!p) return;
    {
        std::lock_guard<std::mutex> lock(g_mem_mutex);
        untrack(p);
    }
    (void)cudaFree(p);
}

void lib_free_async(void *p, cudaStream_t s) {
    if (!p) return;
    {
        std::lock_guard<std::mutex> lock(g_mem_mutex);
        untrack(p);
    }
    (void)cudaFreeAsync(p, s);
}

void memory_held(int64_t *allocations, int64_t *bytes) {
    std::lock_guard<std::mutex> lock(g_mem_mutex);
    if (allocations) *allocations = static_cast<int64_t>(g_mem_live.size());
    if (bytes) *bytes = g_mem_bytes;
}

bool device_memory_here(const void *p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (attr.type == cudaMemoryTypeManaged) return true;
    if (attr.type != cudaMemoryTypeDevice) return false;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return attr.device == dev;
}

namespace {

void clear_error() {
    g_last_error = SPMV_OK;
    g_last_msg[0] = '\0';
}

// ---------------------------------------------------------------------------
// memory helpers
// ---------------------------------------------------------------------------
int dev_alloc(spmv_handle_t h, void **p, size_t bytes) {
    *p = nullptr;
    if (bytes == 0) return SPMV_OK;
    cudaError_t e = lib_malloc(p, bytes);
    if (e != cudaSuccess) {
        *p = nullptr;
        return set_cuda_error(e, "cudaMalloc");
    }
    h->allocations.push_back(*p);
    return SPMV_OK;
}

template <class T>
int dev_alloc_n(spmv_handle_t h, T **p, int64_t count) {
    void *q = nullptr;
    int st = dev_alloc(h, &q, static_cast<size_t>(count) * sizeof(T));
    *p = static_cast<T *>(q);
    return st;
}


// Temporary device buffers of one build call, released when it returns.
struct Temp {
    std::vector<void *> ptrs;
    ~Temp() {
        for (void *p : ptrs) lib_free(p);
    }
    template <class T>
    int get(T **p, int64_t count) {
        *p = nullptr;
        if (count <= 0) count = 1;
        void *q = nullptr;
        cudaError_t e = lib_malloc(&q, static_cast<size_t>(count) * sizeof(T));
        if (e != cudaSuccess) return set_cuda_error(e, "cudaMalloc (build temporary)");
        ptrs.push_back(q);
        *p = static_cast<T *>(q);
        return SPMV_OK;
    }
};

int check_device_pointer(const void *p, const char *name) {
    if (!device_memory_here(p))
        return set_error(SPMV_ERR_INVALID_ARG, std::string(name) + " is not device memory of the current device");
    return SPMV_OK;
}

int bits_for(uint64_t v) {
    int b = 0;
    while (v) {
        ++b;
        v >>= 1;
    }
    return b;
}

int check_fits(double bytes, const char *what) {
    size_t free_b = 0, total_b = 0;
    if (cudaMemGetInfo(&free_b, &total_b) != cudaSuccess) {
        (void)cudaGetLastError();
        return SPMV_OK;
    }
    if (bytes > 0.9 * static_cast<double>(free_b))
        return set_error(SPMV_ERR_TOO_LARGE, std::string(what) + ": layout needs " +
                                                 std::to_string(static_cast<long long>(bytes)) +
                                                 " bytes, more than the free device memory allows");
    return SPMV_OK;
}

// Allocations made after the build can fall inside a stream capture of the calling
// thread (the first apply on a capturing stream).  cudaMalloc does not enqueue work, but
// a capture in the default (global) mode forbids it as potentially unsafe; this guard
// switches the thread to the relaxed mode around such an allocation and back.
struct RelaxedCapture {
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    RelaxedCapture() { (void)cudaThreadExchangeStreamCaptureMode(&mode); }
    ~RelaxedCapture() { (void)cudaThreadExchangeStreamCaptureMode(&mode); }
};

// The row-split counters of a new scratch set must read zero before the first pass that
// uses them.  Cleared on s itself when s is not being captured (ordered before the
// apply's kernels).  On a stream being captured a memset enqueued there would only be a
// node of the graph, run when (and if) the graph is launched, while an apply enqueued
// on s outside the graph would find the counters uncleared; so they are cleared at once
// on a private stream instead (the caller is in the relaxed capture mode).
int clear_counters(int32_t *done, int64_t count, cudaStream_t s) {
    const size_t bytes = sizeof(int32_t) * static_cast<size_t>(count);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    SPMV_TRY_CUDA(cudaStreamIsCapturing(s, &cs));
    if (cs == cudaStreamCaptureStatusNone) {
        SPMV_TRY_CUDA(cudaMemsetAsync(done, 0, bytes, s));
        return SPMV_OK;
    }
    cudaStream_t z = nullptr;
    SPMV_TRY_CUDA(cudaStreamCreateWithFlags(&z, cudaStreamNonBlocking));
    cudaError_t e = cudaMemsetAsync(done, 0, bytes, z);
    if (e == cudaSuccess) e = cudaStreamSynchronize(z);
    (void)cudaStreamDestroy(z);
    SPMV_TRY_CUDA(e);
    return SPMV_OK;
}

// The apply scratch of stream s: found, or allocated on the first apply of the handle
// on s, with its row-split counters at zero.  The column and staging buffers are
// allocated later, on first need.
int acquire_scratch(spmv_handle_t h, cudaStream_t s, ApplyScratch **out) {
    std::lock_guard<std::mutex> lock(h->scratch_mutex);
    for (auto &p : h->scratch)
        if (p->stream == s) {
            *out = p.get();
            return SPMV_OK;
        }
    auto sc = std::make_unique<ApplyScratch>();
    sc->stream = s;
    const Segmented &sg = h->seg;
    RelaxedCapture relaxed;
    if ((sg.kind == 1 || sg.kind == 2) && sg.n_cta > 0) {
        SPMV_TRY(dev_alloc_n(h, &sc->carry_row, sg.n_cta));
        SPMV_TRY(dev_alloc_n(h, &sc->carry_val, sg.n_cta));
    }
    if (sg.kind == 3 && sg.n_rows > 0) {
        SPMV_TRY(dev_alloc_n(h, &sc->partial, std::max<int64_t>(sg.n_chunks, 1) * 8));  // up to 8 right-hand sides
        SPMV_TRY(dev_alloc_n(h, &sc->done, sg.n_rows));
        SPMV_TRY(clear_counters(sc->done, sg.n_rows, s));
    }
    *out = sc.get();
    h->scratch.push_back(std::move(sc));
    return SPMV_OK;
}

// An n-value column of the scratch set (tmp_x, tmp_y, x_stage, y_stage), allocated on
// its first use.
int scratch_column(spmv_handle_t h, void **slot) {
    std::lock_guard<std::mutex> lock(h->scratch_mutex);
    if (*slot) return SPMV_OK;
    RelaxedCapture relaxed;
    return dev_alloc(h, slot, static_cast<size_t>(h->n) * value_bytes(h->dtype));
}

// The segmented part with the scratch pointers of one stream's set filled in.
Segmented with_scratch(const Segmented &sg, const ApplyScratch &sc) {
    Segmented v = sg;
    v.carry_row = sc.carry_row;
    v.carry_val = sc.carry_val;
    v.partial = sc.partial;
    v.done = sc.done;
    return v;
}

const char *ordering_name(int o) {
    switch (o) {
        case SPMV_ORDER_NATURAL: return "natural";
        case SPMV_ORDER_ROW_LENGTH: return "row_length";
        case SPMV_ORDER_RCM: return "rcm";
        case SPMV_ORDER_USER: return "user";
        default: return "?";
    }
}

const char *format_name(int f) {
    switch (f) {
        case SPMV_FMT_AUTO: return "auto";
        case SPMV_FMT_CSR_VECTOR: return "csr_vector";
        case SPMV_FMT_ELL_R: return "ell_r";
        case SPMV_FMT_SELL: return "sell";
        case SPMV_FMT_HYB: return "hyb";
        case SPMV_FMT_MERGE: return "merge";
        default: return "?";
    }
}

// default long-row threshold: keeps every sequential per-thread sum short (at most 128
// terms a thread, 8 a lane for CSR-vector's 32 lanes) and sends rows that would hold a
// warp far longer than its neighbours to the row-split pass.  CSR-vector: 256 measured
// 301 us on the power-law matrix against 352 at 8192.
int32_t default_threshold(int format, int dtype) {
    if (format == SPMV_FMT_CSR_VECTOR) return 256;
    // thread-per-row layouts: longer rows would stall their warp; they go to the
    // row-split pass, which handles them with whole warps
    (void)dtype;
    return 128;
}

// HYB ELL width cap: one thread walks at most this many entries of a row
int32_t hyb_width_cap(int dtype) { return dtype == SPMV_F64 ? 4096 : 128; }

// ---------------------------------------------------------------------------
// build context
// ---------------------------------------------------------------------------
struct BuildCtx {
    spmv_handle_t h;
    cudaStream_t s;
    const int32_t *row_ptr;  // caller's
    const int32_t *col;      // caller's
    const void *val;         // caller's
    int32_t *len = nullptr;  // [n] row lengths (temporary)
    std::vector<int64_t> hist;
    int64_t n_long = 0, long_nnz = 0;
    int32_t max_short = 0;
    int32_t threshold = -1;  // -1 = no long-row cut
    int32_t group = 1;       // threads per row of the sliced apply
    int group_mode = 0;      // 0 row-grouped, 1 interleaved slots, 2 column-grouped
    bool interleaved = false;
    bool vec = false;        // one thread per row, 16-byte vector loads
    Temp temp;
};

int sync(cudaStream_t s) {
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    SPMV_TRY_CUDA(cudaGetLastError());
    return SPMV_OK;
}

// Stable partition of rows by a small bucket id (one 8-bit counting pass).
// rows_out gets the row ids grouped by bucket; bucket_start[b] = first index of bucket b.
int partition_rows(BuildCtx &c, int mode, int32_t a, int32_t forced_g, int32_t *rows_out,
                   std::vector<int64_t> &bucket_start) {
    const int64_t n = c.h->n;
    uint32_t *keys = nullptr, *keys_out = nullptr;
    int64_t *counts = nullptr, *offsets = nullptr, *scan_tmp = nullptr;
    const int64_t nb = radix_blocks(n);
    SPMV_TRY(c.temp.get(&keys, n));
    SPMV_TRY(c.temp.get(&keys_out, n));
    SPMV_TRY(c.temp.get(&counts, 256 * nb + 1));
    SPMV_TRY(c.temp.get(&offsets, 256 * nb + 1));
    SPMV_TRY(c.temp.get(&scan_tmp, scan_temp_elems(256 * nb)));
    int32_t *vals_in = nullptr;
    SPMV_TRY(c.temp.get(&vals_in, n));
    SPMV_TRY_CUDA(launch_bucket_keys(n, c.len, mode, a, forced_g, keys, vals_in, c.s));
    SPMV_TRY_CUDA(launch_radix_pass(keys, vals_in, n, 0, keys_out, rows_out, counts, offsets, scan_tmp, c.s));
    // offsets[b * nb] is where bucket b starts
    bucket_start.assign(9, n);
    std::vector<int64_t> host(8);
    for (int b = 0; b < 8; ++b)
        SPMV_TRY_CUDA(cudaMemcpyAsync(&host[b], offsets + static_cast<int64_t>(b) * nb, sizeof(int64_t),
                                      cudaMemcpyDeviceToHost, c.s));
    SPMV_TRY(sync(c.s));
    for (int b = 0; b < 8; ++b) bucket_start[b] = host[b];
    bucket_start[8] = n;
    return SPMV_OK;
}

// For merge-path, the precomputed split of every CTA boundary (so the apply kernel
// does no search).  The carries the pass writes are per-stream apply scratch.
int alloc_carries(BuildCtx &c, Segmented &sg) {
    spmv_handle_t h = c.h;
    if (sg.n_cta <= 0) return SPMV_OK;
    if (sg.kind == 1) {
        SPMV_TRY(dev_alloc_n(h, &sg.part, sg.n_cta + 1));
        SPMV_TRY_CUDA(launch_merge_partition(sg.n_rows, sg.nnz, sg.ptr, sg.n_cta, sg.part, c.s));
    }
    return SPMV_OK;
}

// Row chunks of the row-split pass (kind 3) over the compact CSR in sg (the partial
// sums and completion counters it writes are per-stream apply scratch).
int build_row_chunks(BuildCtx &c, Segmented &sg) {
    spmv_handle_t h = c.h;
    const int64_t m = sg.n_rows;
    int64_t *count = nullptr, *cptr = nullptr, *scan_tmp = nullptr;
    SPMV_TRY(c.temp.get(&count, m));
    SPMV_TRY(c.temp.get(&cptr, m + 1));
    SPMV_TRY(c.temp.get(&scan_tmp, scan_temp_elems(m)));
    // chunk length: no lane sums more than chunk / 32 terms of a row in sequence (64 in
    // float32, whose rounding bound is the tighter).  In float64, when the chunks share a
    // launch with the sliced rows (one thread per row, element loads, not staged), chunks
    // of 4096 halve the chunk warps the fused launch schedules first (power-law 163.0 ->
    // 158.1 us); a row-split launch of its own keeps 2048, whose extra warps it needs for
    // parallelism (the CSR-vector plan: 301 against 318 us).
    const bool fused = h->sliced.present && h->sliced.group == 1 && !h->sliced.vec && h->params.staged != 1;
    sg.chunk = (h->dtype == SPMV_F64 && fused) ? kSplitChunk64 : kSplitChunk;
    SPMV_TRY_CUDA(launch_chunk_counts(m, sg.ptr, sg.chunk, count, c.s));
    SPMV_TRY_CUDA(launch_exclusive_scan(count, m, cptr, scan_tmp, c.s));
    int64_t total = 0;
    SPMV_TRY_CUDA(cudaMemcpyAsync(&total, cptr + m, sizeof(int64_t), cudaMemcpyDeviceToHost, c.s));
    SPMV_TRY(sync(c.s));
    sg.n_chunks = total;
    SPMV_TRY(dev_alloc_n(h, &sg.row_chunk_ptr, m + 1));
    SPMV_TRY(dev_alloc_n(h, &sg.chunk_begin, total));
    SPMV_TRY(dev_alloc_n(h, &sg.chunk_end, total));
    SPMV_TRY(dev_alloc_n(h, &sg.chunk_row, total));
    SPMV_TRY_CUDA(launch_chunk_fill(m, sg.ptr, sg.chunk, cptr, sg.row_chunk_ptr, sg.chunk_begin, sg.chunk_end,
                                    sg.chunk_row, c.s));
    std::vector<int64_t> counts_host(static_cast<size_t>(m));
    SPMV_TRY_CUDA(cudaMemcpyAsync(counts_host.data(), count, sizeof(int64_t) * m, cudaMemcpyDeviceToHost, c.s));
    SPMV_TRY(sync(c.s));
    sg.n_multi = 0;
    for (int64_t v : counts_host) sg.n_multi += v > 1;
    return SPMV_OK;
}

// Compact CSR of the listed rows, entries from in-row position `offset` on.
int build_segment(BuildCtx &c, const int32_t *rows_dev, int64_t m, int32_t offset, int kind, int accumulate) {
    spmv_handle_t h = c.h;
    Segmented &sg = h->seg;
    sg = Segmented();
    if (m <= 0) return SPMV_OK;
    sg.kind = kind;
    sg.n_rows = m;
    sg.accumulate = accumulate;
    sg.dst_offset = offset;
    SPMV_TRY(dev_alloc_n(h, &sg.rows, m));
    SPMV_TRY_CUDA(cudaMemcpyAsync(sg.rows, rows_dev, sizeof(int32_t) * m, cudaMemcpyDeviceToDevice, c.s));
    int64_t *sizes = nullptr, *cptr = nullptr, *scan_tmp = nullptr;
    SPMV_TRY(c.temp.get(&sizes, m));
    SPMV_TRY(c.temp.get(&cptr, m + 1));
    SPMV_TRY(c.temp.get(&scan_tmp, scan_temp_elems(m)));
    SPMV_TRY_CUDA(launch_compact_sizes(m, sg.rows, c.len, offset, sizes, c.s));
    SPMV_TRY_CUDA(launch_exclusive_scan(sizes, m, cptr, scan_tmp, c.s));
    int64_t total = 0;
    SPMV_TRY_CUDA(cudaMemcpyAsync(&total, cptr + m, sizeof(int64_t), cudaMemcpyDeviceToHost, c.s));
    SPMV_TRY(sync(c.s));
    sg.nnz = total;
    const size_t vb = value_bytes(h->dtype);
    SPMV_TRY(check_fits(static_cast<double>(total) * static_cast<double>(vb + 8) + 8.0 * m, "segmented part"));
    SPMV_TRY(dev_alloc_n(h, &sg.ptr, m + 1));
    SPMV_TRY_CUDA(launch_int64_to_int32(cptr, m + 1, sg.ptr, c.s));
    SPMV_TRY(dev_alloc_n(h, &sg.col, total));
    SPMV_TRY(dev_alloc(h, &sg.val, static_cast<size_t>(total) * vb));
    if (kind == 2) SPMV_TRY(dev_alloc_n(h, &sg.coo_row, total));
    SPMV_TRY_CUDA(launch_compact_copy(h->dtype, m, sg.rows, c.row_ptr, offset, c.col, c.val, cptr, sg.col, sg.val,
                                      sg.coo_row, c.s));
    if (kind == 3) return build_row_chunks(c, sg);
    sg.n_cta = (kind == 1) ? merge_ctas(m, total) : coo_ctas(total);
    SPMV_TRY(alloc_carries(c, sg));
    return SPMV_OK;
}

// Long rows (len > threshold) leave the main format for the row-split pass.
int build_long_rows(BuildCtx &c, int accumulate) {
    if (c.n_long <= 0) return SPMV_OK;
    int32_t *rows = nullptr;
    SPMV_TRY(c.temp.get(&rows, c.h->n));
    std::vector<int64_t> start;
    SPMV_TRY(partition_rows(c, 0, c.threshold, 0, rows, start));
    const int64_t m = start[2] - start[1];
    if (m != c.n_long) return set_error(SPMV_ERR_CUDA, "long-row partition count mismatch");
    return build_segment(c, rows + start[1], m, 0, 3, accumulate);
}

// ---------------------------------------------------------------------------
// sliced part (SELL-C-sigma, ELLPACK-R, HYB's ELL)
// ---------------------------------------------------------------------------

// Kernel-name suffix of the G-threads-per-row apply: _g<G> and r (row-grouped),
// i (interleaved slots) or c (column-grouped).
std::string group_suffix(const BuildCtx &c) {
    return "_g" + std::to_string(c.group) + (c.group_mode == 2 ? "c" : c.group_mode == 1 ? "i" : "r");
}

// Threads per row of the sliced apply when not given: one, unless the rows are too few
// to give about two waves of threads (2 x SMs x 2048) at one per row and long enough to
// share; then double while that stays short of two waves and each thread keeps at least
// 16 entries of an average stored row.
int32_t auto_row_threads(int64_t n, int64_t stored, int sms) {
    if (n <= 0) return 1;
    const double target = 2.0 * sms * 2048.0;
    const double mean = static_cast<double>(stored) / static_cast<double>(n);
    int32_t g = 1;
    while (g < 32 && static_cast<double>(n) * g < target && mean >= 32.0 * g) g *= 2;
    return g;
}

// Plan: order, per-position lengths, slice widths and offsets.  `lens` are the
// lengths to store (long rows already 0).  ell_ld > 0 selects the single-slice
// ELL addressing with that leading dimension and width = max length.
int plan_sliced(BuildCtx &c, const int32_t *lens, int32_t C, int64_t sigma, int64_t ell_ld, int32_t max_len) {
    spmv_handle_t h = c.h;
    const int64_t n = h->n;
    Sliced &sl = h->sliced;
    sl = Sliced();
    sl.present = true;
    sl.sigma = sigma;
    sl.group = c.group;
    sl.log2g = bits_for(static_cast<uint64_t>(c.group)) - 1;
    sl.group_mode = c.group_mode;
    sl.interleaved = c.interleaved || c.vec;
    sl.vec = c.vec;
    if (c.vec) {  // indices in groups of 4 (16 bytes), values in 16-byte groups (2 doubles or 4 floats)
        sl.log2k_col = 2;
        sl.log2k_val = value_bytes(h->dtype) == 8 ? 1 : 2;
    } else if (c.interleaved) {
        sl.log2k_col = sl.log2k_val = sl.log2g;
    }
    const int32_t round_to = c.vec ? 4 : c.interleaved ? c.group : 1;
    if (ell_ld > 0) {
        sl.C = static_cast<int32_t>(std::min<int64_t>(ell_ld, INT32_MAX));
        sl.ld = ell_ld;
        sl.n_pos = ell_ld;
        sl.log2C = 31;
        sl.cmask = 0x7fffffffu;
        sl.stride = ell_ld;
        sl.n_slices = 1;
        sl.sigma = 1;
    } else {
        sl.C = C;
        sl.n_pos = ceil_div(n, C) * C;
        sl.log2C = bits_for(static_cast<uint64_t>(C)) - 1;
        sl.cmask = static_cast<uint32_t>(C - 1);
        sl.stride = C;
        sl.n_slices = sl.n_pos / C;
    }
    // order
    int32_t *perm_tmp = nullptr;
    if (sl.sigma > 1 && n > 1) {
        SPMV_TRY(c.temp.get(&perm_tmp, n));
        const int64_t sig = std::min<int64_t>(sl.sigma, n);
        if (sig <= kWindowSortMax) {
            SPMV_TRY_CUDA(launch_window_sort(lens, n, sig, perm_tmp, c.s));
        } else {
            const int64_t windows = ceil_div(n, sig);
            const int wbits = bits_for(static_cast<uint64_t>(windows - 1));
            const int lbits = bits_for(static_cast<uint64_t>(max_len));
            if (wbits + lbits > 32)
                return set_error(SPMV_ERR_UNSUPPORTED, "SELL sort key does not fit 32 bits for this sigma");
            const int total_bits = wbits + lbits;
            uint32_t *k0 = nullptr, *k1 = nullptr;
            int32_t *v0 = nullptr, *v1 = nullptr;
            int64_t *counts = nullptr, *offsets = nullptr, *scan_tmp = nullptr;
            const int64_t nb = radix_blocks(n);
            SPMV_TRY(c.temp.get(&k0, n));
            SPMV_TRY(c.temp.get(&k1, n));
            SPMV_TRY(c.temp.get(&v0, n));
            SPMV_TRY(c.temp.get(&v1, n));
            SPMV_TRY(c.temp.get(&counts, 256 * nb + 1));
            SPMV_TRY(c.temp.get(&offsets, 256 * nb + 1));
            SPMV_TRY(c.temp.get(&scan_tmp, scan_temp_elems(256 * nb)));
            SPMV_TRY_CUDA(launch_sort_keys(lens, n, sig, lbits, max_len, k0, v0, c.s));
            int passes = std::max(1, (total_bits + 7) / 8);
            for (int p = 0; p < passes; ++p) {
                SPMV_TRY_CUDA(launch_radix_pass(k0, v0, n, 8 * p, k1, v1, counts, offsets, scan_tmp, c.s));
                std::swap(k0, k1);
                std::swap(v0, v1);
            }
            perm_tmp = v0;
        }
        SPMV_TRY(dev_alloc_n(h, &sl.perm, sl.n_pos));
    }
    SPMV_TRY(dev_alloc_n(h, &sl.len, sl.n_pos));
    SPMV_TRY_CUDA(launch_gather_sorted(lens, perm_tmp, n, sl.n_pos, sl.len, sl.perm, c.s));
    // widths and offsets
    SPMV_TRY(dev_alloc_n(h, &sl.width, sl.n_slices));
    SPMV_TRY(dev_alloc_n(h, &sl.slice_ptr, sl.n_slices + 1));
    std::vector<int32_t> widths(static_cast<size_t>(sl.n_slices));
    if (ell_ld > 0) {
        const int32_t w = (max_len + round_to - 1) / round_to * round_to;
        widths[0] = w;
        SPMV_TRY_CUDA(cudaMemcpyAsync(sl.width, widths.data(), sizeof(int32_t), cudaMemcpyHostToDevice, c.s));
        const int64_t sp[2] = {0, ell_ld * static_cast<int64_t>(w)};
        SPMV_TRY_CUDA(cudaMemcpyAsync(sl.slice_ptr, sp, sizeof(sp), cudaMemcpyHostToDevice, c.s));
        SPMV_TRY(sync(c.s));
        sl.slots = sp[1];
        sl.padded_entries = n * static_cast<int64_t>(w);
        sl.max_width = w;
    } else {
        int64_t *sizes = nullptr, *scan_tmp = nullptr;
        SPMV_TRY(c.temp.get(&sizes, sl.n_slices));
        SPMV_TRY(c.temp.get(&scan_tmp, scan_temp_elems(sl.n_slices)));
        SPMV_TRY_CUDA(launch_slice_widths(sl.len, sl.n_slices, sl.C, sl.width, sizes, c.s, round_to));
        SPMV_TRY_CUDA(launch_exclusive_scan(sizes, sl.n_slices, sl.slice_ptr, scan_tmp, c.s));
        SPMV_TRY_CUDA(cudaMemcpyAsync(widths.data(), sl.width, sizeof(int32_t) * sl.n_slices,
                                      cudaMemcpyDeviceToHost, c.s));
        SPMV_TRY(sync(c.s));
        int64_t slots = 0, padded = 0;
        int32_t mw = 0;
        for (int64_t s = 0; s < sl.n_slices; ++s) {
            const int64_t rows_here = std::min<int64_t>(sl.C, n - s * sl.C);
            slots += static_cast<int64_t>(widths[s]) * sl.C;
            padded += static_cast<int64_t>(widths[s]) * rows_here;
            mw = std::max(mw, widths[s]);
        }
        sl.slots = slots;
        sl.padded_entries = padded;
        sl.max_width = mw;
        // the narrow tail of a global sort (widths never increase along the slices)
        if (sl.perm && sl.sigma >= n && sl.C == 32 && round_to == 1 && c.group == 1 && !c.vec) {
            bool monotone = true;
            for (int64_t s = 1; s < sl.n_slices && monotone; ++s) monotone = widths[s] <= widths[s - 1];
            if (monotone) {
                sl.has_tail = true;
                int sms = 0;
                if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c.h->device) != cudaSuccess) {
                    (void)cudaGetLastError();
                    sms = 152;
                }
                sl.tail_cap = 12 * static_cast<int64_t>(sms);
                int64_t s = 0, slot = 0;
                for (int w = kTailMaxW; w >= 0; --w) {  // first slice of width <= w, and its slot
                    while (s < sl.n_slices && widths[s] > w) slot += static_cast<int64_t>(widths[s++]) * sl.C;
                    sl.tail_slice[w] = s;
                    sl.tail_slot[w] = slot;
                }
            }
        }
    }
    return SPMV_OK;
}

int fill_sliced(BuildCtx &c) {
    spmv_handle_t h = c.h;
    Sliced &sl = h->sliced;
    const size_t vb = value_bytes(h->dtype);
    SPMV_TRY(check_fits(static_cast<double>(sl.slots) * static_cast<double>(vb + 4), "sliced part"));
    SPMV_TRY(dev_alloc_n(h, &sl.col, sl.slots));
    SPMV_TRY(dev_alloc(h, &sl.val, static_cast<size_t>(sl.slots) * vb));
    SPMV_TRY_CUDA(launch_fill_sliced(h->dtype, sl, c.row_ptr, c.col, c.val, c.s));
    return SPMV_OK;
}


// ---------------------------------------------------------------------------
// per-format builds
// ---------------------------------------------------------------------------
int build_sell_like(BuildCtx &c, int format, int32_t C, int64_t sigma) {
    spmv_handle_t h = c.h;
    int32_t *clip = nullptr;
    SPMV_TRY(c.temp.get(&clip, h->n));
    SPMV_TRY_CUDA(launch_clip_long(h->n, c.len, c.threshold, clip, c.s));
    if (format == SPMV_FMT_ELL_R) {
        const int64_t ld = ceil_div(std::max<int64_t>(h->n, 1), 32) * 32;
        SPMV_TRY(check_fits(static_cast<double>(ld) * c.max_short * static_cast<double>(value_bytes(h->dtype) + 4),
                            "ELLPACK-R"));
        SPMV_TRY(plan_sliced(c, clip, 0, 1, ld, c.max_short));
    } else {
        SPMV_TRY(plan_sliced(c, clip, C, sigma, 0, c.max_short));
    }
    h->sliced.stored_entries = h->nnz - c.long_nnz;
    if (c.n_long > 0) {
        // long rows: the sliced pass leaves their y entries to the row-split pass
        SPMV_TRY_CUDA(launch_mark_long(h->sliced.n_pos, h->sliced.perm, c.len, h->n, c.threshold, h->sliced.len,
                                       c.s));
    }
    SPMV_TRY(fill_sliced(c));
    SPMV_TRY(build_long_rows(c, 0));
    const std::string name = format == SPMV_FMT_ELL_R ? "ell_r" : "sell";
    if (c.group > 1 || c.vec) {  // grouped / vector kernel, then the long rows' chunks in a launch of their own
        h->kernels.push_back(name + (c.vec ? std::string("_v") : group_suffix(c)));
        if (h->seg.kind == 3) h->kernels.push_back("rowsplit_chunks");
    } else {
        h->kernels.push_back(h->seg.kind == 3 ? name + "+rowsplit" : name);
    }
    return SPMV_OK;
}

int build_hyb(BuildCtx &c, int32_t K, int spill_csr) {
    spmv_handle_t h = c.h;
    const int64_t n = h->n;
    h->K = K;
    int32_t *ell_len = nullptr;
    SPMV_TRY(c.temp.get(&ell_len, n));
    SPMV_TRY_CUDA(launch_min_len(n, c.len, K, ell_len, c.s));
    const int64_t ld = ceil_div(std::max<int64_t>(n, 1), 256) * 256;
    const int32_t width = std::min<int32_t>(K, h->max_len);
    SPMV_TRY(check_fits(static_cast<double>(ld) * width * static_cast<double>(value_bytes(h->dtype) + 4),
                        "HYB ELL part"));
    SPMV_TRY(plan_sliced(c, ell_len, 0, 1, ld, width));
    SPMV_TRY(fill_sliced(c));
    // spill rows: len > K
    int32_t *rows = nullptr;
    SPMV_TRY(c.temp.get(&rows, n));
    std::vector<int64_t> start;
    SPMV_TRY(partition_rows(c, 1, K, 0, rows, start));
    const int64_t m = start[2] - start[1];
    SPMV_TRY(build_segment(c, rows + start[1], m, K, spill_csr ? 1 : 2, 1));
    h->sliced.stored_entries = h->nnz - h->seg.nnz;
    h->kernels.push_back("hyb_ell" + (c.vec ? std::string("_v") : c.group > 1 ? group_suffix(c) : std::string()));
    return SPMV_OK;
}

int build_csr_vector(BuildCtx &c, int32_t forced_g) {
    spmv_handle_t h = c.h;
    const int64_t n = h->n;
    const size_t vb = value_bytes(h->dtype);
    SPMV_TRY(dev_alloc_n(h, &h->csr_col, h->nnz));
    SPMV_TRY(dev_alloc(h, &h->csr_val, static_cast<size_t>(h->nnz) * vb));
    if (h->nnz > 0) {
        SPMV_TRY_CUDA(cudaMemcpyAsync(h->csr_col, c.col, sizeof(int32_t) * h->nnz, cudaMemcpyDeviceToDevice, c.s));
        SPMV_TRY_CUDA(cudaMemcpyAsync(h->csr_val, c.val, vb * h->nnz, cudaMemcpyDeviceToDevice, c.s));
    }
    // bin sizes from the histogram (bins: <=16, <=32, <=64, <=128, longer: about eight
    // entries a lane; the device partition applies the same rule, vector_bin in build.cu)
    const int gs[5] = {2, 4, 8, 16, 32};
    std::vector<int64_t> cnt(5, 0);
    const int64_t n_short = n - c.n_long;
    if (forced_g > 0) {
        int b = 0;
        while (gs[b] != forced_g) ++b;
        cnt[b] = n_short;
    } else {
        const int32_t thr = c.threshold;
        for (int l = 0; l < kHistCap; ++l) {
            if (thr >= 0 && l > thr) continue;  // long row
            const int b = l <= 16 ? 0 : l <= 32 ? 1 : l <= 64 ? 2 : l <= 128 ? 3 : 4;
            cnt[b] += c.hist[l];
        }
        // the top bucket holds every row of kHistCap or more entries
        if (thr < 0)
            cnt[4] += c.hist[kHistCap];
        else if (thr >= kHistCap)
            cnt[4] += c.hist[kHistCap] - c.n_long;
    }
    int nonempty = 0;
    for (int b = 0; b < 5; ++b) nonempty += cnt[b] > 0;
    if (nonempty <= 1 && c.n_long == 0) {
        for (int b = 0; b < 5; ++b)
            if (cnt[b] > 0) h->bins.push_back(Bin{gs[b], cnt[b], 0});
        h->bin_rows = nullptr;
    } else {
        SPMV_TRY(dev_alloc_n(h, &h->bin_rows, n));
        std::vector<int64_t> start;
        SPMV_TRY(partition_rows(c, 2, c.threshold, forced_g, h->bin_rows, start));
        for (int b = 0; b < 5; ++b) {
            const int64_t count = start[b + 1] - start[b];
            if (count != cnt[b]) return set_error(SPMV_ERR_CUDA, "row-bin count mismatch");
            if (count > 0) h->bins.push_back(Bin{gs[b], count, start[b]});
        }
        if (c.n_long > 0) {
            if (start[7] - start[6] != c.n_long) return set_error(SPMV_ERR_CUDA, "long-row bin count mismatch");
            SPMV_TRY(build_segment(c, h->bin_rows + start[6], c.n_long, 0, 3, 0));
        }
    }
    for (const Bin &b : h->bins) h->kernels.push_back("csr_vector_g" + std::to_string(b.g));
    return SPMV_OK;
}

// Every row through merge-path over a copy of the CSR (identity row map, writes y).
int build_merge(BuildCtx &c) {
    spmv_handle_t h = c.h;
    const size_t vb = value_bytes(h->dtype);
    SPMV_TRY(dev_alloc_n(h, &h->csr_col, h->nnz));
    SPMV_TRY(dev_alloc(h, &h->csr_val, static_cast<size_t>(h->nnz) * vb));
    if (h->nnz > 0) {
        SPMV_TRY_CUDA(cudaMemcpyAsync(h->csr_col, c.col, sizeof(int32_t) * h->nnz, cudaMemcpyDeviceToDevice, c.s));
        SPMV_TRY_CUDA(cudaMemcpyAsync(h->csr_val, c.val, vb * h->nnz, cudaMemcpyDeviceToDevice, c.s));
    }
    Segmented &sg = h->seg;
    sg = Segmented();
    sg.kind = 1;
    sg.n_rows = h->n;
    sg.nnz = h->nnz;
    sg.rows = nullptr;
    sg.ptr = h->row_ptr;
    sg.col = h->csr_col;
    sg.val = h->csr_val;
    sg.accumulate = 0;
    sg.n_cta = merge_ctas(h->n, h->nnz);
    SPMV_TRY(alloc_carries(c, sg));
    h->n_long_rows = 0;
    h->long_nnz = 0;
    return SPMV_OK;
}

// Padded slot count of SELL-32 in natural order (sigma = 1), for the AUTO choice.
int probe_sigma1_slots(BuildCtx &c, int64_t *slots) {
    const int64_t n = c.h->n;
    const int64_t ns = ceil_div(n, 32);
    int32_t *clip = nullptr, *len_pad = nullptr, *width = nullptr;
    int64_t *sizes = nullptr, *sp = nullptr, *scan_tmp = nullptr;
    SPMV_TRY(c.temp.get(&clip, n));
    SPMV_TRY(c.temp.get(&len_pad, ns * 32));
    SPMV_TRY(c.temp.get(&width, ns));
    SPMV_TRY(c.temp.get(&sizes, ns));
    SPMV_TRY(c.temp.get(&sp, ns + 1));
    SPMV_TRY(c.temp.get(&scan_tmp, scan_temp_elems(ns)));
    SPMV_TRY_CUDA(launch_clip_long(n, c.len, c.threshold, clip, c.s));
    SPMV_TRY_CUDA(launch_gather_sorted(clip, nullptr, n, ns * 32, len_pad, nullptr, c.s));
    SPMV_TRY_CUDA(launch_slice_widths(len_pad, ns, 32, width, sizes, c.s));
    SPMV_TRY_CUDA(launch_exclusive_scan(sizes, ns, sp, scan_tmp, c.s));
    SPMV_TRY_CUDA(cudaMemcpyAsync(slots, sp + ns, sizeof(int64_t), cudaMemcpyDeviceToHost, c.s));
    return sync(c.s);
}

// Byte weight of a spill entry against a streamed ELL slot in the HYB width rule: a spill
// entry walked by the merge-path pass costs about four times its bytes in time (HYB on
// the HMEp-shaped matrix: 322 us at the unweighted rule's K = 13, 232 at K = 17 from
// weight 4; power-law: 369 us at K = 1, 342 at K = 3).
constexpr int64_t kSpillWeight = 4;

int32_t hyb_auto_width(const BuildCtx &c, int dtype, int64_t n, int32_t cap) {
    // smallest K with kSpillWeight * (vb + 8) * #{len > K} <= ld * (vb + 4)
    const int64_t vb = static_cast<int64_t>(value_bytes(dtype));
    const int64_t ld = ceil_div(std::max<int64_t>(n, 1), 256) * 256;
    int64_t longer = n;  // #{len > K} for K = -1
    int32_t K = 0;
    longer -= c.hist[0];
    while (K < cap && K < kHistCap && kSpillWeight * (vb + 8) * longer > ld * (vb + 4)) {
        ++K;
        longer -= c.hist[K];
    }
    return std::min(K, cap);
}

int build_all(BuildCtx &c, int format, const spmv_format_params &prm) {
    spmv_handle_t h = c.h;
    const int64_t n = h->n, nnz = h->nnz;

    SPMV_TRY(dev_alloc_n(h, &h->row_ptr, n + 1));
    SPMV_TRY_CUDA(cudaMemcpyAsync(h->row_ptr, c.row_ptr, sizeof(int32_t) * (n + 1), cudaMemcpyDeviceToDevice, c.s));

    // a1: validate + lengths
    int32_t *status = nullptr;
    SPMV_TRY(c.temp.get(&c.len, n));
    SPMV_TRY(c.temp.get(&status, 3));
    SPMV_TRY_CUDA(cudaMemsetAsync(status, 0, sizeof(int32_t) * 3, c.s));
    SPMV_TRY_CUDA(launch_validate(n, nnz, c.row_ptr, c.col, c.len, status, c.s));
    int32_t st_host[3] = {0, 0, 0};
    SPMV_TRY_CUDA(cudaMemcpyAsync(st_host, status, sizeof(st_host), cudaMemcpyDeviceToHost, c.s));
    SPMV_TRY(sync(c.s));
    if (st_host[0]) return set_error(SPMV_ERR_BAD_CSR, "row_ptr is not a valid CSR row pointer (row_ptr[0] != 0, "
                                                       "decreasing entries, or row_ptr[n] != nnz)");
    if (st_host[1]) return set_error(SPMV_ERR_BAD_CSR, "a column index lies outside [0, n)");
    h->max_len = st_host[2];
    h->mean_len = n ? static_cast<double>(nnz) / static_cast<double>(n) : 0.0;

    // a2: parameters
    int32_t thr = prm.long_row_threshold;
    const int fmt_for_thr = (format == SPMV_FMT_AUTO) ? SPMV_FMT_SELL : format;
    if (thr < 0) thr = default_threshold(fmt_for_thr, h->dtype);
    if (prm.long_row_threshold == 0) thr = -1;  // 0 = never cut
    if (format == SPMV_FMT_HYB || format == SPMV_FMT_MERGE) thr = -1;  // no separate long-row pass
    c.threshold = thr;

    int64_t *hist_d = nullptr, *stats_d = nullptr;
    SPMV_TRY(c.temp.get(&hist_d, kHistCap + 1));
    SPMV_TRY(c.temp.get(&stats_d, 3));
    SPMV_TRY_CUDA(launch_histogram(n, c.len, thr, hist_d, stats_d, c.s));
    c.hist.assign(kHistCap + 1, 0);
    int64_t stats[3] = {0, 0, 0};
    SPMV_TRY_CUDA(cudaMemcpyAsync(c.hist.data(), hist_d, sizeof(int64_t) * (kHistCap + 1), cudaMemcpyDeviceToHost, c.s));
    SPMV_TRY_CUDA(cudaMemcpyAsync(stats, stats_d, sizeof(stats), cudaMemcpyDeviceToHost, c.s));
    SPMV_TRY(sync(c.s));
    c.n_long = stats[0];
    c.long_nnz = stats[1];
    c.max_short = static_cast<int32_t>(stats[2]);
    h->n_long_rows = c.n_long;
    h->long_nnz = c.long_nnz;

    int32_t C = prm.C > 0 ? prm.C : 32;
    if (C < 32 || C > 1024 || (C & (C - 1)))
        return set_error(SPMV_ERR_INVALID_ARG, "SELL slice height C must be a power of two in [32, 1024]");
    int64_t sigma = prm.sigma > 0 ? prm.sigma : 1;

    if (format == SPMV_FMT_AUTO) {
        // SELL-32 in natural order when that pads little (it keeps x and y accesses in
        // row order); otherwise rows sorted by length over the whole matrix (pJDS), so
        // every slice holds rows of nearly equal length.  Long rows go to the row-split
        // pass in both cases.
        int64_t slots1 = 0;
        SPMV_TRY(probe_sigma1_slots(c, &slots1));
        const int64_t stored = nnz - c.long_nnz;
        format = SPMV_FMT_SELL;
        C = 32;
        sigma = static_cast<double>(slots1) <= 1.10 * static_cast<double>(stored) + 32.0 * 64 ? 1 : std::max<int64_t>(n, 1);
    }
    h->format = format;
    h->params = prm;
    h->params.C = C;
    h->params.sigma = sigma;
    h->params.long_row_threshold = c.threshold;

    // threads per row of the sliced apply (SELL, ELLPACK-R, HYB's ELL part)
    if (format == SPMV_FMT_SELL || format == SPMV_FMT_ELL_R || format == SPMV_FMT_HYB) {
        int32_t g = prm.row_threads;
        if (g > 0 && (g > 32 || (g & (g - 1))))
            return set_error(SPMV_ERR_INVALID_ARG, "row_threads must be 1, 2, 4, 8, 16 or 32");
        if (g <= 0 && (prm.vector_loads == 1 || prm.staged == 1)) g = 1;  // vector loads, staged: one thread per row
        if (g <= 0) {
            int sms = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
                (void)cudaGetLastError();
                sms = 152;
            }
            g = auto_row_threads(n, nnz - c.long_nnz, sms);
        }
        int mode = prm.row_group_mode < 0 ? 1 : prm.row_group_mode;
        if (mode > 2) return set_error(SPMV_ERR_INVALID_ARG, "row_group_mode must be 0, 1 or 2");
        if (g == 1) mode = 0;
        if (mode == 2 && g > 8)
            return set_error(SPMV_ERR_UNSUPPORTED, "the column-grouped mode takes 2, 4 or 8 threads per row");
        c.group = g;
        c.group_mode = mode;
        c.interleaved = mode == 1;
        if (prm.vector_loads > 1) return set_error(SPMV_ERR_INVALID_ARG, "vector_loads must be 0 or 1");
        if (prm.vector_loads == 1 && g > 1)
            return set_error(SPMV_ERR_UNSUPPORTED, "vector loads take one thread per row (row_threads 1)");
        c.vec = prm.vector_loads == 1;
    }
    h->params.row_threads = c.group;
    h->params.row_group_mode = c.group_mode;
    h->params.vector_loads = c.vec ? 1 : 0;
    if (prm.host_blocks > kMaxHostBlocks)
        return set_error(SPMV_ERR_INVALID_ARG, "host_blocks must be at most " + std::to_string(kMaxHostBlocks));
    h->params.host_blocks = prm.host_blocks <= 1 ? 0 : prm.host_blocks;

    switch (format) {
        case SPMV_FMT_CSR_VECTOR: {
            int32_t g = prm.subwarp > 0 ? prm.subwarp : 0;
            if (g && g != 2 && g != 4 && g != 8 && g != 16 && g != 32)
                return set_error(SPMV_ERR_INVALID_ARG, "subwarp must be 2, 4, 8, 16 or 32");
            h->params.subwarp = g;
            SPMV_TRY(build_csr_vector(c, g));
            break;
        }
        case SPMV_FMT_ELL_R:
            h->params.C = 32;
            h->params.sigma = 1;
            SPMV_TRY(build_sell_like(c, format, 32, 1));
            break;
        case SPMV_FMT_SELL:
            SPMV_TRY(build_sell_like(c, format, C, sigma));
            break;
        case SPMV_FMT_MERGE:
            h->params.long_row_threshold = -1;
            SPMV_TRY(build_merge(c));
            break;
        case SPMV_FMT_HYB: {
            const int32_t cap = hyb_width_cap(h->dtype);
            int32_t K = prm.K >= 0 ? prm.K : hyb_auto_width(c, h->dtype, n, cap);
            // automatic: COO (measured faster than the CSR spill on the HMEp-shaped and power-law
            // matrices, 224 / 331 against 230 / 344 us; equal where every row fits the ELL part)
            const int spill_csr = prm.spill_csr >= 0 ? (prm.spill_csr ? 1 : 0) : 0;
            h->params.K = K;
            h->params.spill_csr = spill_csr;
            h->params.long_row_threshold = -1;
            SPMV_TRY(build_hyb(c, K, spill_csr));
            break;
        }
        default:
            return set_error(SPMV_ERR_INVALID_ARG, "unknown format");
    }
    if (h->sliced.present) {
        // x gathers: an L2 evict-last hint keeps x resident while the matrix streams
        // past it.  It pays when the rows are sorted (their gathers reach across all of
        // x for the whole kernel) with float64 x at most L2 / 4 and a matrix stream
        // larger than L2 (power-law 4M: 177.5 against 180.0 us).  In natural order the
        // gathers are local and plain loads are faster (3D Laplacian 128^3: 30.8 against
        // 31.2 us; small L2-resident matrices 3-7 %).
        if (prm.x_policy > 1) return set_error(SPMV_ERR_INVALID_ARG, "x_policy must be 0 or 1");
        int l2 = 0;
        if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, h->device) != cudaSuccess) {
            (void)cudaGetLastError();
            l2 = 0;
        }
        const double stream_bytes = static_cast<double>(h->sliced.slots) * (value_bytes(h->dtype) + 4);
        h->sliced.keep_x = prm.x_policy >= 0 ? prm.x_policy == 1
                                             : h->dtype == SPMV_F64 && h->sliced.perm != nullptr &&
                                                   static_cast<double>(n) * 8.0 <= 0.25 * l2 &&
                                                   stream_bytes > static_cast<double>(l2);
        h->params.x_policy = h->sliced.keep_x ? 1 : 0;
    }
    if (prm.staged > 1) return set_error(SPMV_ERR_INVALID_ARG, "staged must be 0 or 1");
    if (prm.staged == 1) {
        if (format != SPMV_FMT_SELL || !sell_staged_supported(h->sliced))
            return set_error(SPMV_ERR_UNSUPPORTED, "the bulk-staged apply takes SELL-32 with one thread per row");
        h->sliced.staged = true;
        h->kernels.assign(1, "sell_staged");  // long rows: the row-split chunks in a launch of their own
        if (h->seg.kind == 3) h->kernels.push_back("rowsplit_chunks");
    }
    h->params.staged = h->sliced.staged ? 1 : 0;
    SPMV_TRY(dev_alloc_n(h, &h->dev_err, 1));
    SPMV_TRY_CUDA(cudaMemsetAsync(h->dev_err, 0, sizeof(int), c.s));
    if (h->seg.kind == 1) h->kernels.push_back("merge_path");
    if (h->seg.kind == 2) h->kernels.push_back("coo_segmented");
    if ((h->seg.kind == 1 || h->seg.kind == 2) && h->seg.n_cta > 1) h->kernels.push_back("carry_fixup");
    if (h->seg.kind == 3 && !h->sliced.present) h->kernels.push_back("rowsplit_chunks");
    // the apply scratch of the build's stream, so applies there allocate nothing
    ApplyScratch *first = nullptr;
    SPMV_TRY(acquire_scratch(h, c.s, &first));
    return sync(c.s);
}

void free_handle(spmv_handle_t h) {
    if (!h) return;
    for (cudaEvent_t e : h->host_events) cudaEventDestroy(e);
    if (h->host_in) cudaStreamDestroy(h->host_in);
    if (h->host_out) cudaStreamDestroy(h->host_out);
    for (void *p : h->allocations) lib_free(p);
    delete h;
}

// ---------------------------------------------------------------------------
// apply
// ---------------------------------------------------------------------------
struct Recorder {
    std::vector<cudaEvent_t> ev;
    int mark(cudaStream_t s) {
        cudaEvent_t e;
        SPMV_TRY_CUDA(cudaEventCreate(&e));
        ev.push_back(e);
        SPMV_TRY_CUDA(cudaEventRecord(e, s));
        return SPMV_OK;
    }
    ~Recorder() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
    }
};

// Formats whose kernels write y exactly once per row (so alpha/beta fold into that write).
bool fused_epilogue(spmv_handle_t h) {
    // kernels whose long rows run in a launch of their own (whose chunks store plain sums)
    if (h->sliced.group > 1 || h->sliced.vec || h->sliced.staged)
        return (h->format == SPMV_FMT_SELL || h->format == SPMV_FMT_ELL_R) && h->seg.kind == 0;
    return (h->format == SPMV_FMT_SELL || h->format == SPMV_FMT_ELL_R) && (h->seg.kind == 0 || h->seg.kind == 3);
}

int enqueue(spmv_handle_t h, const void *x, void *y, cudaStream_t s, Recorder *rec, const Scale *scale = nullptr) {
    ApplyScratch *sc = nullptr;
    SPMV_TRY(acquire_scratch(h, s, &sc));
    if (scale && !fused_epilogue(h)) {
        // y = alpha * t + beta * y with t = A x computed into a scratch column of this stream
        SPMV_TRY(scratch_column(h, &sc->tmp_y));
        SPMV_TRY(enqueue(h, x, sc->tmp_y, s, rec, nullptr));
        SPMV_TRY_CUDA(launch_axpby_col(h->dtype, h->n, scale->alpha, sc->tmp_y, scale->beta, y, 1, s));
        if (rec) SPMV_TRY(rec->mark(s));
        return SPMV_OK;
    }
    if (rec) SPMV_TRY(rec->mark(s));
    const Segmented seg = with_scratch(h->seg, *sc);
    const bool split = seg.kind == 3;
    if (h->format == SPMV_FMT_CSR_VECTOR) {
        for (const Bin &b : h->bins) {
            SPMV_TRY_CUDA(launch_csr_vector(h->dtype, b.g, b.count, h->bin_rows ? h->bin_rows + b.offset : nullptr,
                                            h->row_ptr, h->csr_col, h->csr_val, x, y, s));
            if (rec) SPMV_TRY(rec->mark(s));
        }
        if (split) {
            SPMV_TRY_CUDA(launch_rowsplit(h->dtype, seg, x, y, s));
            if (rec) SPMV_TRY(rec->mark(s));
        }
    } else if (h->sliced.present && (h->sliced.group > 1 || h->sliced.vec)) {
        // G threads per row or vector loads, then the long rows' chunks
        if (h->sliced.vec)
            SPMV_TRY_CUDA(launch_sellv_apply(h->dtype, h->sliced, h->n, x, y, s, scale));
        else
            SPMV_TRY_CUDA(launch_sellg_apply(h->dtype, h->sliced, h->n, x, y, s, scale));
        if (rec) SPMV_TRY(rec->mark(s));
        if (split) {
            SPMV_TRY_CUDA(launch_rowsplit(h->dtype, seg, x, y, s));
            if (rec) SPMV_TRY(rec->mark(s));
        }
    } else if (h->sliced.present && h->sliced.staged) {
        SPMV_TRY_CUDA(launch_sell_staged(h->dtype, h->sliced, h->n, x, y, h->dev_err, s, scale));
        if (rec) SPMV_TRY(rec->mark(s));
        if (split) {
            SPMV_TRY_CUDA(launch_rowsplit(h->dtype, seg, x, y, s));
            if (rec) SPMV_TRY(rec->mark(s));
        }
    } else if (h->sliced.present) {
        // sliced rows (and, in the same launch, the chunks of the long rows)
        SPMV_TRY_CUDA(launch_sell_apply(h->dtype, h->sliced, h->n, split ? &seg : nullptr, x, y, s, scale));
        if (rec) SPMV_TRY(rec->mark(s));
    }
    if (!split && seg.kind != 0) {
        SPMV_TRY_CUDA(launch_segmented(h->dtype, seg, x, y, s));
        if (rec) SPMV_TRY(rec->mark(s));
        if (seg.n_cta > 1) {
            SPMV_TRY_CUDA(launch_carry_fixup(h->dtype, seg, y, s));
            if (rec) SPMV_TRY(rec->mark(s));
        }
    }
    return SPMV_OK;
}

// After the stream has been synchronised: report (and clear) a bounded device wait of an
// apply kernel that ran out.  Only the bulk-staged kernel waits on the device.
int check_device_flag(spmv_handle_t h) {
    if (!h->sliced.staged || !h->dev_err) return SPMV_OK;
    int v = 0;
    SPMV_TRY_CUDA(cudaMemcpy(&v, h->dev_err, sizeof(int), cudaMemcpyDeviceToHost));
    if (!v) return SPMV_OK;
    SPMV_TRY_CUDA(cudaMemset(h->dev_err, 0, sizeof(int)));
    return set_error(SPMV_ERR_TIMEOUT, "an apply kernel gave up waiting for its bulk copies (results invalid)");
}

// The vector arguments of an apply: device memory of the current device (a host or
// another device's pointer is refused before anything is enqueued).
int check_vectors(const void *a, const char *an, const void *b, const char *bn) {
    SPMV_TRY(check_device_pointer(a, an));
    return check_device_pointer(b, bn);
}

int check_current_device(spmv_handle_t h) {
    int dev = -1;
    SPMV_TRY_CUDA(cudaGetDevice(&dev));
    if (dev != h->device)
        return set_error(SPMV_ERR_INVALID_ARG, "the handle belongs to CUDA device " + std::to_string(h->device) +
                                                   " but device " + std::to_string(dev) + " is current");
    return SPMV_OK;
}

// SPMV_LOG set to anything but "" or "0": every successful build writes its plan (the
// spmv_describe JSON) to stderr, one line.
void log_plan(spmv_handle_t h) {
    const char *v = std::getenv("SPMV_LOG");
    if (!v || !*v || (v[0] == '0' && !v[1])) return;
    std::vector<char> buf(1 << 16);
    if (spmv_describe(h, buf.data(), buf.size()) != SPMV_OK) {
        buf.assign(1 << 22, 0);
        if (spmv_describe(h, buf.data(), buf.size()) != SPMV_OK) {
            clear_error();
            return;
        }
    }
    std::fprintf(stderr, "spmv: built %s\n", buf.data());
}

spmv_handle_t build_impl(int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col_idx, const void *vals,
                         int dtype, int format, const spmv_format_params *params, cudaStream_t s) {
    clear_error();
    if (n < 0 || nnz < 0 || n >= (int64_t(1) << 31) || nnz >= (int64_t(1) << 31)) {
        set_error(SPMV_ERR_INVALID_ARG, "n and nnz must lie in [0, 2^31)");
        return nullptr;
    }
    if (dtype != SPMV_F64 && dtype != SPMV_F32) {
        set_error(SPMV_ERR_INVALID_ARG, "dtype must be SPMV_F64 or SPMV_F32");
        return nullptr;
    }
    if (format < SPMV_FMT_AUTO || format > SPMV_FMT_MERGE) {
        set_error(SPMV_ERR_INVALID_ARG, "unknown format");
        return nullptr;
    }
    if (!row_ptr || (nnz > 0 && (!col_idx || !vals))) {
        set_error(SPMV_ERR_INVALID_ARG, "NULL matrix array");
        return nullptr;
    }
    if (check_device_pointer(row_ptr, "row_ptr") != SPMV_OK) return nullptr;
    if (nnz > 0 && (check_device_pointer(col_idx, "col_idx") != SPMV_OK ||
                    check_device_pointer(vals, "vals") != SPMV_OK))
        return nullptr;
    spmv_format_params prm;
    spmv_default_params(&prm);
    if (params) prm = *params;

    spmv_handle_t h = new (std::nothrow) spmv_handle_s();
    if (!h) {
        set_error(SPMV_ERR_OOM, "host allocation of the handle failed");
        return nullptr;
    }
    h->n = n;
    h->nnz = nnz;
    h->dtype = dtype;
    h->requested_format = format;
    if (cudaGetDevice(&h->device) != cudaSuccess) {
        (void)cudaGetLastError();
        set_error(SPMV_ERR_CUDA, "no CUDA device");
        delete h;
        return nullptr;
    }
    int st;
    {
        BuildCtx c{h, s, row_ptr, col_idx, vals};
        st = build_all(c, format, prm);
        if (st == SPMV_OK) st = sync(s);
    }
    if (st != SPMV_OK) {
        const int keep = g_last_error;
        const std::string msg = g_last_msg;
        cudaStreamSynchronize(s);
        free_handle(h);
        set_error(keep != SPMV_OK ? keep : st, msg);
        return nullptr;
    }
    log_plan(h);
    return h;
}

void append(std::string &out, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
void append(std::string &out, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    out += buf;
}

// ---------------------------------------------------------------------------
// spmv_apply_host pipeline
// ---------------------------------------------------------------------------
int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

bool vectors_alias(spmv_handle_t h, const void *x, const void *y) {
    const size_t bytes = static_cast<size_t>(h->n) * value_bytes(h->dtype);
    return spans_overlap(x, bytes, y, bytes);
}

bool page_locked(const void *p) {
    cudaPointerAttributes attr;
    const bool ok = cudaPointerGetAttributes(&attr, p) == cudaSuccess && attr.type == cudaMemoryTypeHost;
    (void)cudaGetLastError();
    return ok;
}

// The rows at sorted positions [p0, p1) as a sliced part of their own (one thread per
// row, column-major slots).  SELL: p0 is a multiple of C, so the view starts at slice
// p0 / C.  One-slice ELL: slot = slice start + j * ld + position, so the view moves the
// slot arrays by p0 instead.  Launched without programmatic dependent launch: its
// start waits on an event of the copy stream.
Sliced sliced_view(const Sliced &sl, int dtype, int64_t p0, int64_t p1) {
    Sliced v = sl;
    v.n_pos = p1 - p0;
    v.len = sl.len + p0;
    if (sl.perm) v.perm = sl.perm + p0;
    if (sl.log2C < 31) {
        v.slice_ptr = sl.slice_ptr + (p0 >> sl.log2C);
    } else {
        v.col = sl.col + p0;
        v.val = static_cast<char *>(sl.val) + p0 * static_cast<int64_t>(value_bytes(dtype));
    }
    v.pdl = false;
    v.has_tail = false;  // the tail table counts slices of the whole layout
    return v;
}

// Decides, on the first spmv_apply_host call of a handle, whether its calls run
// pipelined, and prepares the blocks, streams and events (host_pipe = 1), or not
// (host_pipe = -1).  Synchronises s once (the column reach goes to the host).
// Off unless host_blocks asks for it.  On a host link where every copy carries about
// 8 us of fixed latency and each direction drops to about 154 GB/s while the other is
// busy, the pipeline can hide little more than the product's own time.
int host_pipe_setup(spmv_handle_t h, cudaStream_t s) {
    h->host_pipe = -1;
    const Sliced &sl = h->sliced;
    const int req = h->params.host_blocks;
    if (req <= 0 || h->n == 0) return SPMV_OK;
    if (!sl.present || !fused_epilogue(h) || h->seg.kind != 0 || sl.group != 1 || sl.vec || sl.interleaved)
        return SPMV_OK;
    // blocks are whole slices (whole warps for ELL) and, when rows are sorted, whole
    // sort windows, so a block's rows are exactly the rows [p0, p1)
    int64_t unit = sl.log2C < 31 ? sl.C : 32;
    if (sl.perm) {  // sorted within windows of min(sigma, n) rows starting at row 0
        const int64_t w = std::min<int64_t>(sl.sigma, h->n);
        if (w <= 0 || w >= h->n) return SPMV_OK;
        unit = unit / gcd64(unit, w) * w;
        if (unit >= sl.n_pos) return SPMV_OK;
    }
    const int64_t block = ceil_div(ceil_div(sl.n_pos, req), unit) * unit;
    const int64_t nb = ceil_div(sl.n_pos, block);
    if (nb < 2) return SPMV_OK;

    void *d_max = nullptr;
    {
        std::lock_guard<std::mutex> lock(h->scratch_mutex);  // guards h->allocations
        SPMV_TRY(dev_alloc(h, &d_max, static_cast<size_t>(nb) * sizeof(int32_t)));
    }
    SPMV_TRY_CUDA(cudaMemsetAsync(d_max, 0xff, static_cast<size_t>(nb) * sizeof(int32_t), s));
    SPMV_TRY_CUDA(launch_block_max_col(sl, block, static_cast<int32_t *>(d_max), s));
    std::vector<int32_t> reach(static_cast<size_t>(nb));
    SPMV_TRY_CUDA(cudaMemcpyAsync(reach.data(), d_max, reach.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    std::vector<int32_t> need(reach.size());
    for (size_t b = 0; b < reach.size(); ++b)  // pieces of x share the blocks' boundaries
        need[b] = reach[b] < 0 ? -1 : static_cast<int32_t>(reach[b] / block);

    if (!h->host_in) SPMV_TRY_CUDA(cudaStreamCreateWithFlags(&h->host_in, cudaStreamNonBlocking));
    if (!h->host_out) SPMV_TRY_CUDA(cudaStreamCreateWithFlags(&h->host_out, cudaStreamNonBlocking));
    while (h->host_events.size() < static_cast<size_t>(2 * nb + 3)) {
        cudaEvent_t e;
        SPMV_TRY_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        h->host_events.push_back(e);
    }
    h->host_block = block;
    h->host_need = std::move(need);
    h->host_pipe = 1;
    return SPMV_OK;
}

// One pipelined spmv_apply_host: x in by pieces on host_in, block b on s once piece
// need[b] is in (pieces arrive in order), its rows of y out on host_out; s waits for
// both copy streams and is synchronised.  Events: [0, nb) pieces of x in, [nb, 2 nb)
// blocks done, 2 nb start, 2 nb + 1 all of x in, 2 nb + 2 all of y out.  (Blocks that
// store y straight into the page-locked y_host instead measured slower: those stores
// overlap the incoming copies less than a second copy engine does.)
int apply_host_pipelined(spmv_handle_t h, const ApplyScratch &sc, const void *x_host, void *y_host, cudaStream_t s) {
    const Sliced &sl = h->sliced;
    const int64_t vb = static_cast<int64_t>(value_bytes(h->dtype));
    const int64_t n = h->n, block = h->host_block;
    const int64_t nb = static_cast<int64_t>(h->host_need.size());
    cudaEvent_t *ev = h->host_events.data();
    const char *xh = static_cast<const char *>(x_host);
    char *yh = static_cast<char *>(y_host);
    char *xs = static_cast<char *>(sc.x_stage);
    char *ys = static_cast<char *>(sc.y_stage);
    SPMV_TRY_CUDA(cudaEventRecord(ev[2 * nb], s));
    SPMV_TRY_CUDA(cudaStreamWaitEvent(h->host_in, ev[2 * nb], 0));
    SPMV_TRY_CUDA(cudaStreamWaitEvent(h->host_out, ev[2 * nb], 0));
    for (int64_t c = 0; c < nb; ++c) {
        const int64_t r0 = c * block, r1 = std::min(n, r0 + block);
        if (r1 > r0)
            SPMV_TRY_CUDA(cudaMemcpyAsync(xs + r0 * vb, xh + r0 * vb, static_cast<size_t>((r1 - r0) * vb),
                                          cudaMemcpyHostToDevice, h->host_in));
        SPMV_TRY_CUDA(cudaEventRecord(ev[c], h->host_in));
    }
    SPMV_TRY_CUDA(cudaEventRecord(ev[2 * nb + 1], h->host_in));
    for (int64_t b = 0; b < nb; ++b) {
        const int64_t p0 = b * block, p1 = std::min(sl.n_pos, p0 + block);
        const int32_t need = h->host_need[static_cast<size_t>(b)];
        if (need >= 0) SPMV_TRY_CUDA(cudaStreamWaitEvent(s, ev[need], 0));
        const Sliced v = sliced_view(sl, h->dtype, p0, p1);
        // natural order: the view's position p is row p0 + p; sorted: perm gives the row
        if (sl.perm)
            SPMV_TRY_CUDA(launch_sell_apply(h->dtype, v, n, nullptr, xs, ys, s, nullptr));
        else
            SPMV_TRY_CUDA(launch_sell_apply(h->dtype, v, n - p0, nullptr, xs, ys + p0 * vb, s, nullptr));
        SPMV_TRY_CUDA(cudaEventRecord(ev[nb + b], s));
        SPMV_TRY_CUDA(cudaStreamWaitEvent(h->host_out, ev[nb + b], 0));
        const int64_t r1 = std::min(n, p1);
        if (r1 > p0)
            SPMV_TRY_CUDA(cudaMemcpyAsync(yh + p0 * vb, ys + p0 * vb, static_cast<size_t>((r1 - p0) * vb),
                                          cudaMemcpyDeviceToHost, h->host_out));
    }
    SPMV_TRY_CUDA(cudaEventRecord(ev[2 * nb + 2], h->host_out));
    SPMV_TRY_CUDA(cudaStreamWaitEvent(s, ev[2 * nb + 1], 0));
    SPMV_TRY_CUDA(cudaStreamWaitEvent(s, ev[2 * nb + 2], 0));
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    return SPMV_OK;
}

}  // namespace
}  // namespace spmv

using namespace spmv;

extern "C" {

int spmv_device_memory(int64_t *allocations, int64_t *bytes) {
    memory_held(allocations, bytes);
    return SPMV_OK;
}

int spmv_default_params(spmv_format_params *p) {
    if (!p) return set_error(SPMV_ERR_INVALID_ARG, "NULL params");
    p->C = -1;
    p->sigma = -1;
    p->K = -1;
    p->spill_csr = -1;
    p->long_row_threshold = -1;
    p->subwarp = -1;
    p->row_threads = -1;
    p->row_group_mode = -1;
    p->x_policy = -1;
    p->vector_loads = -1;
    p->host_blocks = -1;
    p->staged = -1;
    return SPMV_OK;
}

spmv_handle_t spmv_build_from_csr(int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col_idx,
                                  const void *vals, int dtype, int format) {
    return build_impl(n, nnz, row_ptr, col_idx, vals, dtype, format, nullptr, nullptr);
}

spmv_handle_t spmv_build_from_csr_ex(int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col_idx,
                                     const void *vals, int dtype, int format, const spmv_format_params *params,
                                     void *stream) {
    return build_impl(n, nnz, row_ptr, col_idx, vals, dtype, format, params, static_cast<cudaStream_t>(stream));
}

spmv_handle_t spmv_build_permuted(int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col_idx,
                                  const void *vals, int dtype, int format, const spmv_format_params *params,
                                  int ordering, const int32_t *perm, void *stream) {
    clear_error();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto fail = [](int status, const std::string &msg) -> spmv_handle_t {
        set_error(status, msg);
        return nullptr;
    };
    if (n < 0 || nnz < 0 || n >= (int64_t(1) << 31) || nnz >= (int64_t(1) << 31))
        return fail(SPMV_ERR_INVALID_ARG, "n and nnz must lie in [0, 2^31)");
    if (dtype != SPMV_F64 && dtype != SPMV_F32) return fail(SPMV_ERR_INVALID_ARG, "dtype must be SPMV_F64 or SPMV_F32");
    if (ordering < SPMV_ORDER_NATURAL || ordering > SPMV_ORDER_USER) return fail(SPMV_ERR_INVALID_ARG, "unknown ordering");
    if (!row_ptr || (nnz > 0 && (!col_idx || !vals))) return fail(SPMV_ERR_INVALID_ARG, "NULL matrix array");
    if (ordering == SPMV_ORDER_USER && n > 0 && !perm) return fail(SPMV_ERR_INVALID_ARG, "ordering USER needs perm");
    if (check_device_pointer(row_ptr, "row_ptr") != SPMV_OK) return nullptr;
    if (nnz > 0 && (check_device_pointer(col_idx, "col_idx") != SPMV_OK ||
                    check_device_pointer(vals, "vals") != SPMV_OK))
        return nullptr;
    if (ordering == SPMV_ORDER_USER && n > 0 && check_device_pointer(perm, "perm") != SPMV_OK) return nullptr;
    const size_t vb = value_bytes(dtype);
    Temp temp;
    int32_t *len = nullptr, *status = nullptr, *order = nullptr, *b_ptr = nullptr, *b_col = nullptr;
    void *b_val = nullptr;
    if (temp.get(&len, n) || temp.get(&status, 3) || temp.get(&order, n) || temp.get(&b_ptr, n + 1) ||
        temp.get(&b_col, nnz) || temp.get(reinterpret_cast<char **>(&b_val), nnz * static_cast<int64_t>(vb)))
        return nullptr;
    // A must be valid before any ordering kernel indexes through it
    int32_t st[3] = {0, 0, 0};
    if (cudaMemsetAsync(status, 0, sizeof(st), s) != cudaSuccess ||
        launch_validate(n, nnz, row_ptr, col_idx, len, status, s) != cudaSuccess ||
        cudaMemcpyAsync(st, status, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        set_cuda_error(cudaGetLastError(), "validating the CSR");
        return nullptr;
    }
    if (st[0]) return fail(SPMV_ERR_BAD_CSR, "row_ptr is not a valid CSR row pointer");
    if (st[1]) return fail(SPMV_ERR_BAD_CSR, "a column index lies outside [0, n)");
    if (compute_ordering(ordering, n, nnz, row_ptr, col_idx, st[2], perm, order, s) != SPMV_OK) return nullptr;
    if (permute_csr(dtype, n, nnz, row_ptr, col_idx, vals, order, b_ptr, b_col, b_val, s) != SPMV_OK) return nullptr;
    spmv_handle_t h = build_impl(n, nnz, b_ptr, b_col, b_val, dtype, format, params, s);
    if (!h) return nullptr;
    h->ordering = ordering;
    if (n > 0) {
        if (dev_alloc_n(h, &h->basis_perm, n) != SPMV_OK ||
            cudaMemcpyAsync(h->basis_perm, order, sizeof(int32_t) * n, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess) {
            if (spmv_last_error() == SPMV_OK) set_cuda_error(cudaGetLastError(), "storing the permutation");
            free_handle(h);
            return nullptr;
        }
    }
    return h;
}

int spmv_get_permutation(spmv_handle_t h, int32_t *perm, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (h->n == 0) return SPMV_OK;
    if (!perm) return set_error(SPMV_ERR_INVALID_ARG, "NULL perm");
    SPMV_TRY(check_current_device(h));
    SPMV_TRY(check_device_pointer(perm, "perm"));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (h->basis_perm) {
        SPMV_TRY_CUDA(cudaMemcpyAsync(perm, h->basis_perm, sizeof(int32_t) * h->n, cudaMemcpyDeviceToDevice, s));
    } else {
        std::vector<int32_t> iota(static_cast<size_t>(h->n));
        for (int64_t i = 0; i < h->n; ++i) iota[i] = static_cast<int32_t>(i);
        SPMV_TRY_CUDA(cudaMemcpyAsync(perm, iota.data(), sizeof(int32_t) * h->n, cudaMemcpyHostToDevice, s));
    }
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    return SPMV_OK;
}

int spmv_permute_vector(spmv_handle_t h, const void *src, void *dst, int direction, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (direction != 0 && direction != 1) return set_error(SPMV_ERR_INVALID_ARG, "direction must be 0 or 1");
    if (h->n == 0) return SPMV_OK;
    if (!src || !dst) return set_error(SPMV_ERR_INVALID_ARG, "NULL src or dst");
    if (vectors_alias(h, src, dst)) return set_error(SPMV_ERR_INVALID_ARG, "src and dst must not overlap");
    SPMV_TRY(check_current_device(h));
    SPMV_TRY(check_vectors(src, "src", dst, "dst"));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!h->basis_perm) {
        SPMV_TRY_CUDA(cudaMemcpyAsync(dst, src, value_bytes(h->dtype) * h->n, cudaMemcpyDeviceToDevice, s));
        return SPMV_OK;
    }
    SPMV_TRY_CUDA(launch_permute_vector(h->dtype, h->n, h->basis_perm, src, dst, direction, s));
    return SPMV_OK;
}

int spmv_apply(spmv_handle_t h, const void *x, void *y, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (h->n == 0) return SPMV_OK;
    if (!x || !y) return set_error(SPMV_ERR_INVALID_ARG, "NULL x or y");
    if (vectors_alias(h, x, y)) return set_error(SPMV_ERR_INVALID_ARG, "x and y overlap");
    SPMV_TRY(check_current_device(h));
    SPMV_TRY(check_vectors(x, "x", y, "y"));
    return enqueue(h, x, y, static_cast<cudaStream_t>(stream), nullptr);
}

int spmv_apply_host(spmv_handle_t h, const void *x_host, void *y_host, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (h->n == 0) return SPMV_OK;
    if (!x_host || !y_host) return set_error(SPMV_ERR_INVALID_ARG, "NULL x or y");
    SPMV_TRY(check_current_device(h));
    const size_t bytes = static_cast<size_t>(h->n) * value_bytes(h->dtype);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ApplyScratch *sc = nullptr;
    SPMV_TRY(acquire_scratch(h, s, &sc));
    SPMV_TRY(scratch_column(h, &sc->x_stage));
    {
        // the pipeline's copy streams and events belong to the handle: one call at a time
        std::unique_lock<std::mutex> pipe(h->host_mutex);
        if (h->host_pipe == 0) SPMV_TRY(host_pipe_setup(h, s));
        // in place (x_host and y_host overlapping): unpipelined, where all of x is in before y moves
        if (h->host_pipe == 1 && page_locked(x_host) && page_locked(y_host) && !vectors_alias(h, x_host, y_host)) {
            SPMV_TRY(scratch_column(h, &sc->y_stage));
            h->host_last_blocks = static_cast<int>(h->host_need.size());
            return apply_host_pipelined(h, *sc, x_host, y_host, s);
        }
    }
    h->host_last_blocks = 0;
    SPMV_TRY_CUDA(cudaMemcpyAsync(sc->x_stage, x_host, bytes, cudaMemcpyHostToDevice, s));
    // A plan that writes every row of y exactly once (one sliced launch, no accumulating
    // pass) stores y straight into page-locked host memory: the transfer back then runs
    // inside the product instead of after it.
    void *y_direct = nullptr;
    if (fused_epilogue(h)) {
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, y_host) == cudaSuccess && attr.type == cudaMemoryTypeHost)
            y_direct = attr.devicePointer;
        (void)cudaGetLastError();
    }
    if (y_direct) {
        SPMV_TRY(enqueue(h, sc->x_stage, y_direct, s, nullptr));
    } else {
        SPMV_TRY(scratch_column(h, &sc->y_stage));
        SPMV_TRY(enqueue(h, sc->x_stage, sc->y_stage, s, nullptr));
        SPMV_TRY_CUDA(cudaMemcpyAsync(y_host, sc->y_stage, bytes, cudaMemcpyDeviceToHost, s));
    }
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    return check_device_flag(h);
}

// Device address of page-locked host memory (cudaHostAlloc / cudaHostRegister), or an error.
int mapped_pointer(const void *host, const char *name, void **dev) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, host);
    if (e != cudaSuccess || attr.type != cudaMemoryTypeHost || !attr.devicePointer) {
        (void)cudaGetLastError();
        return set_error(SPMV_ERR_INVALID_ARG, std::string(name) + " is not page-locked host memory");
    }
    *dev = attr.devicePointer;
    return SPMV_OK;
}

int spmv_apply_mapped(spmv_handle_t h, const void *x_host, void *y_host, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (h->n == 0) return SPMV_OK;
    if (!x_host || !y_host) return set_error(SPMV_ERR_INVALID_ARG, "NULL x or y");
    SPMV_TRY(check_current_device(h));
    void *xd = nullptr, *yd = nullptr;
    if (vectors_alias(h, x_host, y_host)) return set_error(SPMV_ERR_INVALID_ARG, "x_host and y_host overlap");
    SPMV_TRY(mapped_pointer(x_host, "x_host", &xd));
    SPMV_TRY(mapped_pointer(y_host, "y_host", &yd));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    SPMV_TRY(enqueue(h, xd, yd, s, nullptr));
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    return check_device_flag(h);
}

int spmv_apply_profiled(spmv_handle_t h, const void *x, void *y, void *stream, float *kernel_ms, int cap) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (h->n == 0) return 0;
    if (!x || !y) return set_error(SPMV_ERR_INVALID_ARG, "NULL x or y");
    if (vectors_alias(h, x, y)) return set_error(SPMV_ERR_INVALID_ARG, "x and y overlap");
    SPMV_TRY(check_current_device(h));
    SPMV_TRY(check_vectors(x, "x", y, "y"));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Recorder rec;
    SPMV_TRY(enqueue(h, x, y, s, &rec));
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    SPMV_TRY(check_device_flag(h));
    const int k = static_cast<int>(rec.ev.size()) - 1;
    for (int i = 0; i < k && i < cap; ++i) {
        float ms = 0.f;
        SPMV_TRY_CUDA(cudaEventElapsedTime(&ms, rec.ev[i], rec.ev[i + 1]));
        if (kernel_ms) kernel_ms[i] = ms;
    }
    return k;
}

int spmv_apply_ex(spmv_handle_t h, double alpha, const void *x, double beta, void *y, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (h->n == 0) return SPMV_OK;
    if (!x || !y) return set_error(SPMV_ERR_INVALID_ARG, "NULL x or y");
    if (vectors_alias(h, x, y)) return set_error(SPMV_ERR_INVALID_ARG, "x and y overlap");
    SPMV_TRY(check_current_device(h));
    SPMV_TRY(check_vectors(x, "x", y, "y"));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (alpha == 1.0 && beta == 0.0) return enqueue(h, x, y, s, nullptr);
    const Scale scale{alpha, beta};
    return enqueue(h, x, y, s, nullptr, &scale);
}

int spmv_apply_multi(spmv_handle_t h, int64_t k, double alpha, const void *X, int64_t ldx, double beta, void *Y,
                     int64_t ldy, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (k < 0 || ldx < k || ldy < k) return set_error(SPMV_ERR_INVALID_ARG, "need 0 <= k <= ldx and k <= ldy");
    if (h->n == 0 || k == 0) return SPMV_OK;
    if (!X || !Y) return set_error(SPMV_ERR_INVALID_ARG, "NULL X or Y");
    {
        const size_t vb0 = value_bytes(h->dtype);
        const size_t xspan = static_cast<size_t>((h->n - 1) * ldx + k) * vb0;
        const size_t yspan = static_cast<size_t>((h->n - 1) * ldy + k) * vb0;
        if (spans_overlap(X, xspan, Y, yspan)) return set_error(SPMV_ERR_INVALID_ARG, "X and Y overlap");
    }
    SPMV_TRY(check_current_device(h));
    SPMV_TRY(check_vectors(X, "X", Y, "Y"));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (k == 1 && ldx == 1 && ldy == 1) return spmv_apply_ex(h, alpha, X, beta, Y, stream);  // contiguous vectors
    const size_t vb = value_bytes(h->dtype);
    const Scale scale{alpha, beta};
    const bool fused = fused_epilogue(h) && sell_multi_supported(h->sliced);
    ApplyScratch *sc = nullptr;
    SPMV_TRY(acquire_scratch(h, s, &sc));
    const Segmented seg = with_scratch(h->seg, *sc);
    const Segmented *split = seg.kind == 3 ? &seg : nullptr;
    int64_t c = 0;
    while (c < k) {
        const char *xc = static_cast<const char *>(X) + c * vb;
        char *yc = static_cast<char *>(Y) + c * vb;
        int nv = 0;
        if (fused) {
            for (int cand : {8, 4, 2}) {
                const size_t align = std::min<size_t>(16, cand * vb);
                if (k - c >= cand && reinterpret_cast<uintptr_t>(xc) % align == 0 && (ldx * vb) % align == 0) {
                    nv = cand;
                    break;
                }
            }
        }
        if (nv) {
            SPMV_TRY_CUDA(launch_sell_multi(h->dtype, nv, h->sliced, h->n, split, xc, ldx, yc, ldy, s, scale));
            c += nv;
        } else {
            // one column through the single-vector path
            SPMV_TRY(scratch_column(h, &sc->tmp_x));
            SPMV_TRY(scratch_column(h, &sc->tmp_y));
            SPMV_TRY_CUDA(launch_gather_col(h->dtype, h->n, xc, ldx, sc->tmp_x, s));
            SPMV_TRY(enqueue(h, sc->tmp_x, sc->tmp_y, s, nullptr));
            SPMV_TRY_CUDA(launch_axpby_col(h->dtype, h->n, alpha, sc->tmp_y, beta, yc, ldy, s));
            c += 1;
        }
    }
    return SPMV_OK;
}

int spmv_device_status(spmv_handle_t h, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    SPMV_TRY(check_current_device(h));
    SPMV_TRY_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    return check_device_flag(h);
}

void spmv_destroy(spmv_handle_t h) { free_handle(h); }

int spmv_last_error(void) { return g_last_error; }
const char *spmv_last_error_message(void) { return g_last_msg; }

const char *spmv_error_string(int status) {
    switch (status) {
        case SPMV_OK: return "success";
        case SPMV_ERR_INVALID_ARG: return "invalid argument";
        case SPMV_ERR_BAD_CSR: return "malformed CSR matrix";
        case SPMV_ERR_CUDA: return "CUDA runtime error";
        case SPMV_ERR_OOM: return "out of device memory";
        case SPMV_ERR_TOO_LARGE: return "layout too large";
        case SPMV_ERR_UNSUPPORTED: return "unsupported parameter combination";
        case SPMV_ERR_TIMEOUT: return "device wait timed out";
        default: return "unknown status";
    }
}

int spmv_to_csr(spmv_handle_t h, int32_t *row_ptr, int32_t *col_idx, void *vals, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (!row_ptr || (h->nnz > 0 && (!col_idx || !vals))) return set_error(SPMV_ERR_INVALID_ARG, "NULL output array");
    SPMV_TRY(check_current_device(h));
    SPMV_TRY(check_device_pointer(row_ptr, "row_ptr"));
    if (h->nnz > 0) {
        SPMV_TRY(check_device_pointer(col_idx, "col_idx"));
        SPMV_TRY(check_device_pointer(vals, "vals"));
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t vb = value_bytes(h->dtype);
    SPMV_TRY_CUDA(cudaMemcpyAsync(row_ptr, h->row_ptr, sizeof(int32_t) * (h->n + 1), cudaMemcpyDeviceToDevice, s));
    if (h->format == SPMV_FMT_CSR_VECTOR || h->format == SPMV_FMT_MERGE) {
        if (h->nnz > 0) {
            SPMV_TRY_CUDA(cudaMemcpyAsync(col_idx, h->csr_col, sizeof(int32_t) * h->nnz, cudaMemcpyDeviceToDevice, s));
            SPMV_TRY_CUDA(cudaMemcpyAsync(vals, h->csr_val, vb * h->nnz, cudaMemcpyDeviceToDevice, s));
        }
    } else {
        SPMV_TRY_CUDA(launch_sliced_to_csr(h->dtype, h->n, h->sliced, h->row_ptr, col_idx, vals, s));
        SPMV_TRY_CUDA(launch_segment_to_csr(h->dtype, h->seg, h->row_ptr, col_idx, vals, s));
    }
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    return SPMV_OK;
}

int spmv_get_layout(spmv_handle_t h, int32_t *perm, int64_t *slice_ptr, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (!h->sliced.present) return set_error(SPMV_ERR_UNSUPPORTED, "the handle has no sliced part");
    SPMV_TRY(check_current_device(h));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (perm && h->n > 0) {
        SPMV_TRY(check_device_pointer(perm, "perm"));
        if (h->sliced.perm) {
            SPMV_TRY_CUDA(cudaMemcpyAsync(perm, h->sliced.perm, sizeof(int32_t) * h->n, cudaMemcpyDeviceToDevice, s));
        } else {
            std::vector<int32_t> iota(static_cast<size_t>(h->n));
            for (int64_t i = 0; i < h->n; ++i) iota[i] = static_cast<int32_t>(i);
            SPMV_TRY_CUDA(cudaMemcpyAsync(perm, iota.data(), sizeof(int32_t) * h->n, cudaMemcpyHostToDevice, s));
            SPMV_TRY_CUDA(cudaStreamSynchronize(s));
        }
    }
    if (slice_ptr) {
        SPMV_TRY(check_device_pointer(slice_ptr, "slice_ptr"));
        SPMV_TRY_CUDA(cudaMemcpyAsync(slice_ptr, h->sliced.slice_ptr, sizeof(int64_t) * (h->sliced.n_slices + 1),
                                      cudaMemcpyDeviceToDevice, s));
    }
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    return SPMV_OK;
}

int spmv_get_slots(spmv_handle_t h, int32_t *col, void *val, void *stream) {
    if (!h) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle");
    if (!h->sliced.present) return set_error(SPMV_ERR_UNSUPPORTED, "the handle has no sliced part");
    SPMV_TRY(check_current_device(h));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t slots = h->sliced.slots;
    if (col && slots > 0) {
        SPMV_TRY(check_device_pointer(col, "col"));
        SPMV_TRY_CUDA(cudaMemcpyAsync(col, h->sliced.col, sizeof(int32_t) * slots, cudaMemcpyDeviceToDevice, s));
    }
    if (val && slots > 0) {
        SPMV_TRY(check_device_pointer(val, "val"));
        SPMV_TRY_CUDA(cudaMemcpyAsync(val, h->sliced.val, value_bytes(h->dtype) * slots, cudaMemcpyDeviceToDevice, s));
    }
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    return SPMV_OK;
}

int spmv_describe(spmv_handle_t h, char *json, size_t cap) {
    if (!h || !json || cap == 0) return set_error(SPMV_ERR_INVALID_ARG, "NULL handle or buffer");
    const int64_t vb = static_cast<int64_t>(value_bytes(h->dtype));
    const Sliced &sl = h->sliced;
    const Segmented &sg = h->seg;
    std::string o = "{";
    append(o, "\"format\":\"%s\",\"requested_format\":\"%s\",\"dtype\":\"%s\",", format_name(h->format),
           format_name(h->requested_format), h->dtype == SPMV_F64 ? "f64" : "f32");
    append(o, "\"n\":%lld,\"nnz\":%lld,\"max_len\":%d,\"mean_len\":%.6f,", (long long)h->n, (long long)h->nnz,
           h->max_len, h->mean_len);
    append(o, "\"C\":%d,\"sigma\":%lld,\"K\":%d,\"spill_csr\":%d,\"long_row_threshold\":%d,\"subwarp\":%d,",
           h->params.C, (long long)h->params.sigma, h->params.K, h->params.spill_csr, h->params.long_row_threshold,
           h->params.subwarp);
    append(o, "\"row_threads\":%d,\"row_group_mode\":%d,\"vector_loads\":%d,", h->params.row_threads,
           h->params.row_group_mode, h->params.vector_loads);
    append(o, "\"sliced\":%s,\"n_slices\":%lld,\"slots\":%lld,\"padded_entries\":%lld,\"stored_entries\":%lld,"
              "\"ld\":%lld,\"max_width\":%d,\"permuted\":%s,",
           sl.present ? "true" : "false", (long long)sl.n_slices, (long long)sl.slots, (long long)sl.padded_entries,
           (long long)sl.stored_entries, (long long)sl.ld, sl.max_width, sl.perm ? "true" : "false");
    append(o, "\"x_evict_last\":%s,\"staged\":%s,", sl.keep_x ? "true" : "false", sl.staged ? "true" : "false");
    // positions of the narrow tail of a globally sorted layout, several rows per thread
    append(o, "\"tail_positions\":%lld,", (long long)sell_tail_positions(sl));
    // host_blocks: the parameter (0 = off); host_pipeline_blocks: blocks of the last
    // spmv_apply_host call (0 = unpipelined, -1 = no call yet)
    append(o, "\"host_blocks\":%d,\"host_pipeline_blocks\":%d,", h->params.host_blocks, h->host_last_blocks.load());
    // once pipelined: rows per block, and for each block the last piece of x it waits for
    if (h->host_pipe == 1) {
        append(o, "\"host_pipeline_block_rows\":%lld,\"host_pipeline_reach\":[", (long long)h->host_block);
        for (size_t b = 0; b < h->host_need.size(); ++b) append(o, b ? ",%d" : "%d", h->host_need[b]);
        o += "],";
    }
    append(o, "\"ordering\":\"%s\",\"permuted_basis\":%s,", ordering_name(h->ordering),
           h->basis_perm ? "true" : "false");
    append(o, "\"n_long_rows\":%lld,\"long_nnz\":%lld,", (long long)h->n_long_rows, (long long)h->long_nnz);
    append(o, "\"segment\":\"%s\",\"segment_rows\":%lld,\"segment_nnz\":%lld,\"segment_ctas\":%lld,",
           sg.kind == 0 ? "none" : sg.kind == 1 ? "csr_merge_path" : sg.kind == 2 ? "coo" : "row_split",
           (long long)sg.n_rows, (long long)sg.nnz, (long long)(sg.kind == 3 ? sg.n_chunks : sg.n_cta));
    append(o, "\"split_chunk\":%d,", sg.kind == 3 ? sg.chunk : 0);
    o += "\"bins\":[";
    for (size_t i = 0; i < h->bins.size(); ++i)
        append(o, "%s[%d,%lld]", i ? "," : "", h->bins[i].g, (long long)h->bins[i].count);
    o += "],\"kernels\":[";
    for (size_t i = 0; i < h->kernels.size(); ++i) append(o, "%s\"%s\"", i ? "," : "", h->kernels[i].c_str());
    o += "],";
    // bytes one apply streams from the format (x counted once, y written once)
    int64_t matrix_bytes = 0;
    if (h->format == SPMV_FMT_CSR_VECTOR) {
        int64_t rows_binned = 0;
        for (const Bin &b : h->bins) rows_binned += b.count;
        matrix_bytes += (h->nnz - h->long_nnz) * (vb + 4) + rows_binned * 8 + (h->bin_rows ? rows_binned * 4 : 0);
    } else if (sl.present) {
        matrix_bytes += sl.stored_entries * (vb + 4) + sl.n_pos * 4 + (sl.perm ? sl.n_pos * 4 : 0) + sl.n_slices * 8;
    }
    if (sg.kind == 1) matrix_bytes += sg.nnz * (vb + 4) + sg.n_rows * (sg.rows ? 8 : 4) + sg.n_cta * 16;
    if (sg.kind == 2) matrix_bytes += sg.nnz * (vb + 8) + sg.n_cta * 12;
    if (sg.kind == 3) matrix_bytes += sg.nnz * (vb + 4) + sg.n_rows * 8 + sg.n_chunks * 16;
    append(o, "\"format_bytes\":%lld,\"vector_bytes\":%lld}", (long long)matrix_bytes, (long long)(2 * h->n * vb));
    std::snprintf(json, cap, "%s", o.c_str());
    if (o.size() + 1 > cap) return set_error(SPMV_ERR_INVALID_ARG, "describe buffer too small");
    return SPMV_OK;
}

}  // extern "C"
