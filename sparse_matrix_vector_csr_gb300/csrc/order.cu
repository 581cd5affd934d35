// Symmetric orderings for the permuted basis B = P A P^T, computed on the device.
//
// The GPGPU spMVM paper (pJDS section) runs the product in a permuted basis and notes
// that a Krylov solver needs the permutation only before and after the iteration; it
// also notes that sorting rows can destroy structure and with it the reuse of the
// right-hand side.  The orderings here:
//   * row length: rows by length, longest first, ties in index order (one stable
//     radix sort) -- the pJDS order over the whole matrix;
//   * reverse Cuthill-McKee on the graph of A + A^T -- the bandwidth-reducing order
//     that brings entries back next to the diagonal, so x is gathered from a narrow,
//     cache-resident window.
//
// Cuthill-McKee, defined as the queue algorithm (vertices of degree 0 first in index
// order; each component started at its unvisited vertex of least (degree, index); the
// unvisited neighbours of each dequeued vertex appended by (degree, index)), is built
// here one breadth-first level at a time: every unvisited neighbour of the current
// level is claimed by its earliest-placed neighbour there (atomicMin of the position),
// and the next level is the claimed vertices sorted by (claiming position, rank of
// (degree, index)).  The two give the same order: a vertex is appended by the first
// dequeued vertex that sees it, and vertices appended by one parent come in (degree,
// index) order.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <vector>

#include "spmv_internal.cuh"

namespace spmv {
namespace {

constexpr int kThreads = 256;
constexpr int kSmallSort = 2048;  // level sizes sorted inside one block

__device__ __forceinline__ int64_t gtid() { return static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; }
__device__ __forceinline__ int64_t gstride() { return static_cast<int64_t>(gridDim.x) * blockDim.x; }

unsigned grid(int64_t work, int64_t cap = 65536) {
    int64_t g = ceil_div(std::max<int64_t>(work, 1), kThreads);
    return static_cast<unsigned>(std::min<int64_t>(g, cap));
}

int bits(uint64_t v) {
    int b = 0;
    while (v) {
        ++b;
        v >>= 1;
    }
    return b;
}

// Stream-ordered device scratch, released when the ordering is done.
struct Scratch {
    cudaStream_t s;
    std::vector<void *> ptrs;
    explicit Scratch(cudaStream_t st) : s(st) {}
    ~Scratch() {
        for (void *p : ptrs) lib_free_async(p, s);
    }
    template <class T>
    int get(T **p, int64_t count) {
        void *q = nullptr;
        cudaError_t e = lib_malloc_async(&q, static_cast<size_t>(std::max<int64_t>(count, 1)) * sizeof(T), s);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaMallocAsync (ordering scratch)");
        ptrs.push_back(q);
        *p = static_cast<T *>(q);
        return SPMV_OK;
    }
};

// ---------------------------------------------------------------------------
// kernels
// ---------------------------------------------------------------------------
__global__ void k_iota(int64_t n, int32_t *__restrict__ v) {
    for (int64_t i = gtid(); i < n; i += gstride()) v[i] = static_cast<int32_t>(i);
}

// Both directions of every entry off the diagonal; diagonal entries get the row key n,
// which sorts after every real vertex and is dropped.  One warp per row.
__global__ void k_sym_edges(int64_t n, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col,
                            uint32_t *__restrict__ u, int32_t *__restrict__ v) {
    const int lane = threadIdx.x & 31;
    for (int64_t r = gtid() >> 5; r < n; r += gstride() >> 5) {
        const int64_t b = row_ptr[r], e = row_ptr[r + 1];
        for (int64_t k = b + lane; k < e; k += 32) {
            const int32_t c = col[k];
            const bool off = c != r;
            u[2 * k] = off ? static_cast<uint32_t>(r) : static_cast<uint32_t>(n);
            v[2 * k] = off ? c : 0;
            u[2 * k + 1] = off ? static_cast<uint32_t>(c) : static_cast<uint32_t>(n);
            v[2 * k + 1] = off ? static_cast<int32_t>(r) : 0;
        }
    }
}

// first of each distinct (u, v) with u < n
__global__ void k_mark_edges(int64_t m, int64_t n, const uint32_t *__restrict__ u, const int32_t *__restrict__ v,
                             int64_t *__restrict__ flag, unsigned long long *__restrict__ deg) {
    for (int64_t i = gtid(); i < m; i += gstride()) {
        const bool keep = u[i] < n && (i == 0 || u[i] != u[i - 1] || v[i] != v[i - 1]);
        flag[i] = keep ? 1 : 0;
        if (keep) atomicAdd(deg + u[i], 1ull);
    }
}

__global__ void k_compact_edges(int64_t m, const int64_t *__restrict__ flag, const int64_t *__restrict__ pos,
                                const int32_t *__restrict__ v, int32_t *__restrict__ adj) {
    for (int64_t i = gtid(); i < m; i += gstride())
        if (flag[i]) adj[pos[i]] = v[i];
}

__global__ void k_deg_keys(int64_t n, const unsigned long long *__restrict__ deg, uint32_t *__restrict__ key) {
    for (int64_t i = gtid(); i < n; i += gstride()) key[i] = static_cast<uint32_t>(deg[i]);
}

// rank[v] = position of v in the (degree, index) order
__global__ void k_invert(int64_t n, const int32_t *__restrict__ order, int32_t *__restrict__ rank) {
    for (int64_t i = gtid(); i < n; i += gstride()) rank[order[i]] = static_cast<int32_t>(i);
}

__global__ void k_fill_i32(int64_t n, int32_t *__restrict__ a, int32_t value) {
    for (int64_t i = gtid(); i < n; i += gstride()) a[i] = value;
}

// first i >= from with by_rank[i] unplaced
__global__ void k_first_unplaced(int64_t from, int64_t n, const int32_t *__restrict__ by_rank,
                                 const int32_t *__restrict__ pos, unsigned long long *__restrict__ out) {
    for (int64_t i = from + gtid(); i < n; i += gstride())
        if (pos[by_rank[i]] < 0) atomicMin(out, static_cast<unsigned long long>(i));
}

// degree-0 vertices: the first z entries of the (degree, index) order
__global__ void k_count_isolated(int64_t n, const int32_t *__restrict__ by_rank,
                                 const unsigned long long *__restrict__ deg, unsigned long long *__restrict__ z) {
    for (int64_t i = gtid(); i < n; i += gstride())
        if (deg[by_rank[i]] > 0) atomicMin(z, static_cast<unsigned long long>(i));
}

__global__ void k_place_prefix(int64_t z, const int32_t *__restrict__ by_rank, int32_t *__restrict__ order,
                               int32_t *__restrict__ pos) {
    for (int64_t i = gtid(); i < z; i += gstride()) {
        order[i] = by_rank[i];
        pos[by_rank[i]] = static_cast<int32_t>(i);
    }
}

__global__ void k_place_one(int64_t at, int64_t n, const int32_t *__restrict__ by_rank,
                            const unsigned long long *__restrict__ idx, int32_t *__restrict__ order,
                            int32_t *__restrict__ pos) {
    if (*idx >= static_cast<unsigned long long>(n)) return;  // nothing left (the host stops)
    const int32_t v = by_rank[*idx];
    order[at] = v;
    pos[v] = static_cast<int32_t>(at);
}

// Every unvisited neighbour of the level [lo, hi) is claimed by its earliest-placed
// neighbour there; the first claim of a vertex appends it to the candidate list.
__global__ void k_claim(int64_t lo, int64_t hi, const int32_t *__restrict__ order, const int64_t *__restrict__ gptr,
                        const int32_t *__restrict__ adj, const int32_t *__restrict__ pos, int32_t *__restrict__ claim,
                        int32_t *__restrict__ cand, unsigned long long *__restrict__ count) {
    const int lane = threadIdx.x & 31;
    for (int64_t i = lo + (gtid() >> 5); i < hi; i += gstride() >> 5) {
        const int32_t u = order[i];
        for (int64_t k = gptr[u] + lane; k < gptr[u + 1]; k += 32) {
            const int32_t v = adj[k];
            if (pos[v] >= 0) continue;
            const int32_t old = atomicMin(claim + v, static_cast<int32_t>(i - lo));
            if (old == INT_MAX) cand[atomicAdd(count, 1ull)] = v;
        }
    }
}

// Sort a level of at most kSmallSort candidates by (claim, rank) in one block
// (bitonic network on 64-bit keys), then place it.
__global__ void __launch_bounds__(1024) k_sort_place_small(int64_t c, int64_t at, const int32_t *__restrict__ cand,
                                                            int32_t *__restrict__ claim, const int32_t *__restrict__ rank,
                                                            const int32_t *__restrict__ by_rank,
                                                            int32_t *__restrict__ order, int32_t *__restrict__ pos) {
    __shared__ unsigned long long key[kSmallSort];
    int size = 1;
    while (size < c) size <<= 1;
    for (int i = threadIdx.x; i < size; i += blockDim.x) {
        if (i < c) {
            const int32_t v = cand[i];
            key[i] = (static_cast<unsigned long long>(claim[v]) << 32) | static_cast<uint32_t>(rank[v]);
        } else {
            key[i] = ~0ull;
        }
    }
    __syncthreads();
    for (int k = 2; k <= size; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < size; i += blockDim.x) {
                const int p = i ^ j;
                if (p > i) {
                    const bool up = (i & k) == 0;
                    const unsigned long long a = key[i], b = key[p];
                    if ((a > b) == up) {
                        key[i] = b;
                        key[p] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int i = threadIdx.x; i < c; i += blockDim.x) {
        const int32_t v = by_rank[static_cast<uint32_t>(key[i])];
        order[at + i] = v;
        pos[v] = static_cast<int32_t>(at + i);
        claim[v] = INT_MAX;
    }
}

__global__ void k_rank_keys(int64_t c, const int32_t *__restrict__ cand, const int32_t *__restrict__ rank,
                            uint32_t *__restrict__ key) {
    for (int64_t i = gtid(); i < c; i += gstride()) key[i] = static_cast<uint32_t>(rank[cand[i]]);
}

__global__ void k_claim_keys(int64_t c, const int32_t *__restrict__ v, const int32_t *__restrict__ claim,
                             uint32_t *__restrict__ key) {
    for (int64_t i = gtid(); i < c; i += gstride()) key[i] = static_cast<uint32_t>(claim[v[i]]);
}

__global__ void k_place_sorted(int64_t c, int64_t at, const int32_t *__restrict__ v, int32_t *__restrict__ claim,
                               int32_t *__restrict__ order, int32_t *__restrict__ pos) {
    for (int64_t i = gtid(); i < c; i += gstride()) {
        order[at + i] = v[i];
        pos[v[i]] = static_cast<int32_t>(at + i);
        claim[v[i]] = INT_MAX;
    }
}

__global__ void k_reverse(int64_t n, const int32_t *__restrict__ in, int32_t *__restrict__ out) {
    for (int64_t i = gtid(); i < n; i += gstride()) out[i] = in[n - 1 - i];
}

__global__ void k_len_keys(int64_t n, const int32_t *__restrict__ row_ptr, int32_t max_len,
                           uint32_t *__restrict__ key) {
    for (int64_t i = gtid(); i < n; i += gstride()) key[i] = static_cast<uint32_t>(max_len - (row_ptr[i + 1] - row_ptr[i]));
}

// status[0] |= entry out of range, status[1] |= index seen twice
__global__ void k_check_perm(int64_t n, const int32_t *__restrict__ perm, int32_t *__restrict__ seen,
                             int32_t *__restrict__ status) {
    for (int64_t i = gtid(); i < n; i += gstride()) {
        const int32_t p = perm[i];
        if (p < 0 || p >= n) {
            status[0] = 1;
            continue;
        }
        if (atomicAdd(seen + p, 1) != 0) status[1] = 1;
    }
}

__global__ void k_perm_lengths(int64_t n, const int32_t *__restrict__ perm, const int32_t *__restrict__ row_ptr,
                               int64_t *__restrict__ len) {
    for (int64_t i = gtid(); i < n; i += gstride()) len[i] = row_ptr[perm[i] + 1] - row_ptr[perm[i]];
}

// row i of B = row perm[i] of A, columns renamed through inv; one warp per row
template <typename T>
__global__ void k_perm_rows(int64_t n, const int32_t *__restrict__ perm, const int32_t *__restrict__ inv,
                            const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col,
                            const T *__restrict__ val, const int64_t *__restrict__ out_ptr,
                            int32_t *__restrict__ out_col, T *__restrict__ out_val) {
    const int lane = threadIdx.x & 31;
    for (int64_t i = gtid() >> 5; i < n; i += gstride() >> 5) {
        const int64_t src = row_ptr[perm[i]], len = row_ptr[perm[i] + 1] - src, dst = out_ptr[i];
        for (int64_t k = lane; k < len; k += 32) {
            out_col[dst + k] = inv[col[src + k]];
            out_val[dst + k] = val[src + k];
        }
    }
}

__global__ void k_i64_to_i32(int64_t n, const int64_t *__restrict__ in, int32_t *__restrict__ out) {
    for (int64_t i = gtid(); i < n; i += gstride()) out[i] = static_cast<int32_t>(in[i]);
}

template <typename T>
__global__ void k_permute_vector(int64_t n, const int32_t *__restrict__ perm, const T *__restrict__ src,
                                 T *__restrict__ dst, int direction) {
    for (int64_t i = gtid(); i < n; i += gstride()) {
        if (direction == 0)
            dst[i] = src[perm[i]];
        else
            dst[perm[i]] = src[i];
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Counting arrays of the radix passes, sized once for the largest sort.
struct RadixTemp {
    int64_t *counts = nullptr, *offsets = nullptr, *scan_tmp = nullptr;
    int init(Scratch &sc, int64_t max_n) {
        const int64_t nb = radix_blocks(max_n);
        SPMV_TRY(sc.get(&counts, 256 * nb + 1));
        SPMV_TRY(sc.get(&offsets, 256 * nb + 1));
        SPMV_TRY(sc.get(&scan_tmp, scan_temp_elems(256 * nb)));
        return SPMV_OK;
    }
};

// Stable LSD radix sort of (keys, vals) over the low `nbits` bits, 8 bits a pass; the
// pointers are swapped so that (keys, vals) hold the result.  k1/v1: same-size buffers.
int radix_sort(uint32_t *&keys, int32_t *&vals, uint32_t *&k1, int32_t *&v1, int64_t n, int nbits,
               const RadixTemp &t, cudaStream_t s) {
    if (n <= 1 || nbits <= 0) return SPMV_OK;
    for (int shift = 0; shift < nbits; shift += 8) {
        SPMV_TRY_CUDA(launch_radix_pass(keys, vals, n, shift, k1, v1, t.counts, t.offsets, t.scan_tmp, s));
        std::swap(keys, k1);
        std::swap(vals, v1);
    }
    return SPMV_OK;
}

int read_u64(const unsigned long long *d, unsigned long long *h, cudaStream_t s) {
    SPMV_TRY_CUDA(cudaMemcpyAsync(h, d, sizeof(*h), cudaMemcpyDeviceToHost, s));
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    return SPMV_OK;
}

int cuthill_mckee(int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col, int32_t *order,
                  cudaStream_t s) {
    Scratch sc(s);
    const int vbits = bits(static_cast<uint64_t>(n));  // keys up to n (the diagonal sentinel)
    // graph of A + A^T: sorted, distinct adjacency lists without self loops
    const int64_t m = 2 * nnz;
    uint32_t *u0 = nullptr, *u1 = nullptr;
    int32_t *v0 = nullptr, *v1 = nullptr;
    SPMV_TRY(sc.get(&u0, m));
    SPMV_TRY(sc.get(&u1, m));
    SPMV_TRY(sc.get(&v0, m));
    SPMV_TRY(sc.get(&v1, m));
    RadixTemp rt;
    SPMV_TRY(rt.init(sc, std::max<int64_t>(m, n)));
    if (m > 0) k_sym_edges<<<grid(n * 32), kThreads, 0, s>>>(n, row_ptr, col, u0, v0);
    SPMV_TRY_CUDA(cudaGetLastError());
    // by column, then stably by row: (row, column) order.  Rows and columns are both in
    // [0, n], so each sort's values serve as the next sort's keys.
    uint32_t *ka = reinterpret_cast<uint32_t *>(v0), *kb = reinterpret_cast<uint32_t *>(v1);
    int32_t *va = reinterpret_cast<int32_t *>(u0), *vb = reinterpret_cast<int32_t *>(u1);
    SPMV_TRY(radix_sort(ka, va, kb, vb, m, vbits, rt, s));  // ka: columns, va: rows
    uint32_t *kc = reinterpret_cast<uint32_t *>(va), *kd = reinterpret_cast<uint32_t *>(vb);
    int32_t *vc = reinterpret_cast<int32_t *>(ka), *vd = reinterpret_cast<int32_t *>(kb);
    SPMV_TRY(radix_sort(kc, vc, kd, vd, m, vbits, rt, s));  // kc: rows, vc: columns
    u0 = kc;
    v0 = vc;
    int64_t *flag = nullptr, *epos = nullptr, *scan_tmp = nullptr, *gptr = nullptr, *deg64 = nullptr;
    unsigned long long *deg;
    int32_t *adj = nullptr;
    SPMV_TRY(sc.get(&flag, m));
    SPMV_TRY(sc.get(&epos, m + 1));
    SPMV_TRY(sc.get(&scan_tmp, scan_temp_elems(std::max<int64_t>(m, n))));
    SPMV_TRY(sc.get(&deg, n));
    SPMV_TRY(sc.get(&gptr, n + 1));
    SPMV_TRY_CUDA(cudaMemsetAsync(deg, 0, sizeof(unsigned long long) * n, s));
    if (m > 0) k_mark_edges<<<grid(m), kThreads, 0, s>>>(m, n, u0, v0, flag, deg);
    SPMV_TRY_CUDA(cudaGetLastError());
    SPMV_TRY_CUDA(launch_exclusive_scan(flag, m, epos, scan_tmp, s));
    unsigned long long h_edges = 0;
    int64_t h_edges64 = 0;
    SPMV_TRY_CUDA(cudaMemcpyAsync(&h_edges64, epos + m, sizeof(int64_t), cudaMemcpyDeviceToHost, s));
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    h_edges = static_cast<unsigned long long>(h_edges64);
    SPMV_TRY(sc.get(&adj, static_cast<int64_t>(h_edges)));
    if (m > 0) k_compact_edges<<<grid(m), kThreads, 0, s>>>(m, flag, epos, v0, adj);
    deg64 = reinterpret_cast<int64_t *>(deg);  // counts < 2^63: same bits as int64
    SPMV_TRY_CUDA(launch_exclusive_scan(deg64, n, gptr, scan_tmp, s));
    SPMV_TRY_CUDA(cudaGetLastError());

    // (degree, index) order: stable sort of the indices by degree
    uint32_t *dk0 = nullptr, *dk1 = nullptr;
    int32_t *by_rank = nullptr, *r1 = nullptr, *rank = nullptr, *pos = nullptr, *claim = nullptr, *cand = nullptr;
    SPMV_TRY(sc.get(&dk0, n));
    SPMV_TRY(sc.get(&dk1, n));
    SPMV_TRY(sc.get(&by_rank, n));
    SPMV_TRY(sc.get(&r1, n));
    SPMV_TRY(sc.get(&rank, n));
    SPMV_TRY(sc.get(&pos, n));
    SPMV_TRY(sc.get(&claim, n));
    SPMV_TRY(sc.get(&cand, n));
    k_deg_keys<<<grid(n), kThreads, 0, s>>>(n, deg, dk0);
    k_iota<<<grid(n), kThreads, 0, s>>>(n, by_rank);
    SPMV_TRY(radix_sort(dk0, by_rank, dk1, r1, n, vbits, rt, s));
    k_invert<<<grid(n), kThreads, 0, s>>>(n, by_rank, rank);
    k_fill_i32<<<grid(n), kThreads, 0, s>>>(n, pos, -1);
    k_fill_i32<<<grid(n), kThreads, 0, s>>>(n, claim, INT_MAX);
    SPMV_TRY_CUDA(cudaGetLastError());

    unsigned long long *cell;  // [0] isolated count / first unplaced, [1] level size
    SPMV_TRY(sc.get(&cell, 2));
    const unsigned long long n_ull = static_cast<unsigned long long>(n);
    SPMV_TRY_CUDA(cudaMemcpyAsync(cell, &n_ull, sizeof(n_ull), cudaMemcpyHostToDevice, s));
    k_count_isolated<<<grid(n), kThreads, 0, s>>>(n, by_rank, deg, cell);
    unsigned long long z = 0;
    SPMV_TRY(read_u64(cell, &z, s));
    if (z > 0) k_place_prefix<<<grid(static_cast<int64_t>(z)), kThreads, 0, s>>>(static_cast<int64_t>(z), by_rank, order, pos);
    SPMV_TRY_CUDA(cudaGetLastError());

    // sort buffers for large levels
    uint32_t *lk0 = nullptr, *lk1 = nullptr;
    int32_t *lv0 = nullptr, *lv1 = nullptr;
    SPMV_TRY(sc.get(&lk0, n));
    SPMV_TRY(sc.get(&lk1, n));
    SPMV_TRY(sc.get(&lv0, n));
    SPMV_TRY(sc.get(&lv1, n));

    int64_t placed = static_cast<int64_t>(z);
    int64_t from = placed;  // vertices before `from` in (degree, index) order are placed
    while (placed < n) {
        // next component: its unplaced vertex of least (degree, index)
        SPMV_TRY_CUDA(cudaMemcpyAsync(cell, &n_ull, sizeof(n_ull), cudaMemcpyHostToDevice, s));
        k_first_unplaced<<<grid(n - from), kThreads, 0, s>>>(from, n, by_rank, pos, cell);
        k_place_one<<<1, 1, 0, s>>>(placed, n, by_rank, cell, order, pos);
        SPMV_TRY_CUDA(cudaGetLastError());
        unsigned long long first = 0;
        SPMV_TRY(read_u64(cell, &first, s));
        if (first >= n_ull) return set_error(SPMV_ERR_CUDA, "Cuthill-McKee: no unplaced vertex left");
        from = static_cast<int64_t>(first) + 1;
        int64_t lo = placed, hi = placed + 1;
        placed = hi;
        while (lo < hi) {
            SPMV_TRY_CUDA(cudaMemsetAsync(cell + 1, 0, sizeof(unsigned long long), s));
            k_claim<<<grid((hi - lo) * 32), kThreads, 0, s>>>(lo, hi, order, gptr, adj, pos, claim, cand, cell + 1);
            SPMV_TRY_CUDA(cudaGetLastError());
            unsigned long long c = 0;
            SPMV_TRY(read_u64(cell + 1, &c, s));
            const int64_t cnt = static_cast<int64_t>(c);
            if (cnt == 0) break;
            if (cnt <= kSmallSort) {
                k_sort_place_small<<<1, 1024, 0, s>>>(cnt, placed, cand, claim, rank, by_rank, order, pos);
            } else {
                // by rank, then stably by claiming position
                k_rank_keys<<<grid(cnt), kThreads, 0, s>>>(cnt, cand, rank, lk0);
                SPMV_TRY_CUDA(cudaMemcpyAsync(lv0, cand, sizeof(int32_t) * cnt, cudaMemcpyDeviceToDevice, s));
                uint32_t *la = lk0, *lb = lk1;
                int32_t *wa = lv0, *wb = lv1;
                SPMV_TRY(radix_sort(la, wa, lb, wb, cnt, vbits, rt, s));
                k_claim_keys<<<grid(cnt), kThreads, 0, s>>>(cnt, wa, claim, la);
                SPMV_TRY(radix_sort(la, wa, lb, wb, cnt, bits(static_cast<uint64_t>(hi - lo)), rt, s));
                k_place_sorted<<<grid(cnt), kThreads, 0, s>>>(cnt, placed, wa, claim, order, pos);
            }
            SPMV_TRY_CUDA(cudaGetLastError());
            lo = hi;
            hi = placed + cnt;
            placed = hi;
        }
    }
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    return SPMV_OK;
}

}  // namespace

int compute_ordering(int ordering, int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col,
                     int32_t max_len, const int32_t *user_perm, int32_t *perm, cudaStream_t s) {
    if (n == 0) return SPMV_OK;
    switch (ordering) {
        case SPMV_ORDER_NATURAL:
            k_iota<<<grid(n), kThreads, 0, s>>>(n, perm);
            SPMV_TRY_CUDA(cudaGetLastError());
            return SPMV_OK;
        case SPMV_ORDER_ROW_LENGTH: {
            Scratch sc(s);
            RadixTemp rt;
            SPMV_TRY(rt.init(sc, n));
            uint32_t *k0 = nullptr, *k1 = nullptr;
            int32_t *v1 = nullptr;
            SPMV_TRY(sc.get(&k0, n));
            SPMV_TRY(sc.get(&k1, n));
            SPMV_TRY(sc.get(&v1, n));
            k_len_keys<<<grid(n), kThreads, 0, s>>>(n, row_ptr, max_len, k0);
            k_iota<<<grid(n), kThreads, 0, s>>>(n, perm);
            SPMV_TRY_CUDA(cudaGetLastError());
            int32_t *vals = perm;
            SPMV_TRY(radix_sort(k0, vals, k1, v1, n, bits(static_cast<uint64_t>(max_len)), rt, s));
            if (vals != perm) SPMV_TRY_CUDA(cudaMemcpyAsync(perm, vals, sizeof(int32_t) * n, cudaMemcpyDeviceToDevice, s));
            SPMV_TRY_CUDA(cudaStreamSynchronize(s));
            return SPMV_OK;
        }
        case SPMV_ORDER_RCM: {
            Scratch sc(s);
            int32_t *order = nullptr;
            SPMV_TRY(sc.get(&order, n));
            SPMV_TRY(cuthill_mckee(n, nnz, row_ptr, col, order, s));
            k_reverse<<<grid(n), kThreads, 0, s>>>(n, order, perm);
            SPMV_TRY_CUDA(cudaGetLastError());
            SPMV_TRY_CUDA(cudaStreamSynchronize(s));
            return SPMV_OK;
        }
        case SPMV_ORDER_USER: {
            if (!user_perm) return set_error(SPMV_ERR_INVALID_ARG, "ordering USER needs a permutation");
            Scratch sc(s);
            int32_t *seen = nullptr, *status = nullptr;
            SPMV_TRY(sc.get(&seen, n));
            SPMV_TRY(sc.get(&status, 2));
            SPMV_TRY_CUDA(cudaMemsetAsync(seen, 0, sizeof(int32_t) * n, s));
            SPMV_TRY_CUDA(cudaMemsetAsync(status, 0, sizeof(int32_t) * 2, s));
            k_check_perm<<<grid(n), kThreads, 0, s>>>(n, user_perm, seen, status);
            SPMV_TRY_CUDA(cudaGetLastError());
            int32_t st[2] = {0, 0};
            SPMV_TRY_CUDA(cudaMemcpyAsync(st, status, sizeof(st), cudaMemcpyDeviceToHost, s));
            SPMV_TRY_CUDA(cudaStreamSynchronize(s));
            if (st[0] || st[1])
                return set_error(SPMV_ERR_INVALID_ARG, "perm is not a permutation of 0..n-1");
            SPMV_TRY_CUDA(cudaMemcpyAsync(perm, user_perm, sizeof(int32_t) * n, cudaMemcpyDeviceToDevice, s));
            return SPMV_OK;
        }
        default:
            return set_error(SPMV_ERR_INVALID_ARG, "unknown ordering");
    }
}

int permute_csr(int dtype, int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col, const void *val,
                const int32_t *perm, int32_t *out_ptr, int32_t *out_col, void *out_val, cudaStream_t s) {
    if (n == 0) {
        SPMV_TRY_CUDA(cudaMemsetAsync(out_ptr, 0, sizeof(int32_t), s));
        return SPMV_OK;
    }
    Scratch sc(s);
    int32_t *inv = nullptr;
    int64_t *len = nullptr, *ptr64 = nullptr, *scan_tmp = nullptr;
    SPMV_TRY(sc.get(&inv, n));
    SPMV_TRY(sc.get(&len, n));
    SPMV_TRY(sc.get(&ptr64, n + 1));
    SPMV_TRY(sc.get(&scan_tmp, scan_temp_elems(n)));
    k_invert<<<grid(n), kThreads, 0, s>>>(n, perm, inv);
    k_perm_lengths<<<grid(n), kThreads, 0, s>>>(n, perm, row_ptr, len);
    SPMV_TRY_CUDA(cudaGetLastError());
    SPMV_TRY_CUDA(launch_exclusive_scan(len, n, ptr64, scan_tmp, s));
    k_i64_to_i32<<<grid(n + 1), kThreads, 0, s>>>(n + 1, ptr64, out_ptr);
    if (nnz > 0) {
        if (dtype == SPMV_F64)
            k_perm_rows<double><<<grid(n * 32), kThreads, 0, s>>>(n, perm, inv, row_ptr, col,
                                                                  static_cast<const double *>(val), ptr64, out_col,
                                                                  static_cast<double *>(out_val));
        else
            k_perm_rows<float><<<grid(n * 32), kThreads, 0, s>>>(n, perm, inv, row_ptr, col,
                                                                 static_cast<const float *>(val), ptr64, out_col,
                                                                 static_cast<float *>(out_val));
    }
    SPMV_TRY_CUDA(cudaGetLastError());
    SPMV_TRY_CUDA(cudaStreamSynchronize(s));
    return SPMV_OK;
}

cudaError_t launch_permute_vector(int dtype, int64_t n, const int32_t *perm, const void *src, void *dst,
                                  int direction, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    if (dtype == SPMV_F64)
        k_permute_vector<double><<<grid(n, 1 << 20), kThreads, 0, s>>>(n, perm, static_cast<const double *>(src),
                                                                       static_cast<double *>(dst), direction);
    else
        k_permute_vector<float><<<grid(n, 1 << 20), kThreads, 0, s>>>(n, perm, static_cast<const float *>(src),
                                                                      static_cast<float *>(dst), direction);
    return cudaGetLastError();
}

}  // namespace spmv
