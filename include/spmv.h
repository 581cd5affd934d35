/*
 * spmv.h -- C interface of the GB300 (sm_103a) sparse matrix-vector product library.
 *
 * The library computes y = A x for a square n x n sparse matrix A handed over in
 * compressed sparse row (CSR) form: row_ptr[n+1], col_idx[nnz], vals[nnz].
 * The GPGPU spMVM paper (arXiv 1112.5588, introduction) identifies this product as
 * the part of iterative sparse solvers that usually takes most of the time; the CSR
 * arrays are the Ap/Aj/Ax of "Development of Krylov and AMG linear solvers for
 * large-scale sparse matrices on GPUs", matrix formats, Figure 3.
 *
 * A build call converts the CSR input, on the device, into one of the storage
 * formats the pages describe and returns an opaque handle; apply calls reuse it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named row_ptr, col_idx, vals, x, y, perm, slice_ptr are DEVICE
 *    pointers of the current CUDA device, unless the name ends in _host.
 *  - Indices are int32; n < 2^31 and nnz < 2^31.  row_ptr[0] = 0, row_ptr is
 *    non-decreasing, row_ptr[n] = nnz, every column lies in [0, n).  Entries of a
 *    row may come in any order; duplicate columns are kept and summed; explicit
 *    zeros are kept as entries.
 *  - Values and vectors use the handle's value type: SPMV_F64 (double) or
 *    SPMV_F32 (float).  x and y have n elements and must not overlap.
 *  - Streams are cudaStream_t values passed as void*; NULL is the legacy default stream.
 *  - Errors: functions returning int return an spmv_status (0 = success); functions
 *    returning a handle return NULL on failure.  In both cases spmv_last_error()
 *    and spmv_last_error_message() describe the failure for the calling thread.
 *    No entry point traps or aborts on bad input; every entry point except
 *    spmv_csr_apply_noalloc validates its matrix.
 *  - Environment: SPMV_LOG set to anything but "" or "0" makes every successful build
 *    write its plan (the spmv_describe JSON) to stderr as one line "spmv: built {...}";
 *    SPMV_FAIL_ALLOC injects a device allocation failure (see spmv_device_memory).
 */
#ifndef SPMV_GB300_H
#define SPMV_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPMV_API __attribute__((visibility("default")))
#else
#define SPMV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spmv_handle_s *spmv_handle_t;

/* value type of the matrix, x and y */
typedef enum { SPMV_F64 = 0, SPMV_F32 = 1 } spmv_dtype;

/*
 * Storage formats.
 *  SPMV_FMT_CSR_VECTOR  CSR kept as given; a group of g lanes (g = 2..32, chosen per
 *      row-length bin) works on one row and combines its partial sums with warp
 *      shuffles.  Source: "Load-balancing Sparse Matrix Vector Product Kernels on
 *      GPUs" (scite report), quoted "Sparse Linear Algebra on AMD and NVIDIA GPUs",
 *      the subwarp-per-row CSR algorithm; row-length classes from the Trilinos issue
 *      "Tpetra::CrsMatrix::unpackAndCombine: Optimize GPU unpack for few long rows".
 *  SPMV_FMT_ELL_R       ELLPACK-R: rows shifted left into an n x max-row-length
 *      rectangle stored column by column (leading dimension a multiple of 32) plus a
 *      row-length array, one thread per row that stops at its row's end.  GPGPU
 *      spMVM paper, ELLPACK-R section, Figs. 1-2.
 *  SPMV_FMT_SELL        SELL-C-sigma: rows sorted by length inside windows of sigma
 *      rows, cut into slices of C rows, each slice padded to its longest row and
 *      stored column by column.  sigma = n is pJDS (GPGPU spMVM paper, pJDS section,
 *      Fig. 1 "sort" and "pad"), sigma = 1 keeps the natural order; SELL-P is the
 *      sliced ELL of the scite report's abstract.
 *  SPMV_FMT_HYB         ELL part of width K plus a spill holding the rest of each
 *      row, as COO (HYB) or CSR (HEC); the ELL part is computed first and writes y,
 *      the spill adds into y.  Krylov/AMG paper, matrix formats, Figs. 1-3 and the
 *      HEC SpMV algorithm.
 *  SPMV_FMT_MERGE       CSR kept as given, every row processed by the load-balanced
 *      merge-path pass: each CTA takes an equal share of the sequence that merges
 *      row ends with entries, whatever the row lengths (the merge-path split the
 *      Trilinos issue attributes to the vendor library; the load-balanced CSR/COO
 *      kernels of the scite report's abstract).  Suited to irregular matrices.
 *  SPMV_FMT_AUTO        the builder picks one of the above from the row lengths.
 * In SELL, ELLPACK-R and CSR-vector, rows longer than the long-row threshold are
 * taken out and handled by a row-split pass: each is cut into chunks of 2048 entries
 * (4096 in float64 when the chunks run in the same launch as one-thread-per-row
 * slices), one warp per chunk, and the chunk sums of a row combine in a tree (the class of the
 * longest rows in the Trilinos issue, processed in pieces).  So no single thread walks
 * a very long row.
 */
typedef enum {
    SPMV_FMT_AUTO = 0,
    SPMV_FMT_CSR_VECTOR = 1,
    SPMV_FMT_ELL_R = 2,
    SPMV_FMT_SELL = 3,
    SPMV_FMT_HYB = 4,
    SPMV_FMT_MERGE = 5
} spmv_format;

/*
 * Tuning parameters; a negative value (or 0 where noted) means "choose automatically".
 *   C                   SELL slice height: a power of two from 32 to 1024 (a whole number of
 *                       warps; 32 and 64 have compiled-in addressing).  Automatic = 32.
 *   sigma               SELL sort window in rows: 1 = no sort, >= n = global sort (pJDS).
 *   K                   HYB ELL width.  Automatic: the smallest K with
 *                       4 * (value_bytes + 8) * #{rows longer than K} <= ld * (value_bytes + 4):
 *                       each spilled entry's bytes count four times, since the spill pass
 *                       costs about four times its bytes in time against the streamed ELL
 *                       slots.
 *   spill_csr           HYB spill kind: 1 = CSR (HEC), 0 = COO (HYB).  Automatic = COO
 *                       (faster on the irregular matrices measured).
 *   long_row_threshold  rows with more entries go to the row-split pass.  0 = never.
 *                       Automatic: 128 for SELL / ELLPACK-R, 256 for CSR-vector.
 *   subwarp             CSR-vector lanes per row (2, 4, 8, 16 or 32) for every row;
 *                       automatic = per row-length bin, about eight entries a lane: 2
 *                       lanes up to 16 entries, 4 up to 32, 8 up to 64, 16 up to 128,
 *                       32 above.
 *   row_threads         threads per row in the SELL / ELLPACK-R / HYB-ELL apply (1, 2, 4,
 *                       8, 16 or 32), the multi-thread-per-row ELL variants of the
 *                       load-balancing SpMV paper.  Automatic: 1, unless one thread per
 *                       row gives fewer than two waves of threads on the device; then it
 *                       doubles while that holds and an average stored row still gives
 *                       each thread at least 16 entries.
 *   row_group_mode      with row_threads = G > 1: 0 = row-grouped (column-major slots,
 *                       G adjacent threads per row striding over its entries); 1 =
 *                       interleaved slots (a row's entries in groups of G side by side,
 *                       same threads, so a warp reads 32 consecutive slots); 2 =
 *                       column-grouped (column-major slots, a warp per 32 rows and
 *                       residue class of entries mod G, G warps per row combined in
 *                       shared memory; G <= 8).  Automatic = 1.
 *   x_policy            L2 policy of the x gathers in the sliced formats: 0 = plain
 *                       read-only loads, 1 = evict-last hint (x stays in L2 while the
 *                       matrix streams past it).  Automatic: 1 for float64 when the rows
 *                       are sorted (sigma > 1), x is at most a quarter of L2 and the
 *                       matrix stream is larger than L2; otherwise 0.
 *   vector_loads        1 = one thread per row reads its row 4 entries at a time with
 *                       16-byte loads (indices in groups of 4, values in 16-byte groups,
 *                       slice widths rounded up to a multiple of 4); 0 = element loads.
 *                       Takes one thread per row (an automatic row_threads becomes 1; an
 *                       explicit row_threads > 1 is SPMV_ERR_UNSUPPORTED).  Automatic = 0.
 *   host_blocks         row blocks of the spmv_apply_host pipeline: k >= 2 = k blocks of
 *                       row positions, each multiplied as soon as the pieces of x its
 *                       columns reach have arrived, its rows of y copied back while later
 *                       pieces of x are still coming in; 0 or 1 = off (x is copied in whole,
 *                       then the product runs).  Needs a plan of one-thread-per-row sliced
 *                       rows with no separate pass (SELL / ELLPACK-R, column-major slots, no
 *                       long rows), blocks that are whole sort windows, and page-locked host
 *                       arrays; otherwise the unpipelined path runs.  Automatic = off: it
 *                       pays only where the product takes long against the transfers.  On
 *                       a GB300 host link where each copy carries about 8 us of fixed
 *                       latency and each direction slows to about 154 GB/s while the other
 *                       is busy: -10 % per call on the HMEp-shaped matrix with 8 blocks,
 *                       -3 % on the 3D Laplacian in float64 with 4, +9 % in float32.
 *   staged              SELL-32 with one thread per row: 1 = the slots of each group of 8
 *                       slices reach shared memory by bulk copies (the copy engine streams
 *                       the matrix; the load units serve only the gathers of x), and long
 *                       rows' chunks run in a launch of their own; 0 = every thread loads its
 *                       own slots.  Automatic = 0.  Takes one thread per row (an automatic
 *                       row_threads becomes 1); SPMV_ERR_UNSUPPORTED when asked for on another
 *                       layout.
 */
typedef struct {
    int32_t C;
    int64_t sigma;
    int32_t K;
    int32_t spill_csr;
    int32_t long_row_threshold;
    int32_t subwarp;
    int32_t row_threads;
    int32_t row_group_mode;
    int32_t x_policy;
    int32_t vector_loads;
    int32_t host_blocks;
    int32_t staged;
} spmv_format_params;

typedef enum {
    SPMV_OK = 0,
    SPMV_ERR_INVALID_ARG = -1, /* NULL pointer, bad size, bad enum value */
    SPMV_ERR_BAD_CSR = -2,     /* row_ptr not monotone / wrong ends, column out of range */
    SPMV_ERR_CUDA = -3,        /* a CUDA runtime call failed (message has the CUDA error) */
    SPMV_ERR_OOM = -4,         /* device allocation failed */
    SPMV_ERR_TOO_LARGE = -5,   /* the requested layout would exceed the library's size limits */
    SPMV_ERR_UNSUPPORTED = -6, /* parameter combination not supported */
    SPMV_ERR_TIMEOUT = -7      /* reserved: a bounded device wait ran out */
} spmv_status;

/* Fill *p with "all automatic" values.  Returns SPMV_OK or SPMV_ERR_INVALID_ARG. */
SPMV_API int spmv_default_params(spmv_format_params *p);

/*
 * The device memory this library holds right now, over all handles and all calls in
 * progress: the number of its live device allocations and their total size in bytes
 * (build temporaries, handle arrays, per-stream scratch, solver workspaces; not the
 * fixed scratch array of spmv_csr_apply_noalloc, which is part of the library's device
 * image).  No page has a counterpart: it lets a caller account for the library's share
 * of device memory, and tests check with it that failed calls release what they took.
 * Either pointer (host memory) may be NULL.  Always returns SPMV_OK.
 *
 * Fault injection (host side, for tests): when the environment variable SPMV_FAIL_ALLOC
 * holds a positive integer k, the k-th device allocation the library attempts after the
 * variable took that value fails as if the device were out of memory -- once; the count
 * restarts whenever the value changes, unset included.  The call that made it returns
 * SPMV_ERR_OOM after releasing what it had allocated.
 */
SPMV_API int spmv_device_memory(int64_t *allocations, int64_t *bytes);

/*
 * Build a handle from a device CSR matrix.
 *   n, nnz    matrix order and number of stored entries (0 allowed for both).
 *   row_ptr   int32[n+1], col_idx int32[nnz], vals double/float[nnz]: device memory,
 *             only read; the handle keeps its own copies, so the caller may free or
 *             overwrite them once the call returns.
 *   dtype     spmv_dtype; format: spmv_format.
 * The work runs on the legacy default stream and the call returns after it has
 * finished; inputs written on other streams must be complete before the call.
 * The CSR is validated on the device; a malformed matrix returns NULL with
 * SPMV_ERR_BAD_CSR.  A fixed format whose storage would not fit returns NULL with
 * SPMV_ERR_TOO_LARGE or SPMV_ERR_OOM; there is never a silent change of format.
 */
SPMV_API spmv_handle_t spmv_build_from_csr(int64_t n, int64_t nnz, const int32_t *row_ptr,
                                  const int32_t *col_idx, const void *vals, int dtype, int format);

/* As spmv_build_from_csr, with tuning parameters (NULL = automatic) and a stream
 * (the build is ordered after earlier work on that stream and synchronises it). */
SPMV_API spmv_handle_t spmv_build_from_csr_ex(int64_t n, int64_t nnz, const int32_t *row_ptr,
                                     const int32_t *col_idx, const void *vals, int dtype,
                                     int format, const spmv_format_params *params, void *stream);

/*
 * y = A x, overwriting y (no scaling, no accumulation into the old y).
 * x and y are device arrays of n elements of the handle's value type, in the
 * caller's original row order (any row permutation of the format is internal);
 * overlapping x and y, and an x or y that is not memory of the current device (host
 * memory, pinned or not, or another device's), are refused with SPMV_ERR_INVALID_ARG
 * before anything is enqueued.  The same holds for the vectors of spmv_apply_ex,
 * spmv_apply_multi, spmv_apply_profiled, spmv_permute_vector and the solvers.
 * Asynchronous on `stream`: returns after enqueueing 1 to 6 kernel launches (one for the
 * SELL / ELLPACK-R plans AUTO picks; CSR-vector: one per row-length bin and the row-split).
 * The apply only reads the handle's matrix data.  What it writes besides y (the carries
 * of the merge-path and COO passes, the chunk partials and counters of the row-split
 * pass) the handle keeps once per stream: the first apply of a handle on a stream
 * allocates that stream's set (a few bytes per long row or per chunk of the
 * segmented part; the build's own stream gets its set during the build), and later
 * applies on the stream reuse it in stream order.  A first apply inside a stream
 * capture allocates and initialises the set at once, outside the graph, so the graph
 * and applies enqueued on that stream outside it both find the set ready.  So applies of one handle on
 * different streams may run concurrently, and so may applies of different handles.
 * The sets are keyed by the stream handle and live until spmv_destroy; a graph
 * captured on a stream keeps using that stream's set, so replaying it concurrently
 * with other work on the same stream races.  A stream created after another was
 * destroyed may get the same handle value and so the same set: destroy a stream only
 * once its applies have finished (cudaStreamDestroy returns before they do).
 * Empty rows give +0.
 */
SPMV_API int spmv_apply(spmv_handle_t h, const void *x, void *y, void *stream);

/*
 * y_host = A x_host with host arrays: copies x to the device, applies, moves y back
 * and waits for the stream.  Page-locked (pinned) host buffers give the full copy
 * bandwidth.  Three ways, chosen per call:
 *  - pipelined (see host_blocks): x goes in by pieces on a copy stream, each block of
 *    rows is multiplied once the pieces of x it reads have arrived and its rows of y
 *    go back on a second copy stream, so the two link directions and the product
 *    overlap.  The first call on a handle reads the column reach of every block (one
 *    pass over the matrix, synchronous) and decides;
 *  - y direct: when y_host is page-locked and the plan writes each row of y once (SELL
 *    / ELLPACK-R without a separate accumulating pass), the kernels store y straight
 *    into it, so the transfer back overlaps the product;
 *  - staged: x copied in, product, y copied out.
 * The result is the same in every way (the same kernel sums each row in the same
 * order).  x_host and y_host may be the same array (in place); such a call runs
 * unpipelined, with all of x on the device before any of y moves.  The device staging
 * columns belong to the stream's scratch set (allocated on the first call on each
 * stream); the pipeline's copy streams and events are created by the first call on a
 * handle, kept until spmv_destroy, and shared, so pipelined calls of one handle run
 * one at a time.
 */
SPMV_API int spmv_apply_host(spmv_handle_t h, const void *x_host, void *y_host, void *stream);

/*
 * y_host = A x_host with page-locked host arrays (cudaHostAlloc, or cudaHostRegister'ed)
 * read and written by the kernels themselves through their device mapping: no staging
 * copy.  On a GPU attached to its CPU by a coherent link (Grace + Blackwell over
 * NVLink-C2C) the gathers of x and the stores of y cross the link while the matrix
 * streams from HBM, instead of two copy-engine transfers around the product.  Waits
 * for the stream.  SPMV_ERR_INVALID_ARG if either array is not page-locked host memory or
 * the two overlap.
 */
SPMV_API int spmv_apply_mapped(spmv_handle_t h, const void *x_host, void *y_host, void *stream);

/*
 * As spmv_apply, but records CUDA events around each kernel it launches, waits for
 * them and writes each launch's device time in milliseconds to kernel_ms[0..cap).
 * Returns the number of kernels launched (>= 0) or a negative spmv_status.  Meant
 * for measurement, not for the hot loop.
 */
SPMV_API int spmv_apply_profiled(spmv_handle_t h, const void *x, void *y, void *stream, float *kernel_ms,
                        int cap);

/*
 * y = alpha * A x + beta * y.  When beta == 0, y is not read (any content, NaN
 * included, is overwritten); alpha = 1, beta = 0 is spmv_apply.  Solvers use this
 * form for residuals r = b - A x (alpha = -1, beta = 1 with y holding b), as the
 * Krylov iterations of the Krylov/AMG paper (BiCGSTAB algorithm) combine SpMV with
 * vector updates.  SELL and ELLPACK-R handles fold alpha and beta into the kernel's
 * single write of each row; the other formats compute A x into a scratch column first
 * (n values, allocated on the first such call on each stream and kept with the
 * stream's scratch set).  x and y must not overlap.  Asynchronous; same stream rules
 * as spmv_apply.
 */
SPMV_API int spmv_apply_ex(spmv_handle_t h, double alpha, const void *x, double beta, void *y, void *stream);

/*
 * Y = alpha * A X + beta * Y for k right-hand sides at once.  X and Y are row-major
 * n x k blocks in device memory: element (row j, vector c) at X[j * ldx + c] and
 * Y[j * ldy + c], with ldx >= k and ldy >= k.  The matrix is streamed once per group
 * of up to 8 vectors and each gather of a row of X fetches that row's values with
 * one or two wide loads (SELL handles, slice height 32 or 64; X aligned to
 * min(16, 8 * value size) bytes with ldx a multiple of that); other formats and
 * left-over columns go one column at a time through two scratch columns of the
 * stream's scratch set (allocated on first need).
 * beta == 0: Y is not read.  k = 0 is a no-op.  X and Y must not overlap (their spans
 * of (n - 1) * ld + k elements; SPMV_ERR_INVALID_ARG otherwise).  Asynchronous.
 */
SPMV_API int spmv_apply_multi(spmv_handle_t h, int64_t k, double alpha, const void *X, int64_t ldx, double beta,
                              void *Y, int64_t ldy, void *stream);

/*
 * Solve A x = b by conjugate gradients (Hestenes-Stiefel), the Krylov iteration the
 * Krylov/AMG paper lists among its solvers (section on Krylov subspace algorithms),
 * built on this handle's apply and on device vector kernels.  A must be symmetric
 * positive definite; the handle's format does not matter.
 *
 *   b     device vector, length n, the handle's value type; read only.
 *   x     device vector, length n: the initial guess on entry, the iterate on return.
 *         Must not overlap b.
 *   rtol  stop at the first iteration k with ||r_k||_2 <= rtol * ||b||_2, where r_k is
 *         the recurrence residual (||b|| is replaced by 1 when b = 0).  rtol = 0 runs
 *         exactly max_iter iterations unless the residual reaches 0.
 *   max_iter  upper bound on iterations (0: only the initial residual is computed).
 *   iterations, relative_residual  (host pointers, may be NULL) iterations done and
 *         ||r_k|| / ||b|| at the end.
 *
 * Arithmetic: vectors in the value type; every dot product and the step lengths in
 * double, reduced in a fixed order (results are reproducible).  Workspace (4 vectors:
 * r, p, A p and the iterate) is taken from the stream-ordered pool of `stream` and
 * returned before the call ends.  While the solve runs, the calling thread keeps two
 * iterations queued, pacing itself on a small page-locked progress record (allocated
 * once per thread) that the kernels update; at most two iterations' products run
 * after the stop.
 * Synchronises `stream`.  Returns SPMV_ERR_UNSUPPORTED (after filling the outputs) if
 * p.Ap <= 0 at some step, i.e. A is not positive definite; SPMV_ERR_INVALID_ARG for a
 * NULL handle or vector, overlapping b and x, max_iter < 0 or rtol < 0 / NaN.
 */
SPMV_API int spmv_cg(spmv_handle_t h, const void *b, void *x, double rtol, int32_t max_iter, void *stream,
                     int32_t *iterations, double *relative_residual);

/*
 * Solve A x = b by BiCGSTAB (van der Vorst), unpreconditioned, with the shadow residual
 * r_hat = r_0: the nonsymmetric Krylov solver the Krylov/AMG paper uses for its 3D
 * Poisson tests.  Two products per step on this handle plus device vector kernels.
 * Arguments, stopping rule, arithmetic, workspace (7 vectors) and errors as spmv_cg;
 * SPMV_ERR_UNSUPPORTED (after filling the outputs) on a breakdown: (r_hat, r) = 0,
 * (r_hat, A p) = 0, or omega = 0 before convergence.
 */
SPMV_API int spmv_bicgstab(spmv_handle_t h, const void *b, void *x, double rtol, int32_t max_iter, void *stream,
                           int32_t *iterations, double *relative_residual);

/*
 * Solve A x = b by restarted GMRES(m) (Saad and Schultz), unpreconditioned: the third
 * Krylov solver the Krylov/AMG paper lists beside CG and BiCGSTAB.  Each Arnoldi step
 * is one product on this handle, Gram-Schmidt orthogonalisation applied twice (fused
 * multi-dot and multi-axpy kernels over the basis), and a Givens rotation of the
 * Hessenberg column; a cycle ends after `restart` steps or when the rotated residual
 * estimate meets the test, and then x is updated and the true residual b - A x is
 * recomputed.
 *   restart  m, the Krylov dimension of a cycle: 1 .. 64.
 * Other arguments, arithmetic and pacing as spmv_cg.  The solve stops when the true
 * residual at the end of a cycle meets ||b - A x|| <= rtol ||b|| (||b|| -> 1 when
 * b = 0) or after max_iter Arnoldi steps over all cycles; iterations counts those steps
 * and relative_residual is the true residual.  Workspace: m + 2 vectors and the small
 * Hessenberg state.  Returns SPMV_ERR_UNSUPPORTED (after filling the outputs) on a zero
 * pivot of the rotated Hessenberg matrix (A singular on the Krylov space).
 */
SPMV_API int spmv_gmres(spmv_handle_t h, const void *b, void *x, int32_t restart, double rtol, int32_t max_iter,
                        void *stream, int32_t *iterations, double *relative_residual);

/*
 * Orderings of the permuted basis (spmv_build_permuted).  perm maps a position of the
 * basis to an original index (new -> old).
 *   NATURAL     the identity.
 *   ROW_LENGTH  rows by length, longest first, ties in index order: the sort of the
 *               GPGPU spMVM paper's pJDS format, over the whole matrix.
 *   RCM         reverse Cuthill-McKee on the graph of A + A^T (an edge for every stored
 *               entry off the diagonal): vertices of degree 0 first in index order, each
 *               component started at its unvisited vertex of least (degree, index),
 *               neighbours appended by (degree, index), the whole order reversed.  It
 *               brings entries next to the diagonal, so the gathers of x stay within a
 *               narrow window.  Build cost grows with the number of breadth-first levels
 *               and of connected components (each is a few kernel launches).
 *   USER        the caller's permutation.
 */
typedef enum {
    SPMV_ORDER_NATURAL = 0,
    SPMV_ORDER_ROW_LENGTH = 1,
    SPMV_ORDER_RCM = 2,
    SPMV_ORDER_USER = 3
} spmv_ordering;

/*
 * Build a handle for the matrix in a permuted basis, B = P A P^T: row and column i of
 * B are row and column perm[i] of A.  The GPGPU spMVM paper (pJDS section) notes that a
 * Krylov solver needs the permutation only before the first and after the last
 * iteration, all products in between running on permuted vectors; this is that mode.
 * Every apply, scaled apply, multi-vector apply and spmv_cg of the handle works in the
 * permuted basis (x and y are permuted vectors); spmv_permute_vector moves vectors in
 * and out, spmv_get_permutation returns perm, spmv_to_csr returns B.
 *   n .. format, params, stream  as spmv_build_from_csr_ex (A is validated first).
 *   ordering   spmv_ordering; perm (ordering USER only): device int32[n], a permutation
 *              of 0..n-1 (checked: SPMV_ERR_INVALID_ARG otherwise).
 * The ordering and B are computed on the device.  Returns NULL on error.
 */
SPMV_API spmv_handle_t spmv_build_permuted(int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col_idx,
                                           const void *vals, int dtype, int format,
                                           const spmv_format_params *params, int ordering, const int32_t *perm,
                                           void *stream);

/* perm (device int32[n]) = the handle's basis order, new -> old (the identity for a
 * handle built by spmv_build_from_csr).  Synchronises `stream`. */
SPMV_API int spmv_get_permutation(spmv_handle_t h, int32_t *perm, void *stream);

/*
 * Move a vector between the original basis and the handle's: direction 0 (into the
 * basis) dst[i] = src[perm[i]]; direction 1 (back) dst[perm[i]] = src[i].  src and dst
 * are device arrays of n values of the handle's type and must not overlap.  Asynchronous.
 */
SPMV_API int spmv_permute_vector(spmv_handle_t h, const void *src, void *dst, int direction, void *stream);

/*
 * None of the pages has a counterpart to this entry point: it reports the library's own
 * bounded device waits.  Synchronise `stream` and report whether an apply kernel of this
 * handle gave up a bounded wait on the device since the last report: SPMV_ERR_TIMEOUT (results of the
 * applies since then are invalid; the flag is cleared) or SPMV_OK.  Only the
 * bulk-staged apply (parameter `staged`) waits on the device, for its own bulk copies,
 * each wait bounded by about a second.  spmv_apply_host, spmv_apply_mapped and
 * spmv_apply_profiled make this check themselves.
 */
SPMV_API int spmv_device_status(spmv_handle_t h, void *stream);

/* Release every device buffer of the handle.  NULL is accepted and ignored. */
SPMV_API void spmv_destroy(spmv_handle_t h);

/* Status of the last failing call on this thread (SPMV_OK if none) and its message. */
SPMV_API int spmv_last_error(void);
SPMV_API const char *spmv_last_error_message(void);
/* Static description of a status code. */
SPMV_API const char *spmv_error_string(int status);

/*
 * Rebuild the CSR held by the handle, in the caller's row order and in the input's
 * in-row order: row_ptr int32[n+1], col_idx int32[nnz], vals[nnz] (device memory
 * owned by the caller).  Every format stores exactly the input entries, so the
 * result equals the build input array for array.  Synchronises `stream`.
 */
SPMV_API int spmv_to_csr(spmv_handle_t h, int32_t *row_ptr, int32_t *col_idx, void *vals, void *stream);

/*
 * Write a JSON object describing the handle (format, resolved parameters, padded
 * and allocated slots, long rows, spill size, kernels launched per apply, bytes
 * streamed per apply) into json[0..cap).  Returns SPMV_OK, or SPMV_ERR_INVALID_ARG
 * when cap is too small (the text is then truncated but NUL-terminated).
 */
SPMV_API int spmv_describe(spmv_handle_t h, char *json, size_t cap);

/*
 * Copy layout arrays of the sliced part (SELL, ELL-R or the HYB ELL part):
 *   perm       int32[n]: perm[p] = original row stored at sorted position p
 *              (the identity when the format keeps the natural order);
 *   slice_ptr  int64[n_slices + 1]: start of every slice in the slot arrays.
 * Either pointer may be NULL.  Sizes are in spmv_describe ("n_slices").  Returns
 * SPMV_ERR_UNSUPPORTED for a handle without a sliced part.  Synchronises `stream`.
 */
SPMV_API int spmv_get_layout(spmv_handle_t h, int32_t *perm, int64_t *slice_ptr, void *stream);

/*
 * Copy the slot arrays of the sliced part: col int32[slots] and val[slots] (value
 * type of the handle), slots as in spmv_describe ("slots").  Entry j of the row at
 * in-slice position q of a slice starting at slice_ptr[s] sits at
 *   slice_ptr[s] + j * stride + q                                   (column-major), or
 *   slice_ptr[s] + ((j / g) * stride + q) * g + j % g   (interleaved, g = row_threads,
 *                                                        "row_group_mode": 1),
 * stride = C for SELL and the leading dimension "ld" for ELLPACK-R / HYB-ELL.  Padding
 * slots hold column 0 and value 0.  Either pointer may be NULL (device memory owned
 * by the caller).  SPMV_ERR_UNSUPPORTED without a sliced part.  Synchronises `stream`.
 */
SPMV_API int spmv_get_slots(spmv_handle_t h, int32_t *col, void *val, void *stream);

/*
 * Measurement aid: the device's rates of gathers from x at random positions, the ceiling
 * of the matrices whose column indices have no locality.  The GPGPU spMVM paper's
 * code-balance model (performance-model section) charges x by its reuse factor; with
 * random columns nothing is reused and the x accesses are scattered.  An SM sends its
 * L1 misses to L2 as one request per 128-byte line (carrying the sectors of that line a
 * warp instruction needs), and two limits apply at once: requests per second and
 * sectors per second.  So the time of a product cannot fall below
 *   max(lines / rate(sectors_per_line = 1), sectors / rate(sectors_per_line = 4)),
 * counting, per warp instruction, the distinct lines and 32-byte sectors of x it reads,
 * however much HBM bandwidth the streamed matrix leaves unused.
 *   x        device array of n values of `dtype` (n < 2^31), only read.  Lines are
 *            counted from x, which should start on a 128-byte boundary (as memory from
 *            cudaMalloc does).
 *   sectors_per_line  1: every lane gathers a random element of its own (one request
 *            per gather); 2 or 4: groups of that many consecutive lanes read distinct
 *            32-byte sectors of one random 128-byte line of x (needs n >= 128 bytes of
 *            values).  Any other value is SPMV_ERR_INVALID_ARG.
 *   gathers  lane loads to perform (one sector each), rounded up to whole rounds of 8
 *            per thread of a full wave (2048 threads per SM); the count done is written
 *            to *gathers_done (host pointer, may be NULL).
 *   out_sum  device double: the sum of the gathered values is ADDED to it (so no load
 *            can be dropped); its value has no other meaning.
 * Positions come from a per-thread (per-group) linear congruential sequence mapped onto
 * [0, n) or onto the whole lines of x, so no index array is read.  One kernel launch on
 * `stream`; time it with events around the call.  Returns an spmv_status.
 */
SPMV_API int spmv_probe_gather(const void *x, int64_t n, int dtype, int sectors_per_line, int64_t gathers,
                               void *out_sum, void *stream, int64_t *gathers_done);

/*
 * y = A x computed directly from a CSR matrix in the caller's device memory, with
 * no device allocation at all (no handle, no cudaMalloc / cudaFree, no allocating
 * library call).  None of the pages has a counterpart to this entry point: it is
 * there for callers that cannot allocate device memory -- for example a program
 * that hands all device memory to its own pool at start-up and forbids other
 * allocations, or a time-critical loop that cannot afford the implicit device
 * synchronisation of cudaMalloc / cudaFree -- and therefore cannot build a handle.
 *
 * The computation is the load-balanced merge-path pass of the `merge` format (and of
 * HYB's CSR spill), applied to every row; y is overwritten.  Its only scratch (one partial sum per
 * 2048-item share of the work) sits in a fixed 768 KiB array inside this
 * library's device image, which every GPU that loads the library keeps until the
 * process exits.  Hence:
 *   - n + nnz must not exceed 134,217,728; larger matrices return SPMV_ERR_TOO_LARGE
 *     before anything runs;
 *   - all calls share that array: calls that overlap on the GPU (different streams,
 *     or different host threads) race on it and give wrong results; serialise them;
 *   - the first call on a device (and the first after a cudaDeviceReset) looks up the
 *     array's device address (and, with lazy module loading, makes the driver load the
 *     library's device code); make that first call before any stream capture;
 *   - the CSR is NOT validated (validation would need a device-to-host round trip):
 *     pass a matrix that spmv_build_from_csr would accept.
 * Arguments are as in spmv_build_from_csr plus x, y (device arrays of n values of
 * `dtype`) and `stream`.  Every array must be memory of the current device.  y is
 * written while other parts of the work still read x and the matrix, so a y that
 * overlaps x, row_ptr, col_idx or vals is refused with SPMV_ERR_INVALID_ARG (no
 * in-place product).  Asynchronous; returns an spmv_status.
 */
SPMV_API int spmv_csr_apply_noalloc(int64_t n, int64_t nnz, const int32_t *row_ptr, const int32_t *col_idx,
                                    const void *vals, int dtype, const void *x, void *y, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPMV_GB300_H */
