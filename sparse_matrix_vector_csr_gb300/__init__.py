"""GB300 (sm_103a) sparse matrix-vector product, y = A x, for CSR input.

The computation lives in the CUDA library ``libspmv_gb300.so`` (C interface in
``include/spmv.h``); this package is its Python binding.  ``_abi`` mirrors the C
entry points one to one; :class:`SpmvMatrix` wraps a handle for torch tensors.

    import torch, sparse_matrix_vector_csr_gb300 as spmv
    A = spmv.SpmvMatrix.from_csr(row_ptr, col_idx, vals)        # CUDA tensors
    y = A @ x                                                   # or A.apply(x, y)
"""
from __future__ import annotations

from . import _abi
from ._abi import (  # noqa: F401
    FORMATS,
    ORDERINGS,
    SpmvError,
    spmv_apply,
    spmv_apply_ex,
    spmv_apply_host,
    spmv_apply_mapped,
    spmv_apply_multi,
    spmv_apply_profiled,
    spmv_build_from_csr,
    spmv_build_from_csr_ex,
    spmv_cg,
    spmv_csr_apply_noalloc,
    spmv_default_params,
    spmv_describe,
    spmv_destroy,
    spmv_error_string,
    spmv_get_layout,
    spmv_get_permutation,
    spmv_build_permuted,
    spmv_bicgstab,
    spmv_gmres,
    spmv_permute_vector,
    spmv_probe_gather,
    spmv_device_memory,
    spmv_device_status,
    spmv_get_slots,
    spmv_last_error,
    spmv_last_error_message,
    spmv_to_csr,
)

__all__ = ["SpmvMatrix", "SpmvError", "FORMATS", "ORDERINGS"] + [n for n in _abi.EXPORTS]


class SpmvMatrix:
    """A square sparse matrix held by the CUDA library in one storage format."""

    def __init__(self, handle: int, n: int, nnz: int, dtype):
        self._h = handle
        self.n = n
        self.nnz = nnz
        self.dtype = dtype

    @classmethod
    def from_csr(cls, row_ptr, col_idx, vals, format: str = "auto", stream=None, ordering=None,
                 **params) -> "SpmvMatrix":
        """Build from device CSR tensors (int32 row_ptr/col_idx, float64/float32 vals).

        ``params``: C, sigma, K, spill_csr, long_row_threshold, subwarp, row_threads,
        row_group_mode, x_policy, vector_loads, host_blocks, staged (see spmv.h).  ``ordering`` ("natural", "row_length", "rcm", or an
        int32 CUDA tensor holding a permutation): build B = P A P^T and work in that
        permuted basis (see ``to_basis`` / ``from_basis``).
        """
        import torch

        for name, t in (("row_ptr", row_ptr), ("col_idx", col_idx), ("vals", vals)):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
                raise TypeError(f"{name} must be a contiguous CUDA tensor")
        if row_ptr.dtype != torch.int32 or col_idx.dtype != torch.int32:
            raise TypeError("row_ptr and col_idx must be int32")
        n = row_ptr.numel() - 1
        nnz = col_idx.numel()
        if vals.numel() != nnz:
            raise ValueError("vals and col_idx differ in length")
        code = _abi.dtype_code(vals.dtype)
        if ordering is None:
            h = spmv_build_from_csr_ex(n, nnz, row_ptr, col_idx, vals, code, format, params, stream)
        elif isinstance(ordering, torch.Tensor):
            if not (ordering.is_cuda and ordering.dtype == torch.int32 and ordering.numel() == n):
                raise TypeError("a user ordering must be an int32 CUDA tensor of n entries")
            h = spmv_build_permuted(n, nnz, row_ptr, col_idx, vals, code, format, params, "user",
                                    ordering.contiguous(), stream)
        else:
            h = spmv_build_permuted(n, nnz, row_ptr, col_idx, vals, code, format, params, ordering, None, stream)
        return cls(h, n, nnz, vals.dtype)

    def _check_vec(self, v, name):
        import torch

        if not (isinstance(v, torch.Tensor) and v.is_cuda and v.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous CUDA tensor")
        if v.dtype != self.dtype or v.numel() != self.n:
            raise ValueError(f"{name} must hold {self.n} values of {self.dtype}")

    def _check_host(self, v, name, writable=False):
        """A host array of n values of the handle's type, contiguous: a numpy array or a
        CPU tensor (the copies read and write exactly n values through its pointer)."""
        import numpy as np
        import torch

        if isinstance(v, torch.Tensor):
            ok = not v.is_cuda and v.is_contiguous() and v.dtype == self.dtype and v.numel() == self.n
        elif isinstance(v, np.ndarray):
            want = np.float64 if self.dtype == torch.float64 else np.float32
            ok = (v.flags.c_contiguous and v.dtype == want and v.size == self.n
                  and (v.flags.writeable or not writable))
        else:
            ok = False
        if not ok:
            raise ValueError(f"{name} must be a contiguous host array of {self.n} values of {self.dtype}"
                             + (", writable" if writable else ""))

    def apply(self, x, y=None, stream=None, alpha=1.0, beta=0.0):
        """y = alpha * A x + beta * y (default y = A x) on the current (or given) stream;
        allocates y when not given (then beta must be 0)."""
        import torch

        self._check_vec(x, "x")
        if y is None:
            if beta != 0.0:
                raise ValueError("beta != 0 needs an input y")
            y = torch.empty_like(x)
        self._check_vec(y, "y")
        if alpha == 1.0 and beta == 0.0:
            spmv_apply(self._h, x, y, stream)
        else:
            spmv_apply_ex(self._h, alpha, x, beta, y, stream)
        return y

    def apply_multi(self, X, Y=None, alpha=1.0, beta=0.0, stream=None):
        """Y = alpha * A X + beta * Y for the k columns of a row-major n x k CUDA tensor X."""
        import torch

        if not (isinstance(X, torch.Tensor) and X.is_cuda and X.dim() == 2 and X.shape[0] == self.n
                and X.stride(1) == 1 and X.dtype == self.dtype):
            raise TypeError(f"X must be an n x k CUDA tensor of {self.dtype} with unit column stride")
        if Y is None:
            if beta != 0.0:
                raise ValueError("beta != 0 needs an input Y")
            Y = torch.empty_like(X, memory_format=torch.contiguous_format)
        if not (Y.shape == X.shape and Y.stride(1) == 1 and Y.dtype == self.dtype and Y.is_cuda):
            raise TypeError("Y must match X in shape and type, with unit column stride")
        spmv_apply_multi(self._h, X.shape[1], alpha, X, X.stride(0), beta, Y, Y.stride(0), stream)
        return Y

    def cg(self, b, x=None, rtol=1e-8, max_iter=1000, stream=None):
        """Solve A x = b by conjugate gradients on the device (A symmetric positive definite).
        ``x`` is the initial guess (zeros when not given) and is updated in place.
        Returns (x, iterations, relative_residual)."""
        import torch

        self._check_vec(b, "b")
        if x is None:
            x = torch.zeros_like(b)
        self._check_vec(x, "x")
        it, res = spmv_cg(self._h, b, x, rtol, max_iter, stream)
        return x, it, res

    def bicgstab(self, b, x=None, rtol=1e-8, max_iter=1000, stream=None):
        """Solve A x = b by BiCGSTAB on the device (any nonsingular A for which it does not
        break down).  ``x`` is the initial guess (zeros when not given) and is updated in
        place.  Returns (x, iterations, relative_residual)."""
        import torch

        self._check_vec(b, "b")
        if x is None:
            x = torch.zeros_like(b)
        self._check_vec(x, "x")
        it, res = spmv_bicgstab(self._h, b, x, rtol, max_iter, stream)
        return x, it, res

    def gmres(self, b, x=None, restart=30, rtol=1e-8, max_iter=1000, stream=None):
        """Solve A x = b by restarted GMRES(restart) on the device (any nonsingular A).
        ``x`` is the initial guess (zeros when not given) and is updated in place.
        Returns (x, Arnoldi steps, true relative residual)."""
        import torch

        self._check_vec(b, "b")
        if x is None:
            x = torch.zeros_like(b)
        self._check_vec(x, "x")
        it, res = spmv_gmres(self._h, b, x, restart, rtol, max_iter, stream)
        return x, it, res

    __matmul__ = apply

    def apply_host(self, x_host, y_host=None, stream=None):
        """y = A x for numpy host arrays (pinned memory recommended), on the current (or
        given) stream; returns once y_host holds the result."""
        import numpy as np

        self._check_host(x_host, "x_host")
        if y_host is None:
            y_host = np.empty_like(x_host)
        self._check_host(y_host, "y_host", writable=True)
        spmv_apply_host(self._h, x_host, y_host, stream)
        return y_host

    def apply_mapped(self, x_host, y_host=None):
        """y = A x for page-locked host tensors (``tensor.pin_memory()``), read and written
        by the kernels through their device mapping, with no staging copies."""
        import torch

        for name, t in (("x_host", x_host), ("y_host", y_host)):
            if t is not None and not (isinstance(t, torch.Tensor) and t.is_pinned() and t.is_contiguous()):
                raise TypeError(f"{name} must be a contiguous page-locked host tensor")
        if y_host is None:
            y_host = torch.empty_like(x_host).pin_memory()
        self._check_host(x_host, "x_host")
        self._check_host(y_host, "y_host")
        spmv_apply_mapped(self._h, x_host, y_host)
        return y_host

    def apply_profiled(self, x, y, stream=None):
        """Per-kernel device times (ms) of one apply."""
        return spmv_apply_profiled(self._h, x, y, stream)

    def to_csr(self):
        """The stored CSR (original row order and in-row order) as CUDA tensors."""
        import torch

        dev = torch.device("cuda", torch.cuda.current_device())
        rp = torch.empty(self.n + 1, dtype=torch.int32, device=dev)
        ci = torch.empty(self.nnz, dtype=torch.int32, device=dev)
        vv = torch.empty(self.nnz, dtype=self.dtype, device=dev)
        spmv_to_csr(self._h, rp, ci, vv)
        return rp, ci, vv

    def describe(self) -> dict:
        return spmv_describe(self._h)

    def layout(self):
        """(perm, slice_ptr) of the sliced part as CUDA tensors."""
        import torch

        d = self.describe()
        dev = torch.device("cuda", torch.cuda.current_device())
        perm = torch.empty(self.n, dtype=torch.int32, device=dev)
        sp = torch.empty(d["n_slices"] + 1, dtype=torch.int64, device=dev)
        spmv_get_layout(self._h, perm, sp)
        return perm, sp

    def permutation(self):
        """The basis order as an int32 CUDA tensor (position -> original index)."""
        import torch

        perm = torch.empty(self.n, dtype=torch.int32, device=torch.device("cuda", torch.cuda.current_device()))
        spmv_get_permutation(self._h, perm)
        return perm

    def to_basis(self, v, out=None, stream=None):
        """A vector of the original basis in the handle's basis: out[i] = v[perm[i]]."""
        import torch

        self._check_vec(v, "v")
        out = torch.empty_like(v) if out is None else out
        self._check_vec(out, "out")
        spmv_permute_vector(self._h, v, out, 0, stream)
        return out

    def from_basis(self, v, out=None, stream=None):
        """A vector of the handle's basis back in the original one: out[perm[i]] = v[i]."""
        import torch

        self._check_vec(v, "v")
        out = torch.empty_like(v) if out is None else out
        self._check_vec(out, "out")
        spmv_permute_vector(self._h, v, out, 1, stream)
        return out

    def slots(self):
        """(col, val): the sliced part's slot arrays as CUDA tensors."""
        import torch

        d = self.describe()
        dev = torch.device("cuda", torch.cuda.current_device())
        col = torch.empty(d["slots"], dtype=torch.int32, device=dev)
        val = torch.empty(d["slots"], dtype=self.dtype, device=dev)
        spmv_get_slots(self._h, col, val)
        return col, val

    def close(self):
        if self._h:
            spmv_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
