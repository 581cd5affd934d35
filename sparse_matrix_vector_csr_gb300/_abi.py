"""ctypes binding of ``libspmv_gb300.so`` (declared in ``include/spmv.h``).

Argument marshalling only: torch CUDA tensors become device pointers, numpy
arrays host pointers, torch streams ``cudaStream_t`` values.  Every step of the
computation runs in the CUDA library; if it is missing this module raises on
import instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import json
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspmv_gb300.so")

SPMV_F64, SPMV_F32 = 0, 1
FORMATS = {"auto": 0, "csr_vector": 1, "ell_r": 2, "sell": 3, "hyb": 4, "merge": 5}
STATUS = {
    0: "SPMV_OK", -1: "SPMV_ERR_INVALID_ARG", -2: "SPMV_ERR_BAD_CSR", -3: "SPMV_ERR_CUDA",
    -4: "SPMV_ERR_OOM", -5: "SPMV_ERR_TOO_LARGE", -6: "SPMV_ERR_UNSUPPORTED", -7: "SPMV_ERR_TIMEOUT",
}

#: every function the header declares (checked by the tests)
EXPORTS = (
    "spmv_default_params", "spmv_build_from_csr", "spmv_build_from_csr_ex", "spmv_apply",
    "spmv_apply_host", "spmv_apply_profiled", "spmv_destroy", "spmv_last_error",
    "spmv_last_error_message", "spmv_error_string", "spmv_to_csr", "spmv_describe", "spmv_get_layout",
    "spmv_csr_apply_noalloc", "spmv_apply_ex", "spmv_apply_multi", "spmv_cg", "spmv_get_slots",
    "spmv_build_permuted", "spmv_get_permutation", "spmv_permute_vector", "spmv_apply_mapped", "spmv_bicgstab",
    "spmv_gmres", "spmv_probe_gather", "spmv_device_status", "spmv_device_memory",
)

#: spmv_ordering codes
ORDERINGS = {"natural": 0, "row_length": 1, "rcm": 2, "user": 3}


class SpmvError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {message}")


class FormatParams(ctypes.Structure):
    _fields_ = [
        ("C", ctypes.c_int32),
        ("sigma", ctypes.c_int64),
        ("K", ctypes.c_int32),
        ("spill_csr", ctypes.c_int32),
        ("long_row_threshold", ctypes.c_int32),
        ("subwarp", ctypes.c_int32),
        ("row_threads", ctypes.c_int32),
        ("row_group_mode", ctypes.c_int32),
        ("x_policy", ctypes.c_int32),
        ("vector_loads", ctypes.c_int32),
        ("host_blocks", ctypes.c_int32),
        ("staged", ctypes.c_int32),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python sparse_matrix_vector_csr_gb300/_build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
    lib.spmv_default_params.argtypes = [ctypes.POINTER(FormatParams)]
    lib.spmv_default_params.restype = c_int
    lib.spmv_build_from_csr.argtypes = [i64, i64, vp, vp, vp, c_int, c_int]
    lib.spmv_build_from_csr.restype = vp
    lib.spmv_build_from_csr_ex.argtypes = [i64, i64, vp, vp, vp, c_int, c_int, ctypes.POINTER(FormatParams), vp]
    lib.spmv_build_from_csr_ex.restype = vp
    lib.spmv_apply.argtypes = [vp, vp, vp, vp]
    lib.spmv_apply.restype = c_int
    lib.spmv_apply_host.argtypes = [vp, vp, vp, vp]
    lib.spmv_apply_host.restype = c_int
    lib.spmv_apply_mapped.argtypes = [vp, vp, vp, vp]
    lib.spmv_apply_mapped.restype = c_int
    lib.spmv_apply_profiled.argtypes = [vp, vp, vp, vp, ctypes.POINTER(ctypes.c_float), c_int]
    lib.spmv_apply_profiled.restype = c_int
    lib.spmv_destroy.argtypes = [vp]
    lib.spmv_destroy.restype = None
    lib.spmv_last_error.argtypes = []
    lib.spmv_last_error.restype = c_int
    lib.spmv_last_error_message.argtypes = []
    lib.spmv_last_error_message.restype = ctypes.c_char_p
    lib.spmv_error_string.argtypes = [c_int]
    lib.spmv_error_string.restype = ctypes.c_char_p
    lib.spmv_to_csr.argtypes = [vp, vp, vp, vp, vp]
    lib.spmv_to_csr.restype = c_int
    lib.spmv_describe.argtypes = [vp, ctypes.c_char_p, ctypes.c_size_t]
    lib.spmv_describe.restype = c_int
    lib.spmv_get_layout.argtypes = [vp, vp, vp, vp]
    lib.spmv_get_layout.restype = c_int
    lib.spmv_get_slots.argtypes = [vp, vp, vp, vp]
    lib.spmv_get_slots.restype = c_int
    lib.spmv_csr_apply_noalloc.argtypes = [i64, i64, vp, vp, vp, c_int, vp, vp, vp]
    lib.spmv_csr_apply_noalloc.restype = c_int
    lib.spmv_probe_gather.argtypes = [vp, i64, c_int, c_int, i64, vp, vp, ctypes.POINTER(i64)]
    lib.spmv_probe_gather.restype = c_int
    lib.spmv_device_memory.argtypes = [ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.spmv_device_memory.restype = c_int
    lib.spmv_device_status.argtypes = [vp, vp]
    lib.spmv_device_status.restype = c_int
    f64 = ctypes.c_double
    lib.spmv_apply_ex.argtypes = [vp, f64, vp, f64, vp, vp]
    lib.spmv_apply_ex.restype = c_int
    lib.spmv_apply_multi.argtypes = [vp, i64, f64, vp, i64, f64, vp, i64, vp]
    lib.spmv_apply_multi.restype = c_int
    lib.spmv_cg.argtypes = [vp, vp, vp, f64, i32, vp, ctypes.POINTER(i32), ctypes.POINTER(f64)]
    lib.spmv_cg.restype = c_int
    lib.spmv_bicgstab.argtypes = lib.spmv_cg.argtypes
    lib.spmv_bicgstab.restype = c_int
    lib.spmv_gmres.argtypes = [vp, vp, vp, i32, f64, i32, vp, ctypes.POINTER(i32), ctypes.POINTER(f64)]
    lib.spmv_gmres.restype = c_int
    lib.spmv_build_permuted.argtypes = [i64, i64, vp, vp, vp, c_int, c_int, ctypes.POINTER(FormatParams), c_int, vp,
                                        vp]
    lib.spmv_build_permuted.restype = vp
    lib.spmv_get_permutation.argtypes = [vp, vp, vp]
    lib.spmv_get_permutation.restype = c_int
    lib.spmv_permute_vector.argtypes = [vp, vp, vp, c_int, vp]
    lib.spmv_permute_vector.restype = c_int
    del i32
    return lib


lib = _load()


# --------------------------------------------------------------------------- #
# marshalling helpers
# --------------------------------------------------------------------------- #


def _ptr(t):
    """Device pointer of a torch tensor, host pointer of a numpy array, or None."""
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        return t.data_ptr() or None
    if hasattr(t, "ctypes"):
        return t.ctypes.data or None
    return int(t)


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream or None
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream or None
    return int(stream) or None


def _raise_last(status: int | None = None):
    st = lib.spmv_last_error() if status is None else status
    msg = lib.spmv_last_error_message().decode(errors="replace")
    raise SpmvError(st, msg)


def _check(status: int) -> int:
    if status < 0:
        _raise_last(status)
    return status


def dtype_code(dtype) -> int:
    name = str(dtype)
    if name.endswith("float64") or name == "f64":
        return SPMV_F64
    if name.endswith("float32") or name == "f32":
        return SPMV_F32
    raise TypeError(f"unsupported value type {dtype}")


def make_params(C=-1, sigma=-1, K=-1, spill_csr=-1, long_row_threshold=-1, subwarp=-1, row_threads=-1,
                row_group_mode=-1, x_policy=-1, vector_loads=-1, host_blocks=-1, staged=-1) -> FormatParams:
    p = FormatParams()
    lib.spmv_default_params(ctypes.byref(p))
    p.C, p.sigma, p.K = int(C), int(sigma), int(K)
    p.spill_csr, p.long_row_threshold, p.subwarp = int(spill_csr), int(long_row_threshold), int(subwarp)
    p.row_threads, p.row_group_mode, p.x_policy = int(row_threads), int(row_group_mode), int(x_policy)
    p.vector_loads = int(vector_loads)
    p.host_blocks = int(host_blocks)
    p.staged = int(staged)
    return p


# --------------------------------------------------------------------------- #
# the C entry points, same names
# --------------------------------------------------------------------------- #


def spmv_default_params() -> FormatParams:
    p = FormatParams()
    _check(lib.spmv_default_params(ctypes.byref(p)))
    return p


def spmv_build_from_csr(n, nnz, row_ptr, col_idx, vals, dtype, fmt) -> int:
    h = lib.spmv_build_from_csr(int(n), int(nnz), _ptr(row_ptr), _ptr(col_idx), _ptr(vals),
                                int(dtype), int(FORMATS.get(fmt, fmt)))
    if not h:
        _raise_last()
    return h


def spmv_build_from_csr_ex(n, nnz, row_ptr, col_idx, vals, dtype, fmt, params=None, stream=None) -> int:
    p = params if isinstance(params, FormatParams) else make_params(**(params or {}))
    h = lib.spmv_build_from_csr_ex(int(n), int(nnz), _ptr(row_ptr), _ptr(col_idx), _ptr(vals), int(dtype),
                                   int(FORMATS.get(fmt, fmt)), ctypes.byref(p), _stream(stream))
    if not h:
        _raise_last()
    return h


def spmv_build_permuted(n, nnz, row_ptr, col_idx, vals, dtype, fmt, params=None, ordering="rcm", perm=None,
                        stream=None) -> int:
    """Handle for B = P A P^T in the given ordering (see spmv.h)."""
    p = params if isinstance(params, FormatParams) else make_params(**(params or {}))
    h = lib.spmv_build_permuted(int(n), int(nnz), _ptr(row_ptr), _ptr(col_idx), _ptr(vals), int(dtype),
                                int(FORMATS.get(fmt, fmt)), ctypes.byref(p), int(ORDERINGS.get(ordering, ordering)),
                                _ptr(perm), _stream(stream))
    if not h:
        _raise_last()
    return h


def spmv_get_permutation(h, perm, stream=None) -> None:
    _check(lib.spmv_get_permutation(h, _ptr(perm), _stream(stream)))


def spmv_permute_vector(h, src, dst, direction, stream=None) -> None:
    _check(lib.spmv_permute_vector(h, _ptr(src), _ptr(dst), int(direction), _stream(stream)))


def spmv_apply(h, x, y, stream=None) -> None:
    _check(lib.spmv_apply(h, _ptr(x), _ptr(y), _stream(stream)))


def spmv_apply_host(h, x_host, y_host, stream=None) -> None:
    _check(lib.spmv_apply_host(h, _ptr(x_host), _ptr(y_host), _stream(stream)))


def spmv_apply_mapped(h, x_host, y_host, stream=None) -> None:
    """y_host = A x_host, the kernels reading and writing page-locked host arrays directly."""
    _check(lib.spmv_apply_mapped(h, _ptr(x_host), _ptr(y_host), _stream(stream)))


def spmv_apply_profiled(h, x, y, stream=None, cap: int = 16) -> list:
    buf = (ctypes.c_float * cap)()
    k = _check(lib.spmv_apply_profiled(h, _ptr(x), _ptr(y), _stream(stream), buf, cap))
    return [float(buf[i]) for i in range(min(k, cap))]


def spmv_destroy(h) -> None:
    lib.spmv_destroy(h)


def spmv_last_error() -> int:
    return lib.spmv_last_error()


def spmv_last_error_message() -> str:
    return lib.spmv_last_error_message().decode(errors="replace")


def spmv_error_string(status: int) -> str:
    return lib.spmv_error_string(int(status)).decode()


def spmv_to_csr(h, row_ptr, col_idx, vals, stream=None) -> None:
    _check(lib.spmv_to_csr(h, _ptr(row_ptr), _ptr(col_idx), _ptr(vals), _stream(stream)))


def spmv_describe(h) -> dict:
    cap = 1 << 16
    buf = ctypes.create_string_buffer(cap)
    _check(lib.spmv_describe(h, buf, cap))
    return json.loads(buf.value.decode())


def spmv_get_layout(h, perm=None, slice_ptr=None, stream=None) -> None:
    _check(lib.spmv_get_layout(h, _ptr(perm), _ptr(slice_ptr), _stream(stream)))


def spmv_get_slots(h, col=None, val=None, stream=None) -> None:
    """Copy the sliced part's slot arrays into device tensors (see spmv.h)."""
    _check(lib.spmv_get_slots(h, _ptr(col), _ptr(val), _stream(stream)))


def spmv_csr_apply_noalloc(n, nnz, row_ptr, col_idx, vals, dtype, x, y, stream=None) -> None:
    """y = A x from a device CSR without any device allocation (see spmv.h)."""
    _check(lib.spmv_csr_apply_noalloc(int(n), int(nnz), _ptr(row_ptr), _ptr(col_idx), _ptr(vals), int(dtype),
                                      _ptr(x), _ptr(y), _stream(stream)))


def spmv_device_status(h, stream=None) -> None:
    """Synchronise the stream; raise SPMV_ERR_TIMEOUT if an apply kernel gave up a wait."""
    _check(lib.spmv_device_status(h, _stream(stream)))


def spmv_device_memory() -> tuple:
    """(live device allocations, their bytes) held by the library right now."""
    count, size = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib.spmv_device_memory(ctypes.byref(count), ctypes.byref(size)))
    return int(count.value), int(size.value)


def spmv_probe_gather(x, n, dtype, sectors_per_line, gathers, out_sum, stream=None) -> int:
    """Random gathers from x, `sectors_per_line` lanes to a random 128-byte line
    (measurement aid, see spmv.h); returns the lane loads launched."""
    done = ctypes.c_int64(0)
    _check(lib.spmv_probe_gather(_ptr(x), int(n), int(dtype), int(sectors_per_line), int(gathers), _ptr(out_sum),
                                 _stream(stream), ctypes.byref(done)))
    return int(done.value)


def spmv_apply_ex(h, alpha, x, beta, y, stream=None) -> None:
    """y = alpha * A x + beta * y (y not read when beta == 0)."""
    _check(lib.spmv_apply_ex(h, float(alpha), _ptr(x), float(beta), _ptr(y), _stream(stream)))


def spmv_apply_multi(h, k, alpha, X, ldx, beta, Y, ldy, stream=None) -> None:
    """Y = alpha * A X + beta * Y for k row-major right-hand sides."""
    _check(lib.spmv_apply_multi(h, int(k), float(alpha), _ptr(X), int(ldx), float(beta), _ptr(Y), int(ldy),
                                _stream(stream)))


def spmv_cg(h, b, x, rtol, max_iter, stream=None):
    """Conjugate gradients for A x = b (x holds the initial guess and receives the iterate).
    Returns (iterations, relative_residual)."""
    it = ctypes.c_int32(0)
    res = ctypes.c_double(0.0)
    _check(lib.spmv_cg(h, _ptr(b), _ptr(x), float(rtol), int(max_iter), _stream(stream), ctypes.byref(it),
                       ctypes.byref(res)))
    return int(it.value), float(res.value)


def spmv_bicgstab(h, b, x, rtol, max_iter, stream=None):
    """BiCGSTAB for A x = b (x holds the initial guess and receives the iterate).
    Returns (iterations, relative_residual)."""
    it = ctypes.c_int32(0)
    res = ctypes.c_double(0.0)
    _check(lib.spmv_bicgstab(h, _ptr(b), _ptr(x), float(rtol), int(max_iter), _stream(stream), ctypes.byref(it),
                             ctypes.byref(res)))
    return int(it.value), float(res.value)


def spmv_gmres(h, b, x, restart, rtol, max_iter, stream=None):
    """Restarted GMRES(restart) for A x = b (x holds the initial guess and receives the
    iterate).  Returns (Arnoldi steps, true relative residual)."""
    it = ctypes.c_int32(0)
    res = ctypes.c_double(0.0)
    _check(lib.spmv_gmres(h, _ptr(b), _ptr(x), int(restart), float(rtol), int(max_iter), _stream(stream),
                          ctypes.byref(it), ctypes.byref(res)))
    return int(it.value), float(res.value)
