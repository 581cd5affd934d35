"""The C library builds, loads without a GPU, and exports every symbol include/spmv.h declares.

No compute call is made here: these run on machines without a GPU.
"""
import ctypes
import os
import re
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spmv.h")
PKG = os.path.join(ROOT, "sparse_matrix_vector_csr_gb300")


@pytest.fixture(scope="module")
def libpath():
    import __graft_entry__

    return __graft_entry__._build_module().build()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SPMV_API\s+[\w\s\*]*?\b(spmv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("spmv_build_from_csr", "spmv_apply", "spmv_destroy"):
        assert required in names
    assert len(names) >= 13


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_binding_covers_every_declared_symbol(libpath):
    import sparse_matrix_vector_csr_gb300 as spmv

    assert sorted(spmv._abi.EXPORTS) == declared_functions()
    for name in declared_functions():
        assert callable(getattr(spmv, name))


def test_exports_are_only_the_c_abi(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True).stdout
    text_syms = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(declared_functions()) <= text_syms
    assert all(s.startswith("spmv_") for s in text_syms), sorted(s for s in text_syms if not s.startswith("spmv_"))


def test_host_only_calls_without_gpu(libpath):
    import sparse_matrix_vector_csr_gb300 as spmv

    assert spmv.spmv_error_string(0) == "success"
    assert spmv.spmv_error_string(-2) == "malformed CSR matrix"
    p = spmv.spmv_default_params()
    assert (p.C, p.sigma, p.K, p.spill_csr, p.long_row_threshold, p.subwarp) == (-1, -1, -1, -1, -1, -1)
    # a NULL handle is rejected before any CUDA call
    with pytest.raises(spmv.SpmvError):
        spmv.spmv_apply(None, None, None, 0)
    assert spmv.spmv_last_error() == -1
    spmv.spmv_destroy(None)


def test_missing_library_fails_loudly(libpath):
    with tempfile.TemporaryDirectory() as d:
        dst = os.path.join(d, "sparse_matrix_vector_csr_gb300")
        shutil.copytree(PKG, dst, ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__"))
        code = "import sparse_matrix_vector_csr_gb300"
        res = subprocess.run([sys.executable, "-c", code], cwd=d, capture_output=True, text=True)
        assert res.returncode != 0 and "ImportError" in res.stderr


def _imports(path):
    mods = set()
    for dirpath, _, files in os.walk(path):
        for f in files:
            if f.endswith(".py"):
                src = open(os.path.join(dirpath, f)).read()
                mods |= set(re.findall(r"^\s*(?:from|import)\s+([\w\.]+)", src, re.M))
    return mods


def test_product_and_oracle_share_nothing():
    prod = _imports(PKG)
    assert not any(m.split(".")[0] in ("oracle", "workloads") for m in prod), prod
    orc = _imports(os.path.join(ROOT, "oracle"))
    assert not any(m.split(".")[0] == "sparse_matrix_vector_csr_gb300" for m in orc), orc
    gen = _imports(os.path.join(ROOT, "workloads"))
    assert not any(m.split(".")[0] in ("oracle", "sparse_matrix_vector_csr_gb300") for m in gen), gen
    # no C/CUDA source is shared either
    csrc = os.path.join(PKG, "csrc")
    for f in os.listdir(csrc):
        assert "oracle" not in open(os.path.join(csrc, f)).read().lower()


def test_params_struct_layout_matches_header(tmp_path):
    """The binding's spmv_format_params has the C struct's size and field offsets (gcc
    compiles the header and prints them), and spmv_default_params fills every field with
    -1 (automatic)."""
    import sparse_matrix_vector_csr_gb300 as spmv

    fields = [f for f, _ in spmv._abi.FormatParams._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "spmv.h"\nint main(void) {\n'
                   '  printf("size %zu\\n", sizeof(spmv_format_params));\n'
                   + "".join(f'  printf("{f} %zu\\n", offsetof(spmv_format_params, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(ln.split() for ln in subprocess.run([str(exe)], capture_output=True, text=True,
                                                    check=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(spmv._abi.FormatParams)
    for f in fields:
        assert int(got[f]) == getattr(spmv._abi.FormatParams, f).offset, f
    p = spmv.spmv_default_params()
    assert all(getattr(p, f) == -1 for f in fields), {f: getattr(p, f) for f in fields}


def test_size_and_argument_limits_refused_before_any_cuda_call(libpath):
    """n and nnz must lie in [0, 2^31), dtype must be F64 or F32, the probe takes 1, 2 or 4
    sectors per line, and the allocation-free call refuses sizes past its fixed scratch:
    each refusal comes before the library touches CUDA or dereferences a pointer, so
    host arrays stand in for device ones here and nothing runs on a device."""
    import numpy as np

    import sparse_matrix_vector_csr_gb300 as spmv

    dummy = np.zeros(4, np.int32)  # never read
    for n, nnz in ((1 << 31, 0), (4, 1 << 31), (-1, 0), (4, -1)):
        with pytest.raises(spmv.SpmvError) as ei:
            spmv.spmv_build_from_csr(n, nnz, dummy, dummy, dummy, 0, "auto")
        assert ei.value.status == -1, (n, nnz)
        with pytest.raises(spmv.SpmvError) as ei:
            spmv.spmv_csr_apply_noalloc(n, nnz, dummy, dummy, dummy, 0, dummy, dummy, 0)
        assert ei.value.status == -1, (n, nnz)
    with pytest.raises(spmv.SpmvError) as ei:
        spmv.spmv_build_from_csr(4, 0, dummy, None, None, 7, "auto")  # no such value type
    assert ei.value.status == -1
    with pytest.raises(spmv.SpmvError) as ei:
        spmv.spmv_build_from_csr(4, 0, dummy, None, None, 0, 9)  # no such format
    assert ei.value.status == -1
    # n + nnz above the allocation-free limit (134,217,728 path items)
    with pytest.raises(spmv.SpmvError) as ei:
        spmv.spmv_csr_apply_noalloc(100_000_000, 100_000_000, dummy, dummy, dummy, 0, dummy, dummy, 0)
    assert ei.value.status == -5
    spmv.spmv_csr_apply_noalloc(0, 0, None, None, None, 0, None, None, 0)  # n = 0: nothing to do
    for spl in (0, 3, 8):
        with pytest.raises(spmv.SpmvError) as ei:
            spmv.spmv_probe_gather(dummy, 4, 0, spl, 10, dummy, 0)
        assert ei.value.status == -1
    assert spmv.spmv_device_memory() == (0, 0)  # nothing allocated in this process
