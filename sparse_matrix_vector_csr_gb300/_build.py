"""Compile the CUDA library ``libspmv_gb300.so`` in-tree for sm_103a.

The translation units are compiled in parallel with nvcc and linked into a
shared library inside this package directory.  Run it as a script (importing
the package itself needs the built library)::

    python sparse_matrix_vector_csr_gb300/_build.py
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libspmv_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
SOURCES = ["api.cu", "build.cu", "sell.cu", "sellmm.cu", "vector.cu", "merge.cu", "vecops.cu", "noalloc.cu", "solve.cu", "sellg.cu", "order.cu", "sellv.cu", "probe.cu", "sellb.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    return os.path.join(home, "bin", "nvcc")


def common_flags() -> list[str]:
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                   "-I", INCLUDE, "-I", CSRC]


def _newer(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(OBJ_DIR, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src), os.path.join(CSRC, "spmv_internal.cuh"), os.path.join(CSRC, "device_util.cuh"),
            os.path.join(CSRC, "sell_common.cuh"), os.path.join(INCLUDE, "spmv.h")]
    if _newer(obj, deps):
        return obj
    cmd = [nvcc_path()] + common_flags() + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    if res.stderr.strip():
        sys.stderr.write(res.stderr)
    return obj


def build(verbose_ptxas: bool = False, force: bool = False) -> str:
    """Build (or reuse an up-to-date) ``libspmv_gb300.so``; returns its path."""
    os.makedirs(OBJ_DIR, exist_ok=True)
    if force:
        for f in os.listdir(OBJ_DIR):
            os.remove(os.path.join(OBJ_DIR, f))
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    if not _newer(LIB_PATH, objs):
        cmd = [nvcc_path()] + ARCH + ["-shared", "-cudart", "static", "-o", LIB_PATH] + objs
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv, force="--force" in sys.argv))
