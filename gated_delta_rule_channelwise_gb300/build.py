"""Builds libcgdr.so (the CUDA library behind include/cgdr.h) for sm_103a.

Every translation unit is compiled by nvcc in parallel, then linked into one
shared library next to this file.  No CMake; a rebuild happens only when a
source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcgdr.so")
# The debug build: the same sources with CGDR_DEBUG_CHECKS, whose kernels test every global
# access against the tensor's footprint and report a failed test as CGDR_ERR_BOUNDS instead of
# touching the memory (a stand-in for a memory checker on machines where none may run).
OBJDIR_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libcgdr_debug.so")
SOURCES = ["api.cu", "decode.cu", "prefill_simt.cu", "prefill_tc05.cu", "prefill_cluster.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcgdr")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Builds libcgdr.so (or, with debug=True, libcgdr_debug.so) when a source is newer."""
    lib, objdir = (LIB_DEBUG, OBJDIR_DEBUG) if debug else (LIB, OBJDIR)
    if debug:
        extra_flags = (*extra_flags, "-DCGDR_DEBUG_CHECKS")
    if not force and not is_stale(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False, verbose: bool = False) -> list:
    """Both libraries, built side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        futs = [ex.submit(build, force, verbose, (), d) for d in (False, True)]
        return [f.result() for f in futs]


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
