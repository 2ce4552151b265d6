"""Build libqmlp.so (in-tree) with nvcc for sm_103a.

Each .cu translation unit is compiled in parallel, then linked into one
shared library under weight_quantized_swiglu_gb300/lib/. The CUDA runtime is
linked statically so the library depends only on the driver.

build(bounds=True) builds the same sources with -DQMLP_DEBUG_BOUNDS into
lib/libqmlp_bounds.so: every kernel then checks the indices of its computed
global accesses and records the first bad one instead of making it (see
qmlp_debug_bounds in include/qmlp.h). Tests load it in a process of its own.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libqmlp.so")
LIB_BOUNDS = os.path.join(LIBDIR, "libqmlp_bounds.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqmlp.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), bounds: bool = False) -> str:
    lib = LIB_BOUNDS if bounds else LIB
    if not force and up_to_date(lib):
        return lib
    objdir = os.path.join(LIBDIR, "obj_bounds" if bounds else "obj")
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                    "--expt-relaxed-constexpr"] + list(extra_flags)
    if bounds:
        flags += ["-DQMLP_DEBUG_BOUNDS"]
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [cc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose:
        for _, err in results:
            sys.stderr.write(err)
    tmp = lib + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results] + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, bounds="--bounds" in sys.argv))
