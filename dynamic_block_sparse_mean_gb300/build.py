"""Build libbsa.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each csrc/*.cu is compiled to an object in parallel, then the objects are linked
into dynamic_block_sparse_mean_gb300/libbsa.so against the shared CUDA runtime.
``bounds_check=True`` builds the same sources with -DBSA_BOUNDS_CHECK=1 into
libbsa_bounds.so: every worklist / selection / block-table index a kernel is about
to use is range-checked on the device (BSA_ERR_INDEX_RANGE) instead of trusted.
The package loads that library when the environment sets BSA_BOUNDS_CHECK=1.
Run as ``python -m dynamic_block_sparse_mean_gb300.build [--force] [--verbose]
[--bounds-check]``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbsa.so")
LIB_BOUNDS = os.path.join(PKG, "libbsa_bounds.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                     "-Xcompiler", "-fPIC,-O3", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbsa.so")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    deps += glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, bounds_check: bool = False) -> str:
    """Compile every CUDA source and link libbsa.so (libbsa_bounds.so with
    bounds_check); returns its path."""
    lib = LIB_BOUNDS if bounds_check else LIB
    if not force and not _stale(lib):
        return lib
    objdir = os.path.join(BUILD, "bounds") if bounds_check else BUILD
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []
    if bounds_check:
        extra += ["-DBSA_BOUNDS_CHECK=1"]

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stderr}")
        return obj, res.stderr

    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp] + [o for o, _ in results]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
                bounds_check="--bounds-check" in sys.argv))
