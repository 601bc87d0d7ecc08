"""Build ``libdc.so`` (the C-ABI library with the sm_103a kernels) in-tree.

Each ``csrc/*.cu`` is compiled on its own nvcc process (in parallel), then
linked into ``reduce_copy_rank_gb300/libdc.so`` with the CUDA runtime linked
statically, so the library needs nothing but the driver at run time.
Floating point: no fast-math, no flush-to-zero, no contraction.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdc.so")
# The bounds-checked build (-DDC_DEBUG_BOUNDS): every global access of every
# kernel is checked against its job's range first (include/dc.h,
# dc_bounds_checked); a test build, loaded instead of libdc.so when the
# environment variable DC_LIBRARY is "bounds".
OBJDIR_BOUNDS = os.path.join(PKG, "_build_bounds")
LIB_BOUNDS = os.path.join(PKG, "libdc_bounds.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                  "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=false",
                  "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libdc.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return sources() + hdrs + [os.path.join(INCLUDE, "dc.h"), os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, bounds: bool = False) -> str:
    """Compile and link libdc.so (bounds=True: the bounds-checked
    libdc_bounds.so) unless it is newer than every source."""
    lib, objdir = (LIB_BOUNDS, OBJDIR_BOUNDS) if bounds else (LIB, OBJDIR)
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(objdir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DDC_DEBUG_BOUNDS"] if bounds else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *NVFLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if ptxas_info or verbose:
            sys.stdout.write(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ptxas_info="--ptxas" in sys.argv, bounds="--bounds" in sys.argv))
