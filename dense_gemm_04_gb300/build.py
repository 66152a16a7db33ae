"""Build libphx.so (the CUDA library behind include/phx.h) in-tree with nvcc.

Every translation unit under csrc/ is compiled for sm_103a only, in parallel, then linked
with the CUDA runtime linked statically and a version script that exports nothing but the
phx_* C ABI.  The result lands in dense_gemm_04_gb300/_lib/libphx.so.  With --debug (or
build(debug=True)) the same sources are compiled with -DPHX_DEBUG=1, the kernels' index
checks on, into _lib/libphx_debug.so (objects in _build_debug/).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libphx.so")
ROOT = os.path.dirname(HERE)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libphx")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime() -> float:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh", ".inc", ".map"))]
    hs.append(os.path.join(ROOT, "include", "phx.h"))
    return max(os.path.getmtime(h) for h in hs)


def _paths(debug: bool):
    if debug:
        return os.path.join(HERE, "_build_debug"), os.path.join(OUT_DIR, "libphx_debug.so")
    return BUILD_DIR, LIB


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    build_dir, _ = _paths(debug)
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *(["-DPHX_DEBUG=1"] if debug else []), "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr[-6000:]}")
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link libphx.so (libphx_debug.so with debug) if any source is newer than
    it; return its path."""
    srcs = sources()
    build_dir, lib = _paths(debug)
    if not force and os.path.exists(lib):
        newest = max(max(os.path.getmtime(s) for s in srcs), _headers_mtime(),
                     os.path.getmtime(os.path.abspath(__file__)))
        if os.path.getmtime(lib) >= newest:
            return lib
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
           "-Xlinker", "--version-script=" + os.path.join(CSRC, "libphx.map"),
           "-Xlinker", "-Bsymbolic", "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of libphx.so failed:\n{r.stderr[-6000:]}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
