"""In-tree build of the S3D8 CUDA library (nvcc, sm_103a only).

Each .cu file compiles to an object in parallel, then nvcc links one shared
library, ``_build/libs3d8.so``.  No cmake, no torch extension machinery: the
library exposes a plain C ABI (``include/s3d8.h``) that the ctypes binding in
this package loads.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libs3d8.so")
# The debug-checks variant: every kernel compiled with S3D8_DEBUG_CHECKS, whose
# in-kernel bounds checks record S3D8_ERR_BOUNDS instead of touching memory out
# of range.  Built on request only (build(debug=True)); the binding loads it when
# the environment variable S3D8_LIBRARY is "debug".
DEBUG_OUT = os.path.join(OUT, "debug")
DEBUG_LIB = os.path.join(OUT, "libs3d8_debug.so")
HEADER = os.path.join(ROOT, "include", "s3d8.h")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=false"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the S3D8 CUDA library cannot be built")
    return cand


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs_mtime() -> float:
    files = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files.append(HEADER)
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def up_to_date(lib: str = LIB) -> bool:
    return os.path.exists(lib) and os.path.getmtime(lib) >= _inputs_mtime()


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link ``libs3d8.so`` (or, with
    debug=True, ``libs3d8_debug.so`` with the in-kernel bounds checks)."""
    lib, out = (DEBUG_LIB, DEBUG_OUT) if debug else (LIB, OUT)
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(out, exist_ok=True)
    flags = NVCC_FLAGS + ARCH + list(extra_flags or []) + (["-DS3D8_DEBUG_CHECKS"] if debug else [])

    def compile_one(src):
        obj = os.path.join(out, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
