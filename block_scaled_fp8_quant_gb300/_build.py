"""In-tree build of libbfq.so for sm_103a (nvcc, no cmake).

Each translation unit under csrc/ compiles in parallel to an object in
_build/, then nvcc links the shared library next to this file.  The flags
keep IEEE fp32 semantics (no fast-math): quantized codes depend on exact
fp32 division and rounding.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libbfq.so")
# The debug build: the same sources with BFQ_DEVICE_CHECKS, whose kernels
# check every computed global offset against its array's extent and latch
# BFQ_ERR_DEVICE_BOUNDS instead of accessing out of bounds.
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libbfq_debug.so")
SOURCES = ["bfq_api.cu", "quant_kernels.cu", "gemm_kernels.cu", "gemm_blockscaled.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbfq.so")


def _flags() -> list[str]:
    return ARCH + [
        "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
        "-I", os.path.join(ROOT, "include"), "-I", CSRC,
        "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills",
    ]


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "bfq.h"))
    files.append(os.path.abspath(__file__))
    return files


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD_DEBUG if debug else BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc()] + _flags() + (["-DBFQ_DEVICE_CHECKS"] if debug else []) + [
        "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        sys.stderr.write(res.stdout + res.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile (if stale) and return the path of libbfq.so (debug=True: of
    libbfq_debug.so, the build with device bounds checks)."""
    lib = LIB_DEBUG if debug else LIB
    newest = max(os.path.getmtime(f) for f in _deps())
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return lib
    os.makedirs(BUILD_DEBUG if debug else BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), SOURCES))
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))
