"""Build the in-tree CUDA library libfp8gemm.so for sm_103a with nvcc.

The library is a plain C ABI shared object (include/fp8gemm.h); the CUDA
runtime is linked statically, so loading it needs no GPU driver, and the
driver's tensor-map encoder is resolved at run time.  The translation units
compile in parallel (one nvcc process each) and are linked into one object.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libfp8gemm.so")
SOURCES = ["fp8gemm.cu", "swap.cu"]
HEADERS = ["gemm_kernel.cuh", "gemm_pair_kernel.cuh", "gemm_swap_kernel.cuh", "quantize_kernel.cuh", "ptx.cuh",
           "host_common.cuh", "swap.h"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON_FLAGS = ["-std=c++17", "-O3", "-lineinfo", *ARCH_FLAGS, "-Xcompiler", "-fPIC"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "fp8gemm.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if a source is newer than it; return its path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = f"tmp{os.getpid()}"
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, f"{os.path.splitext(src)[0]}.{tag}.o")
        cmd = [nvcc(), *COMMON_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append(subprocess.Popen(cmd))
        objs.append(obj)
    failed = [p.args for p in procs if p.wait() != 0]
    try:
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        tmp = LIB_PATH + f".{tag}"
        subprocess.run([nvcc(), *ARCH_FLAGS, "-shared", "-cudart", "static", *objs, "-o", tmp], check=True)
        os.replace(tmp, LIB_PATH)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
