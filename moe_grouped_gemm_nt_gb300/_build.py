"""Build the in-tree CUDA libraries for sm_103a with nvcc.

libfp8gemm.so is the library; libfp8gemm_debug.so is the same sources compiled
with FG_DEBUG: device-side checks of every TMA box, ring index and TMEM column
(a failed check records FG_ERR_DEVICE_CHECK and skips the access) and the
shallowest pipelines (one operand stage), for bisecting a race.  Both are plain
C ABI shared objects (include/fp8gemm.h); the CUDA runtime is linked
statically, so loading one needs no GPU driver, and the driver's tensor-map
encoder is resolved at run time.  All translation units compile in parallel
(one nvcc process each) and each library is linked into one object.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libfp8gemm.so")
DEBUG_LIB_PATH = os.path.join(BUILD_DIR, "libfp8gemm_debug.so")
VARIANTS = {LIB_PATH: [], DEBUG_LIB_PATH: ["-DFG_DEBUG"]}
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


def _stale(lib_path: str) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "fp8gemm.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def _build(lib_paths, force: bool, verbose: bool) -> None:
    todo = [p for p in lib_paths if force or _stale(p)]
    if not todo:
        return
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = f"tmp{os.getpid()}"
    jobs = []  # (library, objects, processes)
    for lib_path in todo:
        stem = os.path.splitext(os.path.basename(lib_path))[0]
        objs, procs = [], []
        for src in SOURCES:
            obj = os.path.join(BUILD_DIR, f"{stem}.{os.path.splitext(src)[0]}.{tag}.o")
            cmd = [nvcc(), *COMMON_FLAGS, *VARIANTS[lib_path], "-I", os.path.join(ROOT, "include"), "-c",
                   os.path.join(CSRC, src), "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append(subprocess.Popen(cmd))
            objs.append(obj)
        jobs.append((lib_path, objs, procs))
    try:
        failed = [p.args for _, _, procs in jobs for p in procs if p.wait() != 0]
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        for lib_path, objs, _ in jobs:
            tmp = lib_path + f".{tag}"
            subprocess.run([nvcc(), *ARCH_FLAGS, "-shared", "-cudart", "static", *objs, "-o", tmp], check=True)
            os.replace(tmp, lib_path)
    finally:
        for _, objs, procs in jobs:
            for p in procs:
                p.wait()
            for o in objs:
                if os.path.exists(o):
                    os.remove(o)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile the library (debug: the FG_DEBUG build) if a source is newer
    than it; return its path."""
    path = DEBUG_LIB_PATH if debug else LIB_PATH
    _build([path], force, verbose)
    return path


def build_all(force: bool = False, verbose: bool = False) -> None:
    """Compile both libraries, all translation units in parallel."""
    _build(list(VARIANTS), force, verbose)


if __name__ == "__main__":
    build_all(force=True, verbose=True)
    print(LIB_PATH, DEBUG_LIB_PATH)
