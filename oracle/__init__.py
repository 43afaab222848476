"""CPU oracle for the FP8 NT GEMM with fine-grained scaling -- TEST INFRASTRUCTURE.

This package is test infrastructure, not product code.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it.
It shares no code with the CUDA library under ``moe_grouped_gemm_nt_gb300``
and never imports it.

The arithmetic lives in ``oracle.c`` (plain C, FP64, OpenMP over rows); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
What is computed, and the page passages each function follows, are stated in
the header of ``oracle.c``:

* ``gemm_fp8_nt``            -- dense NT GEMM, page "DeepSeek开源周第三天DeepGEMM",
  sections "基本用法" and "两级精度累加与细粒度缩放".
* ``grouped_contiguous``     -- same page, "连续布局分组GEMM".
* ``grouped_masked``         -- same page, "掩码布局分组GEMM".
* ``k_grouped``              -- the same scaled NT product with the groups
  concatenated along K (one K segment per group, the weight-gradient step of
  MoE training; a reading of the same page's "DeepGEMM提供三种FP8GEMM实现",
  which names the grouped kinds by the training forward pass).
* ``decode`` / ``bf16_rne``  -- FP8 decoding and FP64 -> bfloat16 rounding.
* ``encode_fp8``             -- float32 -> FP8 code, nearest even, saturating.
* ``quantize_per_token``     -- 1x128 activation quantization producing the
  GEMM's LHS and its scales (same page, "基本用法"; page "企业官网建设流程全解析",
  section 5.2).
* ``*_at`` variants          -- the same definitions at sampled positions.

Every function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3 = 0
E5M2 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so with gcc (no CUDA involved)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", "-Wall", "-Wextra",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        LL = ctypes.c_longlong
        lib.oracle_decode.restype = ctypes.c_double
        lib.oracle_decode.argtypes = [I, I]
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_gemm_fp8_nt.restype = I
        lib.oracle_gemm_fp8_nt.argtypes = [P, I, P, P, I, P, I, I, I, P, P]
        lib.oracle_gemm_fp8_nt_at.restype = I
        lib.oracle_gemm_fp8_nt_at.argtypes = [P, I, P, P, I, P, I, I, I, LL, P, P, P, P]
        lib.oracle_grouped_contiguous.restype = I
        lib.oracle_grouped_contiguous.argtypes = [P, I, P, P, I, P, P, I, I, I, I, P, P]
        lib.oracle_grouped_contiguous_at.restype = I
        lib.oracle_grouped_contiguous_at.argtypes = [P, I, P, P, I, P, P, I, I, I, I, LL, P, P, P, P]
        lib.oracle_grouped_masked.restype = I
        lib.oracle_grouped_masked.argtypes = [P, I, P, P, I, P, P, I, I, I, I, P, P]
        lib.oracle_grouped_masked_at.restype = I
        lib.oracle_grouped_masked_at.argtypes = [P, I, P, P, I, P, P, I, I, I, I, LL, P, P, P, P, P]
        lib.oracle_k_grouped.restype = I
        lib.oracle_k_grouped.argtypes = [P, I, P, P, I, P, P, I, I, I, I, P, P]
        lib.oracle_k_grouped_at.restype = I
        lib.oracle_k_grouped_at.argtypes = [P, I, P, P, I, P, P, I, I, I, I, LL, P, P, P, P, P]
        lib.oracle_encode_fp8.restype = I
        lib.oracle_encode_fp8.argtypes = [I, ctypes.c_float]
        lib.oracle_quantize_per_token.restype = I
        lib.oracle_quantize_per_token.argtypes = [P, I, I, P, P, I, I]
        lib.oracle_num_threads.restype = I
        lib.oracle_num_threads.argtypes = []
        lib.oracle_set_num_threads.restype = None
        lib.oracle_set_num_threads.argtypes = [I]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _u8(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        a = a.view(np.uint8) if a.dtype.itemsize == 1 else a.astype(np.uint8)
    return a


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _i64(a):
    return np.ascontiguousarray(a, dtype=np.int64)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def decode(fmt: int, code: int) -> float:
    """Real value of one FP8 byte (fmt E4M3=0 or E5M2=1)."""
    return _load().oracle_decode(int(fmt), int(code))


def decode_table(fmt: int) -> np.ndarray:
    return np.array([decode(fmt, c) for c in range(256)], dtype=np.float64)


def bf16_rne(x: float) -> int:
    """bfloat16 bit pattern of x rounded to nearest, ties to even, from FP64."""
    return int(_load().oracle_bf16_rne(float(x)))


def encode_fp8(fmt: int, v: float) -> int:
    """FP8 code of the float32 value v: nearest, ties to even, saturating."""
    return int(_load().oracle_encode_fp8(int(fmt), float(np.float32(v))))


def quantize_per_token(x, fmt: int):
    """Per 1x128 row-group quantization of x [..., rows, k] (float32; bfloat16
    values widen exactly).  Returns (q uint8 [..., rows, k], s float32
    [..., rows, ceil(k/128)] row-major)."""
    x = _f32(x)
    *lead, rows, k = x.shape
    kb = _num_kb(k)
    nb = int(np.prod(lead)) if lead else 1
    flat = x.reshape(nb, rows, k)
    q = np.empty((flat.shape[0], rows, k), np.uint8)
    s = np.empty((flat.shape[0], rows, kb), np.float32)
    lib = _load()
    for b in range(flat.shape[0]):
        xb = np.ascontiguousarray(flat[b])
        if lib.oracle_quantize_per_token(_ptr(xb), k, int(fmt), _ptr(q[b]), _ptr(s[b]), rows, k) != 0:
            raise ValueError("oracle_quantize_per_token: bad argument")
    return q.reshape(*lead, rows, k), s.reshape(*lead, rows, kb)


def _num_kb(k):
    return (k + 127) // 128


def gemm_fp8_nt(A, a_fmt, sA, B, b_fmt, sB, want_f64=True):
    """Dense NT GEMM.  A [m,k] u8, sA [m,ceil(k/128)] f32, B [n,k] u8,
    sB [ceil(n/128),ceil(k/128)] f32.  Returns (D_bf16_bits uint16 [m,n], D_f64 or None)."""
    A, B, sA, sB = _u8(A), _u8(B), _f32(sA), _f32(sB)
    m, k = A.shape
    n = B.shape[0]
    assert B.shape == (n, k) and sA.shape == (m, _num_kb(k)), (A.shape, B.shape, sA.shape)
    assert sB.shape == ((n + 127) // 128, _num_kb(k)), sB.shape
    d16 = np.empty((m, n), np.uint16)
    d64 = np.empty((m, n), np.float64) if want_f64 else None
    rc = _load().oracle_gemm_fp8_nt(_ptr(A), a_fmt, _ptr(sA), _ptr(B), b_fmt, _ptr(sB),
                                    m, n, k, _ptr(d64), _ptr(d16))
    if rc != 0:
        raise ValueError(f"oracle_gemm_fp8_nt failed: {rc}")
    return d16, d64


def gemm_fp8_nt_at(A, a_fmt, sA, B, b_fmt, sB, rows, cols):
    """Dense NT GEMM at sampled (rows[i], cols[i]).  Returns (bf16 bits, f64)."""
    A, B, sA, sB = _u8(A), _u8(B), _f32(sA), _f32(sB)
    rows, cols = _i64(rows), _i64(cols)
    m, k = A.shape
    n = B.shape[0]
    d16 = np.empty(rows.shape, np.uint16)
    d64 = np.empty(rows.shape, np.float64)
    rc = _load().oracle_gemm_fp8_nt_at(_ptr(A), a_fmt, _ptr(sA), _ptr(B), b_fmt, _ptr(sB),
                                       m, n, k, rows.size, _ptr(rows), _ptr(cols),
                                       _ptr(d64), _ptr(d16))
    if rc != 0:
        raise ValueError(f"oracle_gemm_fp8_nt_at failed: {rc}")
    return d16, d64


def grouped_contiguous(A, a_fmt, sA, B, b_fmt, sB, m_indices, D16_init, want_f64=False):
    """Contiguous grouped GEMM.  B [G,n,k].  D16_init [M,n] uint16 is copied and
    only rows with a valid group id are overwritten."""
    A, B, sA, sB, mi = _u8(A), _u8(B), _f32(sA), _f32(sB), _i32(m_indices)
    M, k = A.shape
    G, n, _ = B.shape
    d16 = np.array(D16_init, dtype=np.uint16, copy=True, order="C")
    d64 = np.full((M, n), np.nan) if want_f64 else None
    rc = _load().oracle_grouped_contiguous(_ptr(A), a_fmt, _ptr(sA), _ptr(B), b_fmt, _ptr(sB),
                                           _ptr(mi), M, n, k, G, _ptr(d64), _ptr(d16))
    if rc != 0:
        raise ValueError(f"oracle_grouped_contiguous failed: {rc}")
    return d16, d64


def grouped_contiguous_at(A, a_fmt, sA, B, b_fmt, sB, m_indices, rows, cols):
    A, B, sA, sB, mi = _u8(A), _u8(B), _f32(sA), _f32(sB), _i32(m_indices)
    rows, cols = _i64(rows), _i64(cols)
    M, k = A.shape
    G, n, _ = B.shape
    d16 = np.empty(rows.shape, np.uint16)
    d64 = np.empty(rows.shape, np.float64)
    rc = _load().oracle_grouped_contiguous_at(_ptr(A), a_fmt, _ptr(sA), _ptr(B), b_fmt, _ptr(sB),
                                              _ptr(mi), M, n, k, G, rows.size, _ptr(rows),
                                              _ptr(cols), _ptr(d64), _ptr(d16))
    if rc != 0:
        raise ValueError(f"oracle_grouped_contiguous_at failed: {rc}")
    return d16, d64


def grouped_masked(A, a_fmt, sA, B, b_fmt, sB, masked_m, D16_init, want_f64=False):
    """Masked grouped GEMM.  A [G,M_cap,k], sA [G,M_cap,ceil(k/128)], B [G,n,k].
    D16_init [G,M_cap,n] is copied; rows r < masked_m[g] are overwritten."""
    A, B, sA, sB, mm = _u8(A), _u8(B), _f32(sA), _f32(sB), _i32(masked_m)
    G, M_cap, k = A.shape
    n = B.shape[1]
    d16 = np.array(D16_init, dtype=np.uint16, copy=True, order="C")
    d64 = np.full((G, M_cap, n), np.nan) if want_f64 else None
    rc = _load().oracle_grouped_masked(_ptr(A), a_fmt, _ptr(sA), _ptr(B), b_fmt, _ptr(sB),
                                       _ptr(mm), G, M_cap, n, k, _ptr(d64), _ptr(d16))
    if rc != 0:
        raise ValueError(f"oracle_grouped_masked failed: {rc}")
    return d16, d64


def grouped_masked_at(A, a_fmt, sA, B, b_fmt, sB, masked_m, groups, rows, cols):
    A, B, sA, sB, mm = _u8(A), _u8(B), _f32(sA), _f32(sB), _i32(masked_m)
    groups, rows, cols = _i64(groups), _i64(rows), _i64(cols)
    G, M_cap, k = A.shape
    n = B.shape[1]
    d16 = np.empty(rows.shape, np.uint16)
    d64 = np.empty(rows.shape, np.float64)
    rc = _load().oracle_grouped_masked_at(_ptr(A), a_fmt, _ptr(sA), _ptr(B), b_fmt, _ptr(sB),
                                          _ptr(mm), G, M_cap, n, k, rows.size, _ptr(groups),
                                          _ptr(rows), _ptr(cols), _ptr(d64), _ptr(d16))
    if rc != 0:
        raise ValueError(f"oracle_grouped_masked_at failed: {rc}")
    return d16, d64


def k_grouped(A, a_fmt, sA, B, b_fmt, sB, ks, want_f64=True):
    """K-grouped NT GEMM.  A [M,K] u8, sA [M,ceil(K/128)], B [N,K] u8,
    sB [ceil(N/128),ceil(K/128)], ks [G] int32 segment lengths (multiples of
    128, sum <= K).  Returns (D bf16 bits [G,M,N], D f64 [G,M,N] or None)."""
    A, B, sA, sB, ks = _u8(A), _u8(B), _f32(sA), _f32(sB), _i32(ks)
    M, K = A.shape
    N = B.shape[0]
    G = ks.size
    assert B.shape == (N, K) and sA.shape == (M, _num_kb(K)) and sB.shape == ((N + 127) // 128, _num_kb(K))
    d16 = np.empty((G, M, N), np.uint16)
    d64 = np.empty((G, M, N), np.float64) if want_f64 else None
    rc = _load().oracle_k_grouped(_ptr(A), a_fmt, _ptr(sA), _ptr(B), b_fmt, _ptr(sB), _ptr(ks), G, M, N, K,
                                  _ptr(d64), _ptr(d16))
    if rc != 0:
        raise ValueError(f"oracle_k_grouped failed: {rc}")
    return d16, d64


def k_grouped_at(A, a_fmt, sA, B, b_fmt, sB, ks, groups, rows, cols):
    """K-grouped NT GEMM at sampled (groups[i], rows[i], cols[i]).  Returns (bf16 bits, f64)."""
    A, B, sA, sB, ks = _u8(A), _u8(B), _f32(sA), _f32(sB), _i32(ks)
    groups, rows, cols = _i64(groups), _i64(rows), _i64(cols)
    M, K = A.shape
    N = B.shape[0]
    d16 = np.empty(rows.shape, np.uint16)
    d64 = np.empty(rows.shape, np.float64)
    rc = _load().oracle_k_grouped_at(_ptr(A), a_fmt, _ptr(sA), _ptr(B), b_fmt, _ptr(sB), _ptr(ks), ks.size, M, N,
                                     K, rows.size, _ptr(groups), _ptr(rows), _ptr(cols), _ptr(d64), _ptr(d16))
    if rc != 0:
        raise ValueError(f"oracle_k_grouped_at failed: {rc}")
    return d16, d64
