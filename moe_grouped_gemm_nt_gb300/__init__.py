"""FP8 NT GEMM with fine-grained scaling for GB300 (sm_103a): dense and MoE grouped.

A thin Python binding of the C ABI in ``include/fp8gemm.h``: the functions
below carry the same names as the C entry points, check and marshal torch
tensors (device pointers, sizes, the current CUDA stream) and call the
library through ctypes.  Every step of the computation runs in the library's
CUDA kernels; there is no other implementation to fall back to, and a
missing or unloadable library raises.

Layouts (see the header for the full contract):
  A   [m, k] (masked: [G, M_cap, k]) float8_e4m3fn / float8_e5m2 / uint8
  sA  MN-major [ceil(k/128), ld] (masked: [G, ceil(k/128), ld]) float32
  B   [n, k] (grouped: [G, n, k])
  sB  [ceil(n/128), ceil(k/128)] (grouped: [G, ...]) float32
  D   [m, n] (masked: [G, M_cap, n]) bfloat16; float32 for the *_f32out calls
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

E4M3 = 0
E5M2 = 1

FG_OK = 0
STATUS_NAMES = {0: "FG_OK", 1: "FG_ERR_INVALID_ARG", 2: "FG_ERR_MISALIGNED", 3: "FG_ERR_UNSUPPORTED",
                4: "FG_ERR_CUDA", 5: "FG_ERR_TIMEOUT", 6: "FG_ERR_DEVICE_CHECK"}

_lock = threading.Lock()
_libs = {}  # library path -> loaded handle
_use_debug = False

# exported symbols and their ctypes signatures (kept in step with include/fp8gemm.h)
_P, _I, _U32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32
SIGNATURES = {
    "fg_gemm_fp8_nt": (_I, [_P, _I, _P, _I, _P, _I, _P, _P, _I, _I, _I, _P]),
    "fg_grouped_gemm_fp8_contiguous": (_I, [_P, _I, _P, _I, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P]),
    "fg_grouped_gemm_fp8_masked": (_I, [_P, _I, _P, _I, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P]),
    "fg_gemm_fp8_nt_f32out": (_I, [_P, _I, _P, _I, _P, _I, _P, _P, _I, _I, _I, _P]),
    "fg_grouped_gemm_fp8_contiguous_f32out": (_I, [_P, _I, _P, _I, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P]),
    "fg_grouped_gemm_fp8_masked_f32out": (_I, [_P, _I, _P, _I, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P]),
    "fg_k_grouped_gemm_fp8_nt": (_I, [_P, _I, _P, _I, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P]),
    "fg_k_grouped_gemm_fp8_nt_f32out": (_I, [_P, _I, _P, _I, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P]),
    "fg_scales_a_to_mn_major": (_I, [_P, _P, _I, _I, _I, _I, _P]),
    "fg_scales_a_ld": (_I, [_I]),
    "fg_quantize_fp8_per_token": (_I, [_P, _I, _I, _P, _P, _I, _P, _I, _I, _I, _P]),
    "fg_quantize_fp8_per_token_f32in": (_I, [_P, _I, _I, _P, _P, _I, _P, _I, _I, _I, _P]),
    "fg_get_device_status": (_I, [_P, ctypes.POINTER(_U32)]),
    "fg_set_num_sms": (_I, [_I]),
    "fg_set_watchdog_ms": (_I, [_U32]),
    "fg_set_config_override": (_I, [_I, _I]),
    "fg_set_programmatic_launch": (_I, [_I]),
    "fg_query_dense_plan": (_I, [_I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "fg_query_dense_plan_ex": (_I, [_I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "fg_set_pair_mode": (_I, [_I]),
    "fg_set_swap_mode": (_I, [_I]),
    "fg_query_plan": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_I)]),
    "fg_status_string": (ctypes.c_char_p, [_I]),
    "fg_version": (_I, []),
    "fg_debug_skip_producer_iteration": (_I, [_I]),
    "fg_debug_set_pair_defer": (_I, [_I]),
    "fg_debug_bad_coordinate": (_I, [_I]),
    "fg_debug_build": (_I, []),
}


class FGError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


def library_path(debug: bool = False) -> str:
    return _build.DEBUG_LIB_PATH if debug else _build.LIB_PATH


def lib(debug=None):
    """The loaded C library (built in-tree on first use if missing): the one
    `use_debug_library` selected, or the one `debug` names."""
    with _lock:
        dbg = _use_debug if debug is None else bool(debug)
        path = library_path(dbg)
        h = _libs.get(path)
        if h is None:
            if os.environ.get("FG_NO_AUTOBUILD") != "1":
                _build.build(debug=dbg)
            h = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(h, name)
                f.restype = res
                f.argtypes = args
            _libs[path] = h
        return h


def use_debug_library(on: bool) -> None:
    """Route later calls of this module to the debug build (libfp8gemm_debug.so:
    FG_DEBUG device-side checks of every TMA box, ring index and TMEM column,
    single-stage pipelines) or back to the library.  Process-wide; the two
    libraries keep separate knobs and status words.  For bisecting a
    suspected race or an out-of-bounds access, not for speed."""
    global _use_debug
    with _lock:
        _use_debug = bool(on)


def _check(name, st):
    if st != FG_OK:
        raise FGError(name, st)


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _common_device(tensors, stream=None):
    """The one CUDA device that every operand of a call lives on.

    The library launches on the calling thread's current device, so operands on
    another device (or spread over several) would be handed to kernels of the
    wrong GPU: raise instead.  A torch stream must belong to that device too; a
    raw stream handle (an int) cannot be checked and is taken as given."""
    dev = None
    for name, t in tensors:
        if t is None:
            continue
        d = t.device
        if dev is None:
            dev = d
        elif d != dev:
            raise ValueError(f"{name} is on {d}, but the other operands are on {dev}")
    if dev is not None and stream is not None and hasattr(stream, "device") and stream.device != dev:
        raise ValueError(f"stream belongs to {stream.device}, but the operands are on {dev}")
    return dev


def _launch(name, tensors, stream, *args):
    """Call the C entry point `name` with `args` (the stream handle appended),
    on the device of `tensors`: when that is not the current device, it is made
    current for the duration of the call."""
    dev = _common_device(tensors, stream)
    f = getattr(lib(), name)
    if dev is not None and dev.index is not None and dev.index != torch.cuda.current_device():
        with torch.cuda.device(dev):
            s = _stream_ptr(stream if stream is not None else torch.cuda.current_stream(dev))
            st = f(*args, s)
    else:
        st = f(*args, _stream_ptr(stream))
    _check(name, st)


def _fmt_of(t, fmt):
    if fmt is not None:
        return int(fmt)
    if t.dtype == torch.float8_e4m3fn or t.dtype == torch.uint8:
        return E4M3
    if t.dtype == torch.float8_e5m2:
        return E5M2
    raise TypeError(f"FP8 operand must be float8_e4m3fn, float8_e5m2 or uint8, got {t.dtype}")


def _need(t, name, dtypes, dim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_FP8 = (torch.float8_e4m3fn, torch.float8_e5m2, torch.uint8)
_F32 = (torch.float32,)
_BF16 = (torch.bfloat16,)
_I32 = (torch.int32,)


def _cdiv(a, b):
    return (a + b - 1) // b


def fg_gemm_fp8_nt(A, sA, B, sB, D, *, a_fmt=None, b_fmt=None, stream=None):
    """Dense D[m,n] = A[m,k] . B[n,k]^T with 1x128 / 128x128 FP32 scales, BF16 out."""
    return _dense("fg_gemm_fp8_nt", _BF16, A, sA, B, sB, D, a_fmt, b_fmt, stream)


def fg_gemm_fp8_nt_f32out(A, sA, B, sB, D, *, a_fmt=None, b_fmt=None, stream=None):
    """fg_gemm_fp8_nt with an FP32 D (the accumulator before BF16 rounding)."""
    return _dense("fg_gemm_fp8_nt_f32out", _F32, A, sA, B, sB, D, a_fmt, b_fmt, stream)


def _dense(name, d_dtypes, A, sA, B, sB, D, a_fmt, b_fmt, stream):
    _need(A, "A", _FP8, 2), _need(B, "B", _FP8, 2), _need(sA, "sA", _F32, 2)
    _need(sB, "sB", _F32, 2), _need(D, "D", d_dtypes, 2)
    m, k = A.shape
    n = B.shape[0]
    if B.shape[1] != k or tuple(D.shape) != (m, n):
        raise ValueError(f"shape mismatch A{tuple(A.shape)} B{tuple(B.shape)} D{tuple(D.shape)}")
    if sA.shape[0] != _cdiv(k, 128) or tuple(sB.shape) != (_cdiv(n, 128), _cdiv(k, 128)):
        raise ValueError(f"scale shapes sA{tuple(sA.shape)} sB{tuple(sB.shape)} do not fit m={m} n={n} k={k}")
    _launch(name, (("A", A), ("sA", sA), ("B", B), ("sB", sB), ("D", D)), stream,
            A.data_ptr(), _fmt_of(A, a_fmt), sA.data_ptr(), sA.shape[1], B.data_ptr(), _fmt_of(B, b_fmt),
            sB.data_ptr(), D.data_ptr(), m, n, k)
    return D


def fg_grouped_gemm_fp8_contiguous(A, sA, B, sB, D, m_indices, *, a_fmt=None, b_fmt=None, stream=None):
    """Contiguous layout: row r of A multiplies B[m_indices[r]]; rows with -1 stay untouched."""
    return _contiguous("fg_grouped_gemm_fp8_contiguous", _BF16, A, sA, B, sB, D, m_indices, a_fmt, b_fmt, stream)


def fg_grouped_gemm_fp8_contiguous_f32out(A, sA, B, sB, D, m_indices, *, a_fmt=None, b_fmt=None, stream=None):
    """fg_grouped_gemm_fp8_contiguous with an FP32 D."""
    return _contiguous("fg_grouped_gemm_fp8_contiguous_f32out", _F32, A, sA, B, sB, D, m_indices, a_fmt, b_fmt,
                       stream)


def _contiguous(name, d_dtypes, A, sA, B, sB, D, m_indices, a_fmt, b_fmt, stream):
    _need(A, "A", _FP8, 2), _need(B, "B", _FP8, 3), _need(sA, "sA", _F32, 2)
    _need(sB, "sB", _F32, 3), _need(D, "D", d_dtypes, 2), _need(m_indices, "m_indices", _I32, 1)
    M, k = A.shape
    G, n, kb_ = B.shape
    if kb_ != k or tuple(D.shape) != (M, n) or m_indices.shape[0] != M:
        raise ValueError("shape mismatch")
    if sA.shape[0] != _cdiv(k, 128) or tuple(sB.shape) != (G, _cdiv(n, 128), _cdiv(k, 128)):
        raise ValueError("scale shapes do not fit")
    _launch(name, (("A", A), ("sA", sA), ("B", B), ("sB", sB), ("D", D), ("m_indices", m_indices)), stream,
            A.data_ptr(), _fmt_of(A, a_fmt), sA.data_ptr(), sA.shape[1], B.data_ptr(), _fmt_of(B, b_fmt),
            sB.data_ptr(), D.data_ptr(), m_indices.data_ptr(), M, n, k, G)
    return D


def fg_grouped_gemm_fp8_masked(A, sA, B, sB, D, masked_m, *, a_fmt=None, b_fmt=None, stream=None):
    """Masked layout: rows r < masked_m[g] of group g are written; the rest stay untouched."""
    return _masked("fg_grouped_gemm_fp8_masked", _BF16, A, sA, B, sB, D, masked_m, a_fmt, b_fmt, stream)


def fg_grouped_gemm_fp8_masked_f32out(A, sA, B, sB, D, masked_m, *, a_fmt=None, b_fmt=None, stream=None):
    """fg_grouped_gemm_fp8_masked with an FP32 D."""
    return _masked("fg_grouped_gemm_fp8_masked_f32out", _F32, A, sA, B, sB, D, masked_m, a_fmt, b_fmt, stream)


def _masked(name, d_dtypes, A, sA, B, sB, D, masked_m, a_fmt, b_fmt, stream):
    _need(A, "A", _FP8, 3), _need(B, "B", _FP8, 3), _need(sA, "sA", _F32, 3)
    _need(sB, "sB", _F32, 3), _need(D, "D", d_dtypes, 3), _need(masked_m, "masked_m", _I32, 1)
    G, M_cap, k = A.shape
    Gb, n, kb_ = B.shape
    if Gb != G or kb_ != k or tuple(D.shape) != (G, M_cap, n) or masked_m.shape[0] != G:
        raise ValueError("shape mismatch")
    if tuple(sA.shape[:2]) != (G, _cdiv(k, 128)) or tuple(sB.shape) != (G, _cdiv(n, 128), _cdiv(k, 128)):
        raise ValueError("scale shapes do not fit")
    _launch(name, (("A", A), ("sA", sA), ("B", B), ("sB", sB), ("D", D), ("masked_m", masked_m)), stream,
            A.data_ptr(), _fmt_of(A, a_fmt), sA.data_ptr(), sA.shape[2], B.data_ptr(), _fmt_of(B, b_fmt),
            sB.data_ptr(), D.data_ptr(), masked_m.data_ptr(), G, M_cap, n, k)
    return D


def fg_k_grouped_gemm_fp8_nt(A, sA, B, sB, D, k_sizes, *, a_fmt=None, b_fmt=None, stream=None):
    """K-grouped layout: D[g] = A[:, seg_g] . B[:, seg_g]^T with the fine-grained
    scales, one 128-aligned K segment per group (k_sizes [G] int32 on the device).
    A [M, K], sA MN-major [ceil(K/128), ld], B [N, K], sB [ceil(N/128), ceil(K/128)],
    D [G, M, N] bfloat16."""
    return _k_grouped("fg_k_grouped_gemm_fp8_nt", _BF16, A, sA, B, sB, D, k_sizes, a_fmt, b_fmt, stream)


def fg_k_grouped_gemm_fp8_nt_f32out(A, sA, B, sB, D, k_sizes, *, a_fmt=None, b_fmt=None, stream=None):
    """fg_k_grouped_gemm_fp8_nt with an FP32 D [G, M, N]."""
    return _k_grouped("fg_k_grouped_gemm_fp8_nt_f32out", _F32, A, sA, B, sB, D, k_sizes, a_fmt, b_fmt, stream)


def _k_grouped(name, d_dtypes, A, sA, B, sB, D, k_sizes, a_fmt, b_fmt, stream):
    _need(A, "A", _FP8, 2), _need(B, "B", _FP8, 2), _need(sA, "sA", _F32, 2)
    _need(sB, "sB", _F32, 2), _need(D, "D", d_dtypes, 3), _need(k_sizes, "k_sizes", _I32, 1)
    M, K = A.shape
    N = B.shape[0]
    G = k_sizes.shape[0]
    if B.shape[1] != K or tuple(D.shape) != (G, M, N):
        raise ValueError(f"shape mismatch A{tuple(A.shape)} B{tuple(B.shape)} D{tuple(D.shape)} G={G}")
    if sA.shape[0] != _cdiv(K, 128) or tuple(sB.shape) != (_cdiv(N, 128), _cdiv(K, 128)):
        raise ValueError("scale shapes do not fit")
    _launch(name, (("A", A), ("sA", sA), ("B", B), ("sB", sB), ("D", D), ("k_sizes", k_sizes)), stream,
            A.data_ptr(), _fmt_of(A, a_fmt), sA.data_ptr(), sA.shape[1], B.data_ptr(), _fmt_of(B, b_fmt),
            sB.data_ptr(), D.data_ptr(), k_sizes.data_ptr(), G, M, N, K)
    return D


def fg_scales_a_ld(rows: int) -> int:
    return lib().fg_scales_a_ld(int(rows))


def fg_scales_a_to_mn_major(src, dst=None, *, stream=None):
    """Row-major [.., rows, kb] FP32 scales -> MN-major [.., kb, ld] (ld = rows rounded up to 4)."""
    _need(src, "src", _F32, src.dim())
    if src.dim() not in (2, 3):
        raise ValueError("src must be [rows, kb] or [batches, rows, kb]")
    batches = 1 if src.dim() == 2 else src.shape[0]
    rows, kb = src.shape[-2], src.shape[-1]
    ld = fg_scales_a_ld(rows)
    shape = (kb, ld) if src.dim() == 2 else (batches, kb, ld)
    if dst is None:
        dst = torch.empty(shape, dtype=torch.float32, device=src.device)
    else:
        _need(dst, "dst", _F32, src.dim())
        if tuple(dst.shape[:-1]) != shape[:-1] or dst.shape[-1] < rows:
            raise ValueError("dst shape does not fit")
        ld = dst.shape[-1]
    _launch("fg_scales_a_to_mn_major", (("src", src), ("dst", dst)), stream,
            src.data_ptr(), dst.data_ptr(), batches, rows, kb, ld)
    return dst


def fg_quantize_fp8_per_token(X, A=None, sA=None, *, fmt=E4M3, masked_m=None, stream=None):
    """Per-token (1x128) FP8 quantization of BF16 or FP32 activations X
    [rows, k] or [batches, rows, k] into A (same shape, FP8) and MN-major sA
    [.., kb, ld] (FP32 X: fg_quantize_fp8_per_token_f32in).

    X may be a column slice of a wider matrix (last stride 1, rows ld_x apart,
    batches rows * ld_x apart).  A and sA are allocated when not given (sA with
    ld = fg_scales_a_ld(rows); its padding entries are left unwritten).  With
    masked_m ([batches] int32 on the device) rows r >= masked_m[b] are left
    untouched.  Returns (A, sA)."""
    if not isinstance(X, torch.Tensor) or not X.is_cuda or X.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("X must be a CUDA bfloat16 or float32 tensor")
    if X.dim() not in (2, 3):
        raise ValueError("X must be [rows, k] or [batches, rows, k]")
    batches = 1 if X.dim() == 2 else X.shape[0]
    rows, k = X.shape[-2], X.shape[-1]
    if rows > 1:
        ld_x = X.stride(-2)
    else:  # one row per batch: the batch stride is the row pitch
        ld_x = X.stride(0) if X.dim() == 3 and batches > 1 else k
    if X.stride(-1) != 1 or (X.dim() == 3 and batches > 1 and X.stride(0) != rows * ld_x):
        raise ValueError("X must have unit column stride and batches rows * ld_x apart")
    lead = () if X.dim() == 2 else (batches,)
    kb = _cdiv(k, 128)
    fdt = torch.float8_e4m3fn if int(fmt) == E4M3 else torch.float8_e5m2
    if A is None:
        A = torch.empty(lead + (rows, k), dtype=fdt, device=X.device)
    else:
        _need(A, "A", _FP8, X.dim())
        if tuple(A.shape) != lead + (rows, k):
            raise ValueError("A shape does not fit X")
    if sA is None:
        sA = torch.empty(lead + (kb, fg_scales_a_ld(rows)), dtype=torch.float32, device=X.device)
    else:
        _need(sA, "sA", _F32, X.dim())
        if tuple(sA.shape[:-1]) != lead + (kb,) or sA.shape[-1] < rows:
            raise ValueError("sA shape does not fit X")
    mp = 0
    if masked_m is not None:
        _need(masked_m, "masked_m", _I32, 1)
        if masked_m.shape[0] != batches:
            raise ValueError("masked_m must hold one count per batch")
        mp = masked_m.data_ptr()
    name = "fg_quantize_fp8_per_token_f32in" if X.dtype == torch.float32 else "fg_quantize_fp8_per_token"
    _launch(name, (("X", X), ("A", A), ("sA", sA), ("masked_m", masked_m)), stream,
            X.data_ptr(), ld_x, int(fmt), A.data_ptr(), sA.data_ptr(), sA.shape[-1], mp, batches, rows, k)
    return A, sA


def fg_get_device_status(stream=None):
    """Synchronize the stream; return (status, detail) of this device and clear it."""
    d = ctypes.c_uint32(0)
    st = lib().fg_get_device_status(_stream_ptr(stream), ctypes.byref(d))
    return st, d.value


def fg_set_num_sms(n: int) -> None:
    _check("fg_set_num_sms", lib().fg_set_num_sms(int(n)))


def fg_set_config_override(block_n: int = 0, split_k: int = 0) -> None:
    """Force the dense tile plan (block_n 128/256, split_k 1..8; 0 = automatic)."""
    _check("fg_set_config_override", lib().fg_set_config_override(int(block_n), int(split_k)))


def fg_query_dense_plan(m: int, n: int, k: int):
    """(block_n, split_k) that a dense call of this shape would use."""
    bn, sp = ctypes.c_int(0), ctypes.c_int(0)
    _check("fg_query_dense_plan", lib().fg_query_dense_plan(int(m), int(n), int(k), ctypes.byref(bn), ctypes.byref(sp)))
    return bn.value, sp.value


def fg_query_dense_plan_ex(m: int, n: int, k: int):
    """(block_n, split_k, cta_pair) that a dense call of this shape would use."""
    bn, sp, pr = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check("fg_query_dense_plan_ex", lib().fg_query_dense_plan_ex(int(m), int(n), int(k), ctypes.byref(bn),
                                                                ctypes.byref(sp), ctypes.byref(pr)))
    return bn.value, sp.value, pr.value


def fg_set_pair_mode(mode: int) -> None:
    """-1: CTA-pair tiles where they apply (default); 0: never; 1: every persistent 256-wide plan."""
    _check("fg_set_pair_mode", lib().fg_set_pair_mode(int(mode)))


def fg_set_swap_mode(mode: int) -> None:
    """Swapped operand roles (dense m <= 256, masked M_cap <= 256): -1 automatic, which never picks them
    (measured slower on every problem); 0 never; 1 wherever they apply."""
    _check("fg_set_swap_mode", lib().fg_set_swap_mode(int(mode)))


def fg_query_plan(kind: int, rows: int, G: int, n: int, k: int):
    """(tile width, split_k, cta_pair, swap_ab, deferred_stores) of a call: kind 0 dense, 1 contiguous,
    2 masked, 3 K-grouped (rows = M, n = N, k = K)."""
    pl = (ctypes.c_int * 5)()
    _check("fg_query_plan", lib().fg_query_plan(int(kind), int(rows), int(G), int(n), int(k), pl))
    return tuple(pl)


def fg_set_programmatic_launch(enable: bool) -> None:
    _check("fg_set_programmatic_launch", lib().fg_set_programmatic_launch(1 if enable else 0))


def fg_set_watchdog_ms(ms: int) -> None:
    _check("fg_set_watchdog_ms", lib().fg_set_watchdog_ms(int(ms)))


def fg_status_string(st: int) -> str:
    return lib().fg_status_string(int(st)).decode()


def fg_version() -> int:
    return lib().fg_version()
