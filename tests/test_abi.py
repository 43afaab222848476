"""The C ABI library builds, loads without a GPU and exports every function that
include/fp8gemm.h declares; host-side argument checks return the documented
status codes before any CUDA call (no compute is launched here)."""
import ctypes
import os
import re

import pytest

import moe_grouped_gemm_nt_gb300 as fg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8gemm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fg_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_three_gemm_calls():
    names = declared_functions()
    for n in ("fg_gemm_fp8_nt", "fg_grouped_gemm_fp8_contiguous", "fg_grouped_gemm_fp8_masked"):
        assert n in names


def test_library_exports_every_declared_symbol():
    h = ctypes.CDLL(fg._build.build())
    for name in declared_functions():
        assert hasattr(h, name), name
    # the binding knows the signature of every declared function
    assert set(declared_functions()) <= set(fg.SIGNATURES)


def test_debug_build_exports_the_same_symbols_and_says_so():
    """libfp8gemm_debug.so (FG_DEBUG: device-side bounds checks, single-stage
    pipelines) is a drop-in for the library: same C ABI; it reports itself
    as the debug build and accepts the coordinate hook the release build
    refuses."""
    h = fg.lib(debug=True)
    assert os.path.basename(fg.library_path(True)) == "libfp8gemm_debug.so"
    for name in declared_functions():
        assert hasattr(h, name), name
    assert h.fg_debug_build() == 1 and fg.lib(debug=False).fg_debug_build() == 0
    assert fg.lib(debug=False).fg_debug_bad_coordinate(0) == 3  # FG_ERR_UNSUPPORTED
    assert h.fg_debug_bad_coordinate(-1) == 0
    fg.use_debug_library(True)
    try:
        assert fg.lib() is h and fg.fg_version() >= 100
    finally:
        fg.use_debug_library(False)
    assert fg.lib() is not h


def test_host_only_helpers():
    assert fg.fg_scales_a_ld(1) == 4 and fg.fg_scales_a_ld(4) == 4 and fg.fg_scales_a_ld(130) == 132
    assert fg.fg_status_string(0) == "FG_OK" and fg.fg_status_string(5) == "FG_ERR_TIMEOUT"
    assert fg.fg_version() >= 100


FAKE = 1 << 20  # a 16-byte aligned fake device address; never dereferenced by these calls


@pytest.mark.parametrize("kw,expect", [
    (dict(A=0), 1),                      # null pointer
    (dict(a_fmt=3), 1),                  # bad FP8 format
    (dict(k=24), 3),                     # k % 16 != 0
    (dict(n=12), 3),                     # n % 8 != 0
    (dict(ld=130), 2),                   # ld_sA % 4 != 0
    (dict(ld=64), 1),                    # ld_sA < m
    (dict(A=FAKE + 8), 2),               # A not 16-byte aligned
    (dict(D=FAKE + 4), 2),               # D not 16-byte aligned
    (dict(m=-1), 1),
    (dict(m=0, ld=4), 0),                # empty problem: a no-op that touches nothing
])
def test_dense_argument_checks(kw, expect):
    a = dict(A=FAKE, a_fmt=0, sA=FAKE, ld=128, B=FAKE, b_fmt=0, sB=FAKE, D=FAKE, m=128, n=256, k=512)
    a.update(kw)
    st = fg.lib().fg_gemm_fp8_nt(a["A"], a["a_fmt"], a["sA"], a["ld"], a["B"], a["b_fmt"], a["sB"], a["D"],
                                 a["m"], a["n"], a["k"], None)
    assert st == expect


def test_grouped_argument_checks():
    L = fg.lib()
    # contiguous M must be a multiple of 128; m_indices required
    assert L.fg_grouped_gemm_fp8_contiguous(FAKE, 0, FAKE, 200, FAKE, 0, FAKE, FAKE, FAKE, 200, 64, 128, 2,
                                            None) == 3
    assert L.fg_grouped_gemm_fp8_contiguous(FAKE, 0, FAKE, 256, FAKE, 0, FAKE, FAKE, None, 256, 64, 128, 2,
                                            None) == 1
    # masked needs its count tensor and G >= 1
    assert L.fg_grouped_gemm_fp8_masked(FAKE, 0, FAKE, 256, FAKE, 0, FAKE, FAKE, None, 2, 256, 64, 128,
                                        None) == 1
    assert L.fg_grouped_gemm_fp8_masked(FAKE, 0, FAKE, 256, FAKE, 0, FAKE, FAKE, FAKE, 0, 256, 64, 128,
                                        None) == 1
    assert L.fg_scales_a_to_mn_major(FAKE, FAKE, 1, 10, 2, 10, None) == 2
    assert L.fg_scales_a_to_mn_major(FAKE, FAKE, 1, 10, 2, 8, None) == 1


def test_tuning_knob_argument_checks():
    """The plan and pair-mode knobs validate their arguments on the host."""
    h = fg.lib()
    for mode in (-2, 2, 7):
        assert h.fg_set_pair_mode(mode) == 1
    for mode in (-1, 0, 1):
        assert h.fg_set_pair_mode(mode) == 0
    h.fg_set_pair_mode(-1)
    for bn, split in ((64, 1), (256, 9), (128, -1)):
        assert h.fg_set_config_override(bn, split) == 1
    assert h.fg_set_config_override(0, 0) == 0
    out = ctypes.c_int(0)
    assert h.fg_query_dense_plan_ex(128, 256, 512, ctypes.byref(out), ctypes.byref(out), None) == 1
    assert h.fg_query_dense_plan(0, 256, 512, ctypes.byref(out), ctypes.byref(out)) == 1


def test_quantize_argument_checks():
    """fg_quantize_fp8_per_token rejects bad arguments on the host, before any
    CUDA call (the pointers here are never dereferenced)."""
    Q = fg.lib().fg_quantize_fp8_per_token
    #        X     ld_x fmt A     sA    ld_sA masked batches rows k
    ok = [FAKE, 256, 0, FAKE, FAKE, 64, None, 1, 64, 256, None]

    def call(**kw):
        names = ["X", "ld_x", "fmt", "A", "sA", "ld_sA", "masked", "batches", "rows", "k", "stream"]
        args = dict(zip(names, ok))
        args.update(kw)
        return Q(*[args[n] for n in names])

    assert call(X=None) == 1 and call(A=None) == 1 and call(sA=None) == 1
    assert call(fmt=2) == 1 and call(fmt=-1) == 1
    assert call(ld_x=128) == 1            # ld_x < k
    assert call(ld_sA=60) == 1            # ld_sA < rows
    assert call(batches=0) == 1 and call(rows=-1) == 1 and call(k=0) == 1
    assert call(X=FAKE + 4) == 2 and call(A=FAKE + 8) == 2 and call(sA=FAKE + 4) == 2
    assert call(ld_x=260) == 2            # rows of X must stay 16-byte aligned
    assert call(ld_sA=66) == 2            # the GEMM's sA rule: ld_sA % 4 == 0
    assert call(k=136, ld_x=136) == 3     # k % 16 != 0
    assert call(k=128 * 65536, ld_x=128 * 65536) == 3  # more K blocks than a grid dimension holds
    assert call(batches=65536) == 3
    assert call(rows=0) == 0              # nothing to do: no launch


def test_quantize_f32_input_argument_checks():
    """fg_quantize_fp8_per_token_f32in applies the same host checks, with the
    row alignment of 4-byte elements (ld_x % 4 == 0 instead of % 8)."""
    Q = fg.lib().fg_quantize_fp8_per_token_f32in
    ok = [FAKE, 256, 0, FAKE, FAKE, 64, None, 1, 64, 256, None]

    def call(**kw):
        names = ["X", "ld_x", "fmt", "A", "sA", "ld_sA", "masked", "batches", "rows", "k", "stream"]
        args = dict(zip(names, ok))
        args.update(kw)
        return Q(*[args[n] for n in names])

    assert call(X=None) == 1 and call(A=None) == 1 and call(sA=None) == 1
    assert call(fmt=2) == 1 and call(ld_x=128) == 1 and call(ld_sA=60) == 1
    assert call(X=FAKE + 8) == 2 and call(A=FAKE + 8) == 2
    assert call(ld_x=258) == 2            # 1032-byte rows: not 16-byte aligned
    assert call(ld_x=260, rows=0) == 0    # 1040-byte rows are (a BF16 X of this ld_x is not)
    assert call(k=136, ld_x=136) == 3
    assert call(rows=0) == 0


def test_f32out_argument_checks():
    """The FP32-output calls share the BF16 calls' host-side checks."""
    L = fg.lib()
    ok = dict(A=FAKE, a_fmt=0, sA=FAKE, ld=128, B=FAKE, b_fmt=0, sB=FAKE, D=FAKE, m=128, n=256, k=512)

    def dense(**kw):
        a = dict(ok, **kw)
        return L.fg_gemm_fp8_nt_f32out(a["A"], a["a_fmt"], a["sA"], a["ld"], a["B"], a["b_fmt"], a["sB"],
                                       a["D"], a["m"], a["n"], a["k"], None)

    assert dense(D=None) == 1 and dense(a_fmt=3) == 1 and dense(n=0) == 1
    assert dense(D=FAKE + 8) == 2 and dense(ld=130) == 2
    assert dense(k=520) == 3 and dense(n=260) == 3
    assert dense(m=0) == 0  # nothing to do: no launch
    assert L.fg_grouped_gemm_fp8_contiguous_f32out(FAKE, 0, FAKE, 200, FAKE, 0, FAKE, FAKE, FAKE, 200, 64, 128, 2,
                                                   None) == 3
    assert L.fg_grouped_gemm_fp8_masked_f32out(FAKE, 0, FAKE, 256, FAKE, 0, FAKE, FAKE, None, 2, 256, 64, 128,
                                               None) == 1


def test_binding_rejects_host_tensors_and_wrong_dtypes():
    """The Python binding checks tensors before it calls the library: host
    tensors, wrong dtypes and shape mismatches raise (no CUDA call needed)."""
    import torch

    x_host = torch.zeros((4, 128), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fg.fg_quantize_fp8_per_token(x_host)  # not a CUDA tensor
    with pytest.raises(TypeError):
        fg.fg_quantize_fp8_per_token(torch.zeros((4, 128), dtype=torch.float32))
    a = torch.zeros((4, 128), dtype=torch.uint8)
    s = torch.zeros((1, 4), dtype=torch.float32)
    d16 = torch.zeros((4, 8), dtype=torch.bfloat16)
    d32 = torch.zeros((4, 8), dtype=torch.float32)
    b = torch.zeros((8, 128), dtype=torch.uint8)
    sb = torch.zeros((1, 1), dtype=torch.float32)
    with pytest.raises(ValueError):
        fg.fg_gemm_fp8_nt(a, s, b, sb, d16)  # host tensors
    with pytest.raises(ValueError):
        fg.fg_gemm_fp8_nt_f32out(a, s, b, sb, d32)
    with pytest.raises(ValueError):
        fg.fg_grouped_gemm_fp8_masked_f32out(a.view(1, 4, 128), s.view(1, 1, 4), b.view(1, 8, 128),
                                             sb.view(1, 1, 1), d32.view(1, 4, 8),
                                             torch.zeros(1, dtype=torch.int32))


def test_binding_rejects_operands_on_different_devices():
    """The library launches on the current device, so the binding refuses
    operands spread over two devices, and a torch stream of another device
    (checked on stand-ins that carry only a device attribute: no GPU needed)."""
    from types import SimpleNamespace

    import torch

    d0, d1 = torch.device("cuda", 0), torch.device("cuda", 1)
    t0, t1 = SimpleNamespace(device=d0), SimpleNamespace(device=d1)
    assert fg._common_device((("A", t0), ("B", t0), ("D", t0))) == d0
    assert fg._common_device((("A", t1), ("masked_m", None), ("D", t1))) == d1
    with pytest.raises(ValueError, match="D is on cuda:1"):
        fg._common_device((("A", t0), ("B", t0), ("D", t1)))
    with pytest.raises(ValueError, match="stream belongs to cuda:1"):
        fg._common_device((("A", t0), ("D", t0)), stream=SimpleNamespace(device=d1))
    # a raw stream handle cannot be checked and is accepted as given
    assert fg._common_device((("A", t0),), stream=12345) == d0


def test_k_grouped_argument_checks():
    """The K-grouped calls check their arguments on the host (no launch)."""
    L = fg.lib()
    ok = dict(A=FAKE, a_fmt=0, sA=FAKE, ld=128, B=FAKE, b_fmt=0, sB=FAKE, D=FAKE, ks=FAKE, G=2, M=128, N=256,
              K=512)

    def call(f32=False, **kw):
        a = dict(ok, **kw)
        f = L.fg_k_grouped_gemm_fp8_nt_f32out if f32 else L.fg_k_grouped_gemm_fp8_nt
        return f(a["A"], a["a_fmt"], a["sA"], a["ld"], a["B"], a["b_fmt"], a["sB"], a["D"], a["ks"], a["G"],
                 a["M"], a["N"], a["K"], None)

    for f32 in (False, True):
        assert call(f32, ks=None) == 1 and call(f32, A=None) == 1 and call(f32, G=0) == 1
        assert call(f32, b_fmt=5) == 1 and call(f32, ld=64) == 1 and call(f32, N=0) == 1
        assert call(f32, K=520) == 3 and call(f32, N=260) == 3
        assert call(f32, ld=132 + 2) == 2 and call(f32, D=FAKE + 4) == 2
        assert call(f32, M=0) == 0  # nothing to do: no launch
