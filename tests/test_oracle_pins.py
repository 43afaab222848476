"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties one part of the oracle to something fixed outside it: the FP8
format table of the page "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践" (section 3.1), hand
decoded bytes, torch's float8/bfloat16 conversions, numpy's float64 matmul on
the unit-scale special case, closed forms, brute force over all FP8 codes and
invariants of the definition (zero scales, power-of-two linearity, grouped
layouts equal per-group dense calls).  No GPU is used.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_formats():
    rows = {}
    with open(os.path.join(GOLDEN, "fp8_formats.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, s, e, m, mx = line.split()
            rows[name] = (int(s), int(e), int(m), float(mx))
    return rows


# ------------------------------------------------------------------ decoding

@pytest.mark.parametrize("code,val", [
    (0x38, 1.0), (0x7E, 448.0), (0xFE, -448.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9),
    (0x08, 2.0 ** -6), (0x00, 0.0), (0x40, 2.0), (0x3C, 1.5), (0x30, 0.5), (0xB8, -1.0),
])
def test_e4m3_hand_decoded(code, val):
    assert oracle.decode(oracle.E4M3, code) == val


def test_e4m3_signed_zero_and_nan():
    z = oracle.decode(oracle.E4M3, 0x80)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0
    assert math.isnan(oracle.decode(oracle.E4M3, 0x7F))
    assert math.isnan(oracle.decode(oracle.E4M3, 0xFF))


@pytest.mark.parametrize("code,val", [
    (0x7B, 57344.0), (0x01, 2.0 ** -16), (0x3C, 1.0), (0x7C, math.inf), (0xFC, -math.inf),
    (0x04, 2.0 ** -14), (0xBC, -1.0), (0x3E, 1.5),
])
def test_e5m2_hand_decoded(code, val):
    assert oracle.decode(oracle.E5M2, code) == val


def test_e5m2_nans():
    for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF):
        assert math.isnan(oracle.decode(oracle.E5M2, c))


@pytest.mark.parametrize("name,fmt", [("E4M3", oracle.E4M3), ("E5M2", oracle.E5M2)])
def test_formats_match_page_table(name, fmt):
    """Largest finite value and the exponent/mantissa widths of the page's table."""
    sign, ebits, mbits, mx = _golden_formats()[name]
    t = oracle.decode_table(fmt)
    fin = t[np.isfinite(t)]
    assert fin.max() == mx and fin.min() == -mx
    # positive codes: the upper bit is the sign
    assert sign == 1 and all(oracle.decode(fmt, c) == -oracle.decode(fmt, c | 0x80)
                             for c in range(0x80) if np.isfinite(t[c]) and t[c] != 0)
    # within one binade, consecutive codes differ by 2^-mbits relative
    one = [c for c in range(0x80) if t[c] == 1.0][0]
    assert t[one + 1] == 1.0 + 2.0 ** -mbits
    # the smallest normal is 2^(1 - bias), bias = 2^(ebits-1) - 1
    bias = 2 ** (ebits - 1) - 1
    smallest_normal = t[1 << mbits]
    assert smallest_normal == 2.0 ** (1 - bias)
    # the smallest subnormal is one mantissa step below that
    assert t[1] == 2.0 ** (1 - bias - mbits)


@pytest.mark.parametrize("fmt,tdt", [(oracle.E4M3, torch.float8_e4m3fn), (oracle.E5M2, torch.float8_e5m2)])
def test_decode_matches_torch_float8(fmt, tdt):
    ref = torch.arange(256, dtype=torch.uint8).view(tdt).to(torch.float64).numpy()
    ours = oracle.decode_table(fmt)
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.all(both_nan | (ref == ours))
    assert np.array_equal(np.signbit(ref[~both_nan]), np.signbit(ours[~both_nan]))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_decode_roundtrip(fmt):
    """The input generator's encoder inverts the oracle's decoder on every finite code."""
    t = oracle.decode_table(fmt)
    codes = np.array([c for c in range(256) if np.isfinite(t[c])], np.uint8)
    vals = t[codes].astype(np.float32)
    back = wl.encode_fp8(vals, fmt)
    # -0 and +0 both decode to zero; compare values for those, codes elsewhere
    nz = vals != 0
    assert np.array_equal(back[nz], codes[nz])
    assert np.all(t[back[~nz]] == 0)


# ------------------------------------------------------------ bf16 rounding

@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000),
    (1.0 + 2.0 ** -8, 0x3F80),            # tie, even stays
    (1.0 + 3 * 2.0 ** -8, 0x3F82),        # tie, rounds up to even
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),  # just above the tie: direct rounding from FP64
    (1.0 + 2.0 ** -9, 0x3F80),
    (255 * 2.0 ** 120, 0x7F7F),           # largest finite
    (2.0 ** 128, 0x7F80), (-1e300, 0xFF80),
    (255 * 2.0 ** 120 + 2.0 ** 119, 0x7F80),  # tie above max goes to inf (max is odd)
    (2.0 ** -126, 0x0080), (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000),
    (3 * 2.0 ** -134, 0x0002), (127 * 2.0 ** -133, 0x007F),
])
def test_bf16_rne_hand_cases(x, bits):
    assert oracle.bf16_rne(x) == bits


def test_bf16_rne_negative_zero_and_nan():
    assert oracle.bf16_rne(-0.0) == 0x8000
    assert oracle.bf16_rne(float("nan")) == 0x7FC0
    assert oracle.bf16_rne(float("inf")) == 0x7F80


def test_bf16_rne_matches_torch_on_float32_inputs():
    """On values exactly representable in float32, direct rounding from FP64
    equals torch's float32 -> bfloat16 round-to-nearest-even."""
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(1000.0),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),  # subnormal float32 range
        np.float32(1.0) + np.arange(512, dtype=np.float32) * np.float32(2.0 ** -16),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    ours = np.array([oracle.bf16_rne(float(v)) for v in x], np.uint16)
    assert np.array_equal(ref, ours)


# -------------------------------------------------------------- the GEMM

def _dec(codes, fmt):
    return oracle.decode_table(fmt)[np.asarray(codes, np.int64)]


def _bits_to_f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


def test_unit_scales_equal_numpy_matmul_exactly():
    """Scales of one reduce the definition to a plain matmul; for E4M3 every
    partial sum is exact in FP64, so any summation order gives the same bits."""
    p = wl.dense(37, 300, 400, seed=11)  # partial last K block (400 = 3*128 + 16)
    sA = np.ones_like(p.sA)
    sB = np.ones_like(p.sB)
    d16, d64 = oracle.gemm_fp8_nt(p.A, 0, sA, p.B, 0, sB)
    ref = _dec(p.A, 0) @ _dec(p.B, 0).T
    assert np.array_equal(d64, ref)
    # where the sum is exact in float32, torch's float32 -> bfloat16 rounding
    # is a second, independent rounding of the same value
    exact32 = ref.astype(np.float32).astype(np.float64) == ref
    assert exact32.mean() > 0.2
    ref16 = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(d16.view(np.int16)[exact32], ref16[exact32])


def test_row_and_column_block_scales_equal_scaled_numpy_matmul():
    """Scales constant along K (power-of-two per row, per 128-column block):
    D = diag(sA) (A B^T) diag(sB), exact in FP64."""
    rng = np.random.default_rng(3)
    p = wl.dense(20, 260, 256, seed=12)
    ra = np.exp2(rng.integers(-6, 7, size=20)).astype(np.float32)
    rb = np.exp2(rng.integers(-6, 7, size=3)).astype(np.float32)
    sA = np.repeat(ra[:, None], 2, axis=1)
    sB = np.repeat(rb[:, None], 2, axis=1)
    _, d64 = oracle.gemm_fp8_nt(p.A, 0, sA, p.B, 0, sB)
    col_scale = rb[np.arange(260) // 128].astype(np.float64)
    ref = (ra.astype(np.float64)[:, None] * (_dec(p.A, 0) @ _dec(p.B, 0).T)) * col_scale[None, :]
    assert np.array_equal(d64, ref)


def test_mixed_e4m3_e5m2_unit_scales_close_to_numpy():
    p = wl.dense(16, 64, 256, seed=13, b_fmt=wl.E5M2)
    _, d64 = oracle.gemm_fp8_nt(p.A, 0, np.ones_like(p.sA), p.B, 1, np.ones_like(p.sB))
    ref = _dec(p.A, 0) @ _dec(p.B, 1).T
    np.testing.assert_allclose(d64, ref, rtol=1e-14, atol=0)


def test_brute_force_all_code_pairs_k1():
    """k = 1: every E4M3 x E4M3 code pair times power-of-two scales, against
    torch's decode and torch's float32 -> bfloat16 rounding (the product of two
    FP8 values has at most 8 significant bits, so float32 holds it exactly)."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    A = codes.reshape(-1, 1)
    B = codes.reshape(-1, 1)
    rng = np.random.default_rng(5)
    sA = np.exp2(rng.integers(-4, 5, size=(len(codes), 1))).astype(np.float32)
    sB = np.exp2(rng.integers(-4, 5, size=(2, 1))).astype(np.float32)
    d16, d64 = oracle.gemm_fp8_nt(A, 0, sA, B, 0, sB)
    tv = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    colsc = sB[np.arange(len(codes)) // 128, 0].astype(np.float64)
    ref = (tv[:, None] * tv[None, :]) * (sA.astype(np.float64) * colsc[None, :])
    assert np.array_equal(d64, ref)
    ref16 = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    ref16 = ref16.view(np.uint16)
    # the sign of a zero result is not part of the definition (a sum that
    # starts from +0 turns -0 products into +0): compare zeros as zeros
    def unsign0(b):
        return np.where((b & 0x7FFF) == 0, 0, b)
    assert np.array_equal(unsign0(d16), unsign0(ref16))


def test_closed_form_all_ones():
    """A = B = 1.0 everywhere with uniform scales a, b: D = k * a * b."""
    m, n, k = 5, 136, 384
    A = np.full((m, k), 0x38, np.uint8)
    B = np.full((n, k), 0x38, np.uint8)
    sA = np.full((m, 3), 0.75, np.float32)
    sB = np.full((2, 3), 2.5, np.float32)
    d16, d64 = oracle.gemm_fp8_nt(A, 0, sA, B, 0, sB)
    assert np.all(d64 == k * 0.75 * 2.5)
    assert np.all(_bits_to_f(d16) == 720.0)


def test_closed_form_geometric_lhs_scales():
    """sA[m,kb] = 2^kb with ones: D = 128 * sB * (2^KB - 1)."""
    KB = 6
    m, n, k = 3, 128, 128 * KB
    A = np.full((m, k), 0x38, np.uint8)
    B = np.full((n, k), 0x38, np.uint8)
    sA = np.tile(np.exp2(np.arange(KB)).astype(np.float32), (m, 1))
    sB = np.full((1, KB), 0.5, np.float32)
    _, d64 = oracle.gemm_fp8_nt(A, 0, sA, B, 0, sB)
    assert np.all(d64 == 128 * 0.5 * (2 ** KB - 1))


def test_one_hot_selects_the_right_scale_entries():
    """Row r of A holds a single 1.0 at column kr; B is all ones.  Then
    D[r, c] = sA[r, kr // 128] * sB[c // 128, kr // 128]: a transposed or
    shifted scale index picks another entry and fails."""
    m, n, k = 3, 300, 384        # 3 N-blocks, 3 K-blocks, non-square scale grids
    kr = [5, 200, 300]
    A = np.zeros((m, k), np.uint8)
    for r in range(m):
        A[r, kr[r]] = 0x38
    B = np.full((n, k), 0x38, np.uint8)
    sA = (np.arange(m * 3, dtype=np.float32).reshape(m, 3) + 1) * np.float32(0.5)
    sB = (np.arange(9, dtype=np.float32).reshape(3, 3) + 1) * np.float32(4.0)
    _, d64 = oracle.gemm_fp8_nt(A, 0, sA, B, 0, sB)
    for r in range(m):
        kb = kr[r] // 128
        for c in (0, 127, 128, 255, 256, 299):
            assert d64[r, c] == float(sA[r, kb]) * float(sB[c // 128, kb])


def test_one_hot_on_b_selects_the_right_column():
    """B row c holds a single value at column kc; A is all ones.  A swapped
    operand (A[m] paired with B[m]) fails this."""
    m, n, k = 4, 8, 256
    A = np.full((m, k), 0x38, np.uint8)
    B = np.zeros((n, k), np.uint8)
    vals = [0x40, 0x44, 0x48, 0x30, 0xB8, 0x3C, 0x7E, 0x01]  # 2, 3, 4, .5, -1, 1.5, 448, 2^-9
    for c in range(n):
        B[c, (c * 37) % k] = vals[c]
    sA = np.ones((m, 2), np.float32)
    sB = np.ones((1, 2), np.float32)
    _, d64 = oracle.gemm_fp8_nt(A, 0, sA, B, 0, sB)
    for c in range(n):
        assert np.all(d64[:, c] == oracle.decode(0, vals[c]))


def test_zero_scale_block_equals_zeroed_payload():
    p = wl.dense(9, 200, 512, seed=14)
    sA = p.sA.copy()
    sA[:, 2] = 0.0
    A2 = p.A.copy()
    A2[:, 256:384] = 0
    _, d_a = oracle.gemm_fp8_nt(p.A, 0, sA, p.B, 0, p.sB)
    _, d_b = oracle.gemm_fp8_nt(A2, 0, p.sA, p.B, 0, p.sB)
    assert np.array_equal(d_a, d_b)
    sB = p.sB.copy()
    sB[1, :] = 0.0
    _, d_c = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, sB)
    assert np.all(d_c[:, 128:200] == 0.0)
    d16, d_z = oracle.gemm_fp8_nt(p.A, 0, np.zeros_like(p.sA), p.B, 0, p.sB)
    assert np.all(d_z == 0.0) and np.all((d16 & 0x7FFF) == 0)


def test_power_of_two_scale_linearity_is_bitwise():
    p = wl.dense(17, 130, 640, seed=15)
    d16, d64 = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB)
    for e in (-3, 1, 5):
        s = np.float32(2.0 ** e)
        e16, e64 = oracle.gemm_fp8_nt(p.A, 0, p.sA * s, p.B, 0, p.sB)
        assert np.array_equal(e64, d64 * float(s))
        f16, f64 = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB * s)
        assert np.array_equal(f64, d64 * float(s))
        assert np.array_equal(_bits_to_f(e16), _bits_to_f(d16) * float(s))


def test_sampled_positions_equal_full_result():
    p = wl.dense(70, 264, 272, seed=16)
    d16, d64 = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB)
    rng = np.random.default_rng(1)
    rows = rng.integers(0, 70, 500)
    cols = rng.integers(0, 264, 500)
    s16, s64 = oracle.gemm_fp8_nt_at(p.A, 0, p.sA, p.B, 0, p.sB, rows, cols)
    assert np.array_equal(s64, d64[rows, cols]) and np.array_equal(s16, d16[rows, cols])


def test_bf16_output_is_rounding_of_f64_output():
    p = wl.dense(8, 64, 256, seed=17)
    d16, d64 = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB)
    assert all(oracle.bf16_rne(float(v)) == int(b) for v, b in zip(d64.ravel(), d16.ravel()))


# --------------------------------------------------------- grouped layouts

SENTINEL = 0xFFFF


def test_contiguous_equals_per_group_dense_and_leaves_padding():
    p = wl.contiguous([100, 0, 130, 5], n=136, k=272, seed=18)
    assert p.M == 128 + 0 + 256 + 128
    init = np.full((p.M, p.n), SENTINEL, np.uint16)
    d16, d64 = oracle.grouped_contiguous(p.A, 0, p.sA, p.B, 0, p.sB, p.m_indices, init, want_f64=True)
    for g in range(p.G):
        rows = np.nonzero(p.m_indices == g)[0]
        if rows.size == 0:
            continue
        e16, e64 = oracle.gemm_fp8_nt(p.A[rows], 0, p.sA[rows], p.B[g], 0, p.sB[g])
        assert np.array_equal(d16[rows], e16) and np.array_equal(d64[rows], e64)
    pad = p.m_indices < 0
    assert pad.sum() == p.M - 235
    assert np.all(d16[pad] == SENTINEL)


def test_contiguous_out_of_range_group_ids_leave_rows_untouched():
    p = wl.contiguous([128, 128], n=64, k=128, seed=23)
    mi = p.m_indices.copy()
    mi[128:] = 2          # == G: not a group
    mi[5] = 99
    init = np.full((p.M, p.n), SENTINEL, np.uint16)
    d16, _ = oracle.grouped_contiguous(p.A, 0, p.sA, p.B, 0, p.sB, mi, init)
    assert np.all(d16[128:] == SENTINEL) and np.all(d16[5] == SENTINEL)
    assert not np.any(d16[:5] == SENTINEL)
    s16, _ = oracle.grouped_contiguous_at(p.A, 0, p.sA, p.B, 0, p.sB, mi, [5, 130], [0, 1])
    assert np.all(s16 == SENTINEL)


def test_contiguous_sampled_equals_full():
    p = wl.contiguous([60, 128], n=64, k=128, seed=19)
    init = np.full((p.M, p.n), SENTINEL, np.uint16)
    d16, _ = oracle.grouped_contiguous(p.A, 0, p.sA, p.B, 0, p.sB, p.m_indices, init)
    rows = np.arange(p.M).repeat(3)
    cols = np.tile([0, 31, 63], p.M)
    s16, _ = oracle.grouped_contiguous_at(p.A, 0, p.sA, p.B, 0, p.sB, p.m_indices, rows, cols)
    assert np.array_equal(s16, d16[rows, cols])


def test_masked_equals_per_group_dense_and_leaves_rest():
    p = wl.masked(3, 96, n=128, k=256, seed=20, masked_m=[0, 96, 37])
    init = np.full((p.G, p.M_cap, p.n), SENTINEL, np.uint16)
    d16, _ = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, init)
    for g in range(p.G):
        v = int(p.masked_m[g])
        if v:
            e16, _ = oracle.gemm_fp8_nt(p.A[g, :v], 0, p.sA[g, :v], p.B[g], 0, p.sB[g])
            assert np.array_equal(d16[g, :v], e16)
        assert np.all(d16[g, v:] == SENTINEL)


def test_masked_counts_are_clamped():
    p = wl.masked(2, 64, n=64, k=128, seed=21, masked_m=[-5, 1000])
    init = np.full((2, 64, 64), SENTINEL, np.uint16)
    d16, _ = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, init)
    assert np.all(d16[0] == SENTINEL)
    e16, _ = oracle.gemm_fp8_nt(p.A[1], 0, p.sA[1], p.B[1], 0, p.sB[1])
    assert np.array_equal(d16[1], e16)


def test_masked_sampled_equals_full():
    p = wl.masked(2, 64, n=64, k=128, seed=22, masked_m=[10, 64])
    init = np.full((2, 64, 64), SENTINEL, np.uint16)
    d16, _ = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, init)
    g = np.repeat([0, 1], 64 * 2)
    r = np.tile(np.repeat(np.arange(64), 2), 2)
    c = np.tile([3, 60], 128)
    s16, _ = oracle.grouped_masked_at(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, g, r, c)
    assert np.array_equal(s16, d16[g, r, c])


def test_oracle_rejects_bad_shapes():
    A = np.zeros((2, 0), np.uint8)
    with pytest.raises(ValueError):
        oracle.gemm_fp8_nt(A, 0, np.zeros((2, 0), np.float32), np.zeros((2, 0), np.uint8), 0,
                           np.zeros((1, 0), np.float32))


# ------------------------------------------- per-token FP8 quantization
#
# The quantizer's two parts are pinned separately: the float32 -> FP8 encoder
# by hand-worked codes, by torch's float8 conversion and by a brute-force
# nearest-code search written here; the 1x128 group steps (largest magnitude,
# scale = amax / fmax, division) by the input generator's numpy + torch
# quantizer, by brute force on tiny rows and by closed forms.

FMAX = {oracle.E4M3: 448.0, oracle.E5M2: 57344.0}


@pytest.mark.parametrize("fmt,v,code", [
    # E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits
    (oracle.E4M3, 1.5, 0x3C), (oracle.E4M3, -1.5, 0xBC), (oracle.E4M3, 448.0, 0x7E),
    (oracle.E4M3, 500.0, 0x7E), (oracle.E4M3, 1e30, 0x7E), (oracle.E4M3, -1e30, 0xFE),
    (oracle.E4M3, 2.0 ** -9, 0x01),
    (oracle.E4M3, 2.0 ** -10, 0x00),        # tie between 0 and the smallest subnormal: even
    (oracle.E4M3, 3 * 2.0 ** -10, 0x02),    # tie between 0x01 and 0x02: even
    (oracle.E4M3, 1.0625, 0x38),            # tie between 1.0 and 1.125: even (1.0)
    (oracle.E4M3, 1.1875, 0x3A),            # tie between 1.125 and 1.25: even (1.25)
    (oracle.E4M3, 1.0625 + 2.0 ** -20, 0x39),  # just above the tie
    (oracle.E4M3, -0.0, 0x80), (oracle.E4M3, 0.0, 0x00), (oracle.E4M3, -1e-10, 0x80),
    # E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits
    (oracle.E5M2, 1.5, 0x3E), (oracle.E5M2, 57344.0, 0x7B), (oracle.E5M2, 1e9, 0x7B),
    (oracle.E5M2, 2.0 ** -16, 0x01), (oracle.E5M2, 1.125, 0x3C), (oracle.E5M2, 1.375, 0x3E),
    (oracle.E5M2, -2.0 ** -17, 0x80),       # tie between -0 and -2^-16: even
])
def test_encode_hand_worked(fmt, v, code):
    assert oracle.encode_fp8(fmt, v) == code


def _encode_brute(fmt, v):
    """Nearest finite code by scanning all codes of v's sign (rounding is
    symmetric, so the sign bit is v's); ties to the even code; beyond the
    largest finite magnitude, that magnitude."""
    t = oracle.decode_table(fmt)
    v = float(np.float32(v))
    neg = math.copysign(1.0, v) < 0
    fin = [c for c in range(256) if np.isfinite(t[c]) and bool(c & 0x80) == neg]
    if abs(v) >= FMAX[fmt]:
        return next(c for c in fin if abs(t[c]) == FMAX[fmt])
    best = min(abs(t[c] - v) for c in fin)
    cands = [c for c in fin if abs(t[c] - v) == best]
    if len(cands) == 1:
        return cands[0]
    return next(c for c in cands if c % 2 == 0)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_equals_brute_force_at_midpoints(fmt):
    """Every midpoint between neighbouring finite values, one float32 step on
    either side of it, and every code's own value."""
    t = oracle.decode_table(fmt)
    pos = sorted({t[c] for c in range(128) if np.isfinite(t[c])})
    vals = []
    for a, b in zip(pos[:-1], pos[1:]):
        mid = np.float32((a + b) / 2)
        assert float(mid) == (a + b) / 2  # midpoints are exact in float32
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(np.inf))]
    vals += [np.float32(p) for p in pos]
    vals = vals + [-v for v in vals]
    for v in vals:
        assert oracle.encode_fp8(fmt, v) == _encode_brute(fmt, v), (fmt, float(v))


@pytest.mark.parametrize("fmt,tdt", [(oracle.E4M3, torch.float8_e4m3fn), (oracle.E5M2, torch.float8_e5m2)])
def test_encode_matches_torch_float8_in_range(fmt, tdt):
    """Quantizing a group whose largest magnitude is exactly fmax gives scale 1,
    so its codes are the encoder's codes of the values themselves; torch's
    float8 conversion (nearest even) must agree on 30k log-uniform values
    spanning the subnormals up to fmax."""
    rng = wl.rng_for(4242 + fmt)
    fmax = FMAX[fmt]
    lo = math.log2(fmax) - (26 if fmt == oracle.E4M3 else 40)
    mag = np.exp2(rng.uniform(lo, math.log2(fmax), size=(240, 127)))
    x = (mag * rng.choice([-1.0, 1.0], size=mag.shape)).astype(np.float32)
    x = np.concatenate([np.full((240, 1), fmax, np.float32), x], axis=1)  # amax = fmax
    q, s = oracle.quantize_per_token(x, fmt)
    assert np.all(s == 1.0)
    ref = torch.from_numpy(x).to(tdt).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("k", [16, 128, 300, 7168])
def test_quantize_matches_generator(fmt, k):
    """The generator's quantizer (numpy float32 division, torch float8) is an
    independent statement of the same steps."""
    rng = wl.rng_for(77 + k + fmt)
    x = rng.standard_normal((3, 45, k)).astype(np.float32)
    x *= np.exp2(rng.integers(-20, 20, size=(3, 45, 1))).astype(np.float32)  # per-row magnitudes
    x[0, 5, :] = 0.0                       # an all-zero row (all its groups zero)
    x[1, 7, : min(k, 128)] = 0.0           # one zero group
    x[2, 3, 0] = 3.0e38                    # a huge value (scale stays finite)
    q, s = oracle.quantize_per_token(x, fmt)
    q2, s2 = wl.quantize_rows(x, fmt)
    assert np.array_equal(s, s2)
    assert np.array_equal(q, q2)


def test_quantize_brute_force_tiny():
    """Two rows of 144 columns (a full group and a 16-wide tail), every step
    written out with Python floats rounded to float32 and the brute-force
    encoder."""
    rng = wl.rng_for(5)
    x = (rng.standard_normal((2, 144)) * 3).astype(np.float32)
    for fmt in (oracle.E4M3, oracle.E5M2):
        q, s = oracle.quantize_per_token(x, fmt)
        for r in range(2):
            for g, (c0, c1) in enumerate([(0, 128), (128, 144)]):
                amax = max(abs(float(v)) for v in x[r, c0:c1])
                sc = np.float32(np.float32(amax) / np.float32(FMAX[fmt]))
                assert s[r, g] == sc
                for c in range(c0, c1):
                    assert q[r, c] == _encode_brute(fmt, np.float32(x[r, c]) / sc)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_quantize_closed_forms(fmt):
    """Each nonzero group reaches +-fmax at its largest element, its scale is
    amax / fmax, the dequantized values are within half an FP8 step of the
    inputs, and a zero group gets scale 1 with zero codes."""
    rng = wl.rng_for(99 + fmt)
    x = rng.standard_normal((64, 384)).astype(np.float32)
    x[10, 128:256] = 0.0
    q, s = oracle.quantize_per_token(x, fmt)
    t = oracle.decode_table(fmt)
    dq = t[q]
    mbits = 3 if fmt == oracle.E4M3 else 2
    min_normal = 2.0 ** -6 if fmt == oracle.E4M3 else 2.0 ** -14
    for r in range(64):
        for g in range(3):
            xs = x[r, 128 * g:128 * (g + 1)].astype(np.float64)
            d = dq[r, 128 * g:128 * (g + 1)]
            if not np.any(xs):
                assert s[r, g] == 1.0 and np.all(q[r, 128 * g:128 * (g + 1)] == 0)
                continue
            amax = np.abs(xs).max()
            assert s[r, g] == np.float32(np.float32(amax) / np.float32(FMAX[fmt]))
            assert np.abs(d).max() == FMAX[fmt]
            v = xs / float(s[r, g])
            step = np.where(np.abs(v) >= min_normal,
                            np.exp2(np.floor(np.log2(np.maximum(np.abs(v), min_normal))) - mbits),
                            min_normal * 2.0 ** -mbits)
            # half a step, plus the float32 rounding of the division
            assert np.all(np.abs(d - v) <= step / 2 + np.abs(v) * 2.0 ** -23)
            assert np.all((np.sign(d) == np.sign(v)) | (d == 0))


def test_quantize_divides_rather_than_multiplying_by_the_reciprocal():
    """An exact FP8 tie after the division, which multiplying by a rounded
    reciprocal misses.  amax = 3136 gives s = 3136 / 448 = 7 exactly;
    x = 12.6875 (BF16: 1100.1011b) gives x / s = 1.8125 exactly, the midpoint
    between the E4M3 values 1.75 and 1.875, which rounds to the even code
    0x3E (1.75).  With 1/7 rounded to float (0.14285715) the product is
    1.8125001, above the midpoint: code 0x3F."""
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = 3136.0
    x[0, 1] = 12.6875
    x[0, 2] = -12.6875
    q, s = oracle.quantize_per_token(x, oracle.E4M3)
    assert s[0, 0] == 7.0
    assert q[0, 1] == 0x3E and q[0, 2] == 0xBE
    assert q[0, 0] == 0x7E


# ----------------------------------------------------------- K-grouped layout

def _k_problem(M, N, K, seed):
    p = wl.dense(M, N, K, seed=seed)
    return p.A, p.sA, p.B, p.sB


def test_k_grouped_unit_scales_equal_numpy_segment_matmuls():
    """Unit scales reduce each group to a plain matmul over its K segment:
    D[g] = dec(A[:, seg_g]) dec(B[:, seg_g])^T, exact in FP64 for E4M3 (numpy's
    float64 matmul on column slices is the independent reference; a wrong
    segment offset, a segment that runs over all of K, or an off-by-one K
    block all change the result)."""
    A, sA, B, sB = _k_problem(9, 140, 896, seed=41)
    ks = np.array([256, 0, 128, 384], np.int32)    # 768 of the 896 columns; the last 128 belong to no group
    _, d64 = oracle.k_grouped(A, 0, np.ones_like(sA), B, 0, np.ones_like(sB), ks)
    a, b = _dec(A, 0), _dec(B, 0)
    off = 0
    for g, kg in enumerate(ks):
        ref = a[:, off:off + kg] @ b[:, off:off + kg].T
        assert np.array_equal(d64[g], ref), g
        off += kg
    assert np.all(d64[1] == 0.0)


def test_k_grouped_equals_dense_on_segment_slices():
    """With general scales, group g equals the dense definition applied to the
    column slice of A and B and the matching columns of sA and sB (bitwise:
    the same block sums in the same order)."""
    A, sA, B, sB = _k_problem(12, 300, 1024, seed=42)
    ks = np.array([384, 128, 512], np.int32)
    d16, d64 = oracle.k_grouped(A, 0, sA, B, 0, sB, ks)
    off = 0
    for g, kg in enumerate(ks):
        b0, b1 = off // 128, (off + kg) // 128
        e16, e64 = oracle.gemm_fp8_nt(A[:, off:off + kg], 0, sA[:, b0:b1], B[:, off:off + kg], 0, sB[:, b0:b1])
        assert np.array_equal(d64[g], e64) and np.array_equal(d16[g], e16), g
        off += kg


def test_k_grouped_groups_sum_to_the_full_k_product():
    """Segments that tile all of K: the sum over groups is the dense result
    over the whole K (power-of-two scales keep every term exact in FP64)."""
    rng = np.random.default_rng(43)
    A, _, B, _ = _k_problem(8, 130, 640, seed=43)
    sA = np.exp2(rng.integers(-4, 5, size=(8, 5))).astype(np.float32)
    sB = np.exp2(rng.integers(-4, 5, size=(2, 5))).astype(np.float32)
    ks = np.array([128, 256, 0, 256], np.int32)
    _, d64 = oracle.k_grouped(A, 0, sA, B, 0, sB, ks)
    _, full = oracle.gemm_fp8_nt(A, 0, sA, B, 0, sB)
    assert np.array_equal(d64.sum(axis=0), full)


def test_k_grouped_one_hot_scale_picks_the_segment_block():
    """sA zero except one K block (scale 2^3) inside group 1's segment: only
    group 1 is nonzero, and it equals 8 x the unit-scale product of that one
    block -- a shifted segment or scale index would select another block."""
    A, _, B, _ = _k_problem(6, 64, 640, seed=44)
    sA = np.zeros((6, 5), np.float32)
    sA[:, 3] = 8.0
    sB = np.ones((1, 5), np.float32)
    ks = np.array([256, 256, 128], np.int32)        # group 1 = K blocks 2 and 3
    _, d64 = oracle.k_grouped(A, 0, sA, B, 0, sB, ks)
    ref = 8.0 * (_dec(A, 0)[:, 384:512] @ _dec(B, 0)[:, 384:512].T)
    assert np.array_equal(d64[1], ref)
    assert np.all(d64[0] == 0.0) and np.all(d64[2] == 0.0)


def test_k_grouped_sampled_equals_full_and_bad_segments_are_refused():
    A, sA, B, sB = _k_problem(10, 72, 512, seed=45)
    ks = np.array([128, 256, 128], np.int32)
    d16, d64 = oracle.k_grouped(A, 0, sA, B, 0, sB, ks)
    rng = np.random.default_rng(0)
    g, r, c = rng.integers(0, 3, 50), rng.integers(0, 10, 50), rng.integers(0, 72, 50)
    s16, s64 = oracle.k_grouped_at(A, 0, sA, B, 0, sB, ks, g, r, c)
    assert np.array_equal(s16, d16[g, r, c]) and np.array_equal(s64, d64[g, r, c])
    for bad in ([100, 128], [-128, 256], [256, 384]):      # not a multiple of 128; negative; more than K
        with pytest.raises(ValueError):
            oracle.k_grouped(A, 0, sA, B, 0, sB, np.array(bad, np.int32))
