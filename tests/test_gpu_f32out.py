"""GPU parity of the FP32-output GEMM calls (*_f32out).

Two checks per case:
- against the oracle's FP64 result, with the stated bar applied to the
  unrounded values (per element |d| <= 1e-2 * max|ref|, aggregate relative
  error <= 1e-3);
- against the BF16 call on the same inputs and tile plan: rounding the FP32
  output to BF16 (nearest even) must give the BF16 call's bits exactly, since
  both run the same accumulation and differ only in the epilogue.
Rows the grouped calls must leave untouched keep a NaN sentinel."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_nt_gb300 as fg
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_common import d_to_bits, dev, fp8_dtype, sample_positions  # noqa: E402

SENT = 0x7FCADBAD  # float32 NaN pattern the kernels never write


def _empty_f32(shape):
    return torch.full(shape, SENT, dtype=torch.int32, device="cuda").view(torch.float32)


def _compare_f32(got, ref64, what):
    g = got.astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    m = float(np.max(np.abs(ref64))) if ref64.size else 0.0
    d = np.abs(g - ref64)
    assert np.all(d <= 1e-2 * m), f"{what}: max |d| {d.max():.3e} > 1e-2 * {m:.3e}"
    nr = float(np.linalg.norm(ref64))
    agg = float(np.linalg.norm(g - ref64)) / nr if nr > 0 else float(np.linalg.norm(g))
    assert agg <= 1e-3, f"{what}: aggregate relative error {agg:.3e}"
    return agg


def _bf16_bits_of(x32: torch.Tensor) -> np.ndarray:
    return d_to_bits(x32.to(torch.bfloat16))


def _dense_pair(p):
    """(FP32 D, BF16 D) of one dense problem, same plan."""
    A, B = dev(p.A, fp8_dtype(p.a_fmt)), dev(p.B, fp8_dtype(p.b_fmt))
    sA, sB = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB)
    D32 = _empty_f32((p.m, p.n))
    D16 = torch.empty((p.m, p.n), dtype=torch.bfloat16, device="cuda")
    fg.fg_gemm_fp8_nt_f32out(A, sA, B, sB, D32)
    fg.fg_gemm_fp8_nt(A, sA, B, sB, D16)
    torch.cuda.synchronize()
    assert fg.fg_get_device_status()[0] == fg.FG_OK
    return D32, D16


@pytest.fixture
def plan():
    def set_plan(mode):
        if mode == "pair":
            fg.fg_set_pair_mode(1)
            fg.fg_set_config_override(0, 0)
        else:
            fg.fg_set_pair_mode(0)
            bn, split = {"one_cta_256": (256, 1), "one_cta_128": (128, 1), "split_128x4": (128, 4),
                         "split_256x3": (256, 3)}[mode]
            fg.fg_set_config_override(bn, split)

    yield set_plan
    fg.fg_set_pair_mode(-1)
    fg.fg_set_config_override(0, 0)


@pytest.mark.parametrize("mode", ["pair", "one_cta_256", "one_cta_128", "split_128x4", "split_256x3"])
@pytest.mark.parametrize("m,n,k", [(130, 520, 1280), (300, 264, 1040), (64, 2112, 1024), (1, 8, 16)])
def test_dense_f32out(plan, mode, m, n, k):
    plan(mode)
    p = wl.dense(m, n, k, seed=12000 + m + n + k)
    D32, D16 = _dense_pair(p)
    _, ref64 = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB)
    _compare_f32(D32.cpu().numpy(), ref64, f"dense f32 {m}x{n}x{k} {mode}")
    assert np.array_equal(_bf16_bits_of(D32), d_to_bits(D16)), f"{mode}: bf16(f32 out) != bf16 out"


def test_dense_f32out_e5m2_b():
    p = wl.dense(256, 512, 768, seed=12345, b_fmt=wl.E5M2)
    D32, D16 = _dense_pair(p)
    _, ref64 = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 1, p.sB)
    _compare_f32(D32.cpu().numpy(), ref64, "dense f32 e5m2 B")
    assert np.array_equal(_bf16_bits_of(D32), d_to_bits(D16))


def test_contiguous_f32out():
    p = wl.contiguous([100, 0, 300, 5, 128], n=264, k=400, seed=12400)
    A, B = dev(p.A, fp8_dtype(p.a_fmt)), dev(p.B, fp8_dtype(p.b_fmt))
    sA, sB, mi = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB), dev(p.m_indices)
    D32 = _empty_f32((p.M, p.n))
    D16 = torch.full((p.M, p.n), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fg.fg_grouped_gemm_fp8_contiguous_f32out(A, sA, B, sB, D32, mi)
    fg.fg_grouped_gemm_fp8_contiguous(A, sA, B, sB, D16, mi)
    torch.cuda.synchronize()
    assert fg.fg_get_device_status()[0] == fg.FG_OK
    init = np.full((p.M, p.n), 0xFFFF, np.uint16)
    _, ref64 = oracle.grouped_contiguous(p.A, 0, p.sA, p.B, 0, p.sB, p.m_indices, init, want_f64=True)
    got = D32.cpu().numpy()
    w = p.m_indices >= 0
    assert np.all(got[~w].view(np.uint32) == SENT), "padding rows were written"
    _compare_f32(got[w], ref64[w], "contiguous f32")
    assert np.array_equal(_bf16_bits_of(D32)[w], d_to_bits(D16)[w])


@pytest.mark.parametrize("M_cap,counts", [(256, [0, 130, 256]), (128, [1, 128, 77])])
def test_masked_f32out(M_cap, counts):
    """M_cap 256 runs on CTA pairs, 128 on one-CTA tiles."""
    p = wl.masked(3, M_cap, n=256, k=512, seed=12500 + M_cap, masked_m=counts)
    A, B = dev(p.A, fp8_dtype(p.a_fmt)), dev(p.B, fp8_dtype(p.b_fmt))
    sA, sB, mm = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB), dev(p.masked_m)
    D32 = _empty_f32((p.G, p.M_cap, p.n))
    D16 = torch.empty((p.G, p.M_cap, p.n), dtype=torch.bfloat16, device="cuda")
    fg.fg_grouped_gemm_fp8_masked_f32out(A, sA, B, sB, D32, mm)
    fg.fg_grouped_gemm_fp8_masked(A, sA, B, sB, D16, mm)
    torch.cuda.synchronize()
    assert fg.fg_get_device_status()[0] == fg.FG_OK
    init = np.full((p.G, p.M_cap, p.n), 0xFFFF, np.uint16)
    _, ref64 = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, init, want_f64=True)
    got = D32.cpu().numpy()
    valid = np.arange(p.M_cap)[None, :] < np.asarray(counts)[:, None]
    assert np.all(got[~valid].view(np.uint32) == SENT), "rows past the counts were written"
    _compare_f32(got[valid], ref64[valid], "masked f32")
    assert np.array_equal(_bf16_bits_of(D32)[valid], d_to_bits(D16)[valid])


def test_dense_f32out_full_size_sampled():
    """4096 x 7168 x 2048 (a sweep shape, CTA-pair tiles) on sampled outputs."""
    m, n, k = 4096, 7168, 2048
    p = wl.dense(m, n, k, seed=12600)
    D32, D16 = _dense_pair(p)
    assert np.array_equal(_bf16_bits_of(D32), d_to_bits(D16))
    rr, cc = sample_positions(m, n, seed=12601)
    _, ref64 = oracle.gemm_fp8_nt_at(p.A, 0, p.sA, p.B, 0, p.sB, rr, cc)
    got = D32.cpu().numpy()[rr, cc]
    _compare_f32(got, ref64, "dense f32 4096x7168x2048 sampled")
