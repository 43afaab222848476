"""GPU parity of the swapped-operand path (weights in the tensor core's
128-row role, the few rows of A as its N dimension) against the CPU oracle,
through the C ABI: dense calls with m <= 256 (forced with fg_set_swap_mode(1)),
masked calls with capacity <= 256 (forced the same way), 128- and 256-token
tiles, split-K clusters of 1..8 CTAs, FP32 output, rows past the counts left
untouched, bitwise repeatability, agreement with the unswapped path, and the
watchdog on this path."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_nt_gb300 as fg
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_common import SENTINEL, check_status, compare, d_to_bits, dev, fp8_dtype, run_dense, run_masked  # noqa: E402


@pytest.fixture
def swap_mode():
    def set_mode(mode, split=0):
        fg.fg_set_swap_mode(mode)
        fg.fg_set_config_override(0, split)

    yield set_mode
    fg.fg_set_swap_mode(-1)
    fg.fg_set_config_override(0, 0)


def plan_of(kind, rows, G, n, k):
    return list(fg.fg_query_plan(kind, rows, G, n, k))


@pytest.mark.parametrize("m,n,k", [(1, 8, 16), (64, 2112, 1024), (100, 264, 1040), (128, 256, 512),
                                   (129, 520, 384), (200, 2112, 272), (256, 128, 1280), (37, 7168, 2048)])
@pytest.mark.parametrize("split", [0, 1, 3, 8])
def test_swap_dense_matches_oracle(swap_mode, m, n, k, split):
    """Forced swapped path (automatic and forced split-K sizes) on ragged
    shapes: 128-token tiles for m <= 128, 256-token tiles above."""
    if split > 1 and (k + 127) // 128 < split:
        pytest.skip("fewer K blocks than ranks")
    swap_mode(1, split)
    plan = plan_of(0, m, 1, n, k)
    assert plan[3] == 1 and plan[0] == (128 if m <= 128 else 256)
    if split:
        assert plan[1] == split
    p = wl.dense(m, n, k, seed=7000 + m + n + k)
    got = d_to_bits(run_dense(p))
    ref, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(got, ref, what=f"swap dense {m}x{n}x{k} split={split}")


@pytest.mark.parametrize("counts,M_cap", [([0, 1, 127, 128, 129, 256], 256), ([37, 0, 96], 96),
                                          ([200, 64, 3], 200), ([256] * 4, 256), ([5], 128)])
@pytest.mark.parametrize("split", [0, 2, 5])
def test_swap_masked_rows_past_counts_untouched(swap_mode, counts, M_cap, split):
    swap_mode(1, split)
    plan = plan_of(2, M_cap, len(counts), 264, 1040)
    assert plan[3] == 1
    p = wl.masked(len(counts), M_cap, n=264, k=1040, seed=7100 + M_cap + split, masked_m=counts)
    got = d_to_bits(run_masked(p))
    init = np.full((p.G, p.M_cap, p.n), SENTINEL, np.uint16)
    ref, _ = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, init)
    valid = np.arange(M_cap)[None, :] < p.masked_m[:, None]
    assert np.array_equal(got[~valid], ref[~valid]), "rows past the count were written"
    if valid.any():
        compare(got[valid], ref[valid], what=f"swap masked {counts} split={split}")


@pytest.mark.parametrize("masked", [False, True])
def test_swap_f32out_rounds_to_the_bf16_call(swap_mode, masked):
    swap_mode(1)
    if masked:
        p = wl.masked(3, 256, n=264, k=512, seed=7201, masked_m=[0, 130, 256])
        A, B = dev(p.A, fp8_dtype(0)), dev(p.B, fp8_dtype(0))
        sA, sB, mm = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB), dev(p.masked_m)
        d32 = torch.full((p.G, p.M_cap, p.n), float("nan"), dtype=torch.float32, device="cuda")
        d16 = torch.empty((p.G, p.M_cap, p.n), dtype=torch.bfloat16, device="cuda")
        fg.fg_grouped_gemm_fp8_masked_f32out(A, sA, B, sB, d32, mm)
        fg.fg_grouped_gemm_fp8_masked(A, sA, B, sB, d16, mm)
        valid = np.arange(p.M_cap)[None, :] < p.masked_m[:, None]
        _, ref64 = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m,
                                         np.full((p.G, p.M_cap, p.n), SENTINEL, np.uint16), want_f64=True)
    else:
        p = wl.dense(200, 520, 1280, seed=7202)
        A, B = dev(p.A, fp8_dtype(0)), dev(p.B, fp8_dtype(0))
        sA, sB = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB)
        d32 = torch.empty((p.m, p.n), dtype=torch.float32, device="cuda")
        d16 = torch.empty((p.m, p.n), dtype=torch.bfloat16, device="cuda")
        fg.fg_gemm_fp8_nt_f32out(A, sA, B, sB, d32)
        fg.fg_gemm_fp8_nt(A, sA, B, sB, d16)
        valid = np.ones((p.m, p.n), bool)
        _, ref64 = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB)
    torch.cuda.synchronize()
    check_status()
    got32 = d32.cpu().numpy()
    if masked:
        assert np.all(np.isnan(got32[~valid])), "rows past the counts were written"
    g = got32[valid].astype(np.float64)
    r = ref64[valid]
    assert np.max(np.abs(g - r)) <= 1e-2 * np.max(np.abs(r))
    assert np.linalg.norm(g - r) / np.linalg.norm(r) <= 1e-3
    assert np.array_equal(d_to_bits(d32.to(torch.bfloat16))[valid], d_to_bits(d16)[valid])


@pytest.mark.parametrize("split", [1, 4])
def test_swap_is_bitwise_repeatable_and_close_to_unswapped(swap_mode, split):
    p = wl.dense(96, 7168, 2048, seed=7300)
    swap_mode(1, split)
    first = d_to_bits(run_dense(p))
    for _ in range(20):
        assert np.array_equal(d_to_bits(run_dense(p)), first), "repeated calls differ"
    swap_mode(0)
    other = d_to_bits(run_dense(p))
    ref, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(first, ref, what="swap")
    compare(other, ref, what="unswapped")


def test_swap_is_off_unless_forced(swap_mode):
    """The automatic choice keeps the unswapped plans (measured faster)."""
    swap_mode(-1)
    assert plan_of(0, 64, 1, 7168, 16384)[3] == 0
    assert plan_of(2, 256, 4, 4096, 7168)[3] == 0
    swap_mode(1)
    assert plan_of(0, 64, 1, 7168, 16384)[3] == 1
    assert plan_of(0, 257, 1, 7168, 16384)[3] == 0   # more rows than a token tile


def test_swap_watchdog_times_out_and_context_survives(swap_mode):
    """The producer leaves one K iteration unarmed (test hook): the waits run out,
    the call reports FG_ERR_TIMEOUT, and the next call on the context is exact."""
    swap_mode(1)
    p = wl.dense(64, 512, 1024, seed=7400)
    fg.fg_set_watchdog_ms(200)
    try:
        fg.lib().fg_debug_skip_producer_iteration(1)
        A, B = dev(p.A, fp8_dtype(0)), dev(p.B, fp8_dtype(0))
        sA, sB = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB)
        D = torch.empty((p.m, p.n), dtype=torch.bfloat16, device="cuda")
        fg.fg_gemm_fp8_nt(A, sA, B, sB, D)
        st, detail = fg.fg_get_device_status()
        assert st == 5, (st, detail)
    finally:
        fg.fg_set_watchdog_ms(0)
    got = d_to_bits(run_dense(p))
    ref, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(got, ref, what="after timeout")
