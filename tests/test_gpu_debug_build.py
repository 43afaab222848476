"""The FG_DEBUG build (libfp8gemm_debug.so) on the GPU: every layout and tile
plan through single-stage pipelines (split-K: the fewest stages that hold the
partial tile) with the device-side checks of TMA boxes, ring indices and TMEM
columns armed.  A correct run matches the oracle and leaves the status word
clean (no check fired); a load coordinate sent past K by the test hook is
caught before it is issued and reported as FG_ERR_DEVICE_CHECK with its tag,
and the next call is exact again.  The bisection follows the pages' debugging
method (page "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践",
sections 6.2-6.3: a single buffer, assertions on the data after each K step)."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_nt_gb300 as fg
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_common import (SENTINEL, check_status, compare, d_to_bits, dev, fp8_dtype,  # noqa: E402
                        run_contiguous, run_dense, run_masked)

DBG_TMA_A = 0x41


@pytest.fixture
def debug_lib():
    fg.use_debug_library(True)
    assert fg.lib().fg_debug_build() == 1
    yield fg.lib()
    fg.fg_set_config_override(0, 0)
    fg.fg_set_pair_mode(-1)
    fg.lib().fg_debug_set_pair_defer(-1)
    fg.fg_set_watchdog_ms(0)
    fg.use_debug_library(False)


PLANS = {
    "auto": (0, 0, -1, -1),
    "one_cta_256": (256, 1, 0, -1),
    "one_cta_128": (128, 1, 0, -1),
    "split2_128": (128, 2, 0, -1),
    "split4_256": (256, 4, 0, -1),
    "pair": (256, 1, 1, 0),
    "pair_deferred": (256, 1, 1, 1),
}


def _plan(lib, name):
    bn, split, pair, defer = PLANS[name]
    fg.fg_set_config_override(bn, split)
    fg.fg_set_pair_mode(pair)
    lib.fg_debug_set_pair_defer(defer)


@pytest.mark.parametrize("plan", list(PLANS))
@pytest.mark.parametrize("m,n,k", [(300, 520, 1040), (128, 256, 512), (1, 264, 400)])
def test_dense_debug_build_matches_oracle(debug_lib, plan, m, n, k):
    _plan(debug_lib, plan)
    p = wl.dense(m, n, k, seed=7000 + m + n + k)
    ref, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(d_to_bits(run_dense(p)), ref, what=f"debug build dense {m}x{n}x{k} {plan}")


def test_dense_f32_output_debug_build(debug_lib):
    _plan(debug_lib, "pair")
    p = wl.dense(300, 520, 640, seed=7101)
    A, B = dev(p.A, fp8_dtype(0)), dev(p.B, fp8_dtype(0))
    sA, sB = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB)
    d32 = torch.empty((p.m, p.n), dtype=torch.float32, device="cuda")
    fg.fg_gemm_fp8_nt_f32out(A, sA, B, sB, d32)
    torch.cuda.synchronize()
    check_status()
    ref, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(d_to_bits(d32.to(torch.bfloat16)), ref, what="debug build f32 output")


@pytest.mark.parametrize("plan", ["auto", "one_cta_128", "split4_256", "pair", "pair_deferred"])
def test_contiguous_debug_build(debug_lib, plan):
    _plan(debug_lib, plan)
    p = wl.contiguous([130, 0, 256, 77], n=264, k=640, seed=7201)
    got = d_to_bits(run_contiguous(p))
    ref, _ = oracle.grouped_contiguous(p.A, 0, p.sA, p.B, 0, p.sB, p.m_indices,
                                       np.full((p.M, p.n), SENTINEL, np.uint16))
    pad = p.m_indices < 0
    assert np.array_equal(got[pad], ref[pad]), "padding rows were written"
    compare(got[~pad], ref[~pad], what=f"debug build contiguous {plan}")


@pytest.mark.parametrize("plan", ["auto", "one_cta_256", "pair", "pair_deferred"])
def test_masked_debug_build(debug_lib, plan):
    _plan(debug_lib, plan)
    p = wl.masked(3, 384, n=520, k=768, seed=7301, masked_m=[0, 129, 384])
    got = d_to_bits(run_masked(p))
    ref, _ = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m,
                                   np.full((p.G, p.M_cap, p.n), SENTINEL, np.uint16))
    valid = np.arange(p.M_cap)[None, :] < p.masked_m[:, None]
    assert np.array_equal(got[~valid], ref[~valid]), "rows past the count were written"
    compare(got[valid], ref[valid], what=f"debug build masked {plan}")


@pytest.mark.parametrize("plan", ["auto", "one_cta_256", "pair", "pair_deferred"])
def test_k_grouped_debug_build(debug_lib, plan):
    _plan(debug_lib, plan)
    ks = [128, 0, 384, 256]
    p = wl.k_grouped(300, 520, ks, seed=7401, K=896)
    A, B = dev(p.A, fp8_dtype(0)), dev(p.B, fp8_dtype(0))
    sA, sB = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB)
    D = torch.empty((len(ks), p.m, p.n), dtype=torch.bfloat16, device="cuda")
    fg.fg_k_grouped_gemm_fp8_nt(A, sA, B, sB, D, dev(np.array(ks, np.int32)))
    torch.cuda.synchronize()
    check_status()
    ref, _ = oracle.k_grouped(p.A, 0, p.sA, p.B, 0, p.sB, np.array(ks, np.int32))
    compare(d_to_bits(D), ref, what=f"debug build k-grouped {plan}")


@pytest.mark.parametrize("plan", ["one_cta_256", "split4_256", "pair", "pair_deferred"])
def test_load_coordinate_past_k_is_caught(debug_lib, plan):
    """The hook moves one A load of every CTA past K: the box check records
    FG_ERR_DEVICE_CHECK with the A tag and the load is never issued (had it
    been, TMA would only have read zeros there: the coordinate stays aligned).
    The CTAs leave through the abort flag and their bounded waits; the next
    call is exact."""
    _plan(debug_lib, plan)
    fg.fg_set_watchdog_ms(300)
    p = wl.dense(512, 1024, 1024, seed=7501)
    assert fg.fg_get_device_status()[0] == fg.FG_OK
    debug_lib.fg_debug_bad_coordinate(1)  # every CTA runs at least two K iterations here
    A, B = dev(p.A, fp8_dtype(0)), dev(p.B, fp8_dtype(0))
    sA, sB = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB)
    D = torch.empty((p.m, p.n), dtype=torch.bfloat16, device="cuda")
    fg.fg_gemm_fp8_nt(A, sA, B, sB, D)
    st, detail = fg.fg_get_device_status()
    assert st == 6, fg.STATUS_NAMES.get(st, st)
    assert detail >> 24 == DBG_TMA_A, hex(detail)
    assert detail & 0xFFFFFF >= p.k, hex(detail)  # the offending x coordinate
    ref, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(d_to_bits(run_dense(p)), ref, what=f"after the caught coordinate ({plan})")


@pytest.mark.parametrize("case", range(48))
def test_random_calls_on_debug_build(debug_lib, case):
    """Seeded random calls (every layout, FP8 formats, BF16 or FP32 output,
    forced tile plans) through the debug build: each matches the oracle and
    leaves the status word clean, so no box, ring-index or TMEM-column check
    fired on any of the ragged shapes."""
    from random_cases import random_case, reset_knobs

    try:
        if not random_case(case, rng_base=880_000, seed_base=9000):
            pytest.skip("no rows drawn")
    finally:
        reset_knobs()
