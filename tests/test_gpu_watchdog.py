"""Failure detection without a GPU fault: a test hook makes every CTA's
producer leave one K iteration unarmed, so a consumer's bounded mbarrier wait
runs out.  The kernel must record FG_ERR_TIMEOUT in the device status word,
drain what it issued, free its tensor memory and return; the context stays
usable and the next call is correct."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_nt_gb300 as fg
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_common import compare, d_to_bits, dev, fp8_dtype, run_dense  # noqa: E402


@pytest.fixture(params=[0, 1, 2], ids=["one_cta", "cta_pair_deferred_stores", "cta_pair"])
def short_watchdog(request):
    """Persistent 128x256 tiles on one CTA, or 256x256 tiles on CTA pairs
    (with the store warp, or with the promotion warps storing)."""
    fg.fg_set_watchdog_ms(200)
    fg.fg_set_config_override(256, 1)
    fg.fg_set_pair_mode(1 if request.param else 0)
    fg.lib().fg_debug_set_pair_defer(1 if request.param == 1 else 0)
    yield
    fg.fg_set_watchdog_ms(0)
    fg.fg_set_config_override(0, 0)
    fg.fg_set_pair_mode(-1)
    fg.lib().fg_debug_set_pair_defer(-1)
    fg.lib().fg_debug_skip_producer_iteration(-1)


def _launch(p):
    A = dev(p.A, fp8_dtype(0))
    D = torch.zeros((p.m, p.n), dtype=torch.bfloat16, device="cuda")
    fg.fg_gemm_fp8_nt(A, fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.B, fp8_dtype(0)), dev(p.sB), D)
    return D


@pytest.mark.parametrize("skip_iter", [0, 3, 7])  # each CTA runs 8 K iterations here
def test_unarmed_stage_times_out_and_context_survives(short_watchdog, skip_iter):
    p = wl.dense(512, 1024, 1024, seed=90)
    st, _ = fg.fg_get_device_status()
    assert st == fg.FG_OK
    fg.lib().fg_debug_skip_producer_iteration(skip_iter)
    _launch(p)
    st, detail = fg.fg_get_device_status()
    assert st == 5, fg.STATUS_NAMES.get(st, st)  # FG_ERR_TIMEOUT
    assert (detail >> 24) in (1, 2, 3)           # the role whose wait ran out
    # the hook is one-shot and the GPU context is intact: the next call is exact
    got = d_to_bits(run_dense(p))
    ref, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(got, ref, what="after watchdog")
    st, _ = fg.fg_get_device_status()
    assert st == fg.FG_OK


def test_status_is_cleared_by_reading():
    st, _ = fg.fg_get_device_status()
    assert st == fg.FG_OK


@pytest.mark.parametrize("x_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("skip_unit", [0, 5])
def test_quantizer_unfilled_stage_times_out_and_context_survives(skip_unit, x_dtype):
    """The quantizer's producer leaves one unit unfilled in every CTA: the
    consumers' bounded wait expires, the CTA drains the copies it issued and
    returns, and the next call is bit-exact (BF16 and FP32 input)."""
    x = wl.activations((4096, 1024), seed=91)  # 1024 units of 32 rows x 128 columns
    X = torch.from_numpy(x).to(x_dtype).cuda()
    fg.fg_set_watchdog_ms(200)
    fg.fg_set_num_sms(4)  # a few persistent CTAs, each with many units
    try:
        assert fg.fg_get_device_status()[0] == fg.FG_OK
        fg.lib().fg_debug_skip_producer_iteration(skip_unit)
        fg.fg_quantize_fp8_per_token(X)
        st, detail = fg.fg_get_device_status()
        assert st == 5, fg.STATUS_NAMES.get(st, st)  # FG_ERR_TIMEOUT
        assert (detail >> 24) in (1, 3)              # producer or consumer wait
    finally:
        fg.fg_set_watchdog_ms(0)
        fg.fg_set_num_sms(0)
        fg.lib().fg_debug_skip_producer_iteration(-1)
    A, sA = fg.fg_quantize_fp8_per_token(X)
    q, s = oracle.quantize_per_token(x, wl.E4M3)
    assert np.array_equal(A.view(torch.uint8).cpu().numpy(), q)
    assert np.array_equal(sA[:, :4096].cpu().numpy(), s.T)
    assert fg.fg_get_device_status()[0] == fg.FG_OK
