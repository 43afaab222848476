"""GPU parity of the dense FP8 NT GEMM against the CPU oracle, through the C ABI.

Small problems are compared element by element over the whole output; the
full-size workloads (the dense sweep m in {64,128,4096} x five (n,k) weight
shapes, and the 8192^3 problems) are compared on sampled outputs computed by
the oracle one by one, plus properties that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, but never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_common import (bits_to_f32, compare, d_to_bits, run_dense, sample_positions)  # noqa: E402


def _full_check(p, what):
    D = run_dense(p)
    ref16, _ = oracle.gemm_fp8_nt(p.A, p.a_fmt, p.sA, p.B, p.b_fmt, p.sB, want_f64=False)
    return compare(d_to_bits(D), ref16, what=what)


def test_small_dense_128x256x512():
    p = wl.small_dense()
    _full_check(p, "dense 128x256x512")


BOUNDARY = [
    (1, 8, 16), (1, 256, 128), (63, 64, 112), (64, 136, 144), (65, 264, 128), (127, 256, 256),
    (128, 8, 640), (129, 520, 384), (200, 2112, 272), (300, 128, 1280), (2, 7168, 16),
    (257, 256, 1040), (384, 768, 128 * 7),
]


@pytest.mark.parametrize("m,n,k", BOUNDARY)
def test_boundary_shapes(m, n, k):
    """Partial M, N and K tiles, k not a multiple of 128, single-column-block n."""
    p = wl.dense(m, n, k, seed=5000 + m * 7 + n * 3 + k)
    _full_check(p, f"dense {m}x{n}x{k}")


def test_p1_regression_shape_6144_1280():
    """The tutorial's intermittent failure shape M = N = 6144, K = 1280 (page
    "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践", section 6), checked on sampled outputs,
    three times in a row."""
    p = wl.dense(6144, 6144, 1280, seed=4242)
    rows, cols = sample_positions(p.m, p.n, seed=1, n_rows_full=4)
    ref16, _ = oracle.gemm_fp8_nt_at(p.A, 0, p.sA, p.B, 0, p.sB, rows, cols)
    first = None
    for _ in range(3):
        g = d_to_bits(run_dense(p))
        compare(g[rows, cols], ref16, what="dense 6144^2 x 1280")
        if first is None:
            first = g
        else:
            assert np.array_equal(first, g), "results differ between identical calls"


@pytest.mark.parametrize("m", wl.DENSE_SWEEP_M)
@pytest.mark.parametrize("n,k", wl.DENSE_SWEEP_NK)
def test_dense_sweep(m, n, k):
    """The dense sweep workload at full size."""
    p = wl.dense(m, n, k, seed=wl.seed_for(1, wl.DENSE_SWEEP_NK.index((n, k))))
    g = d_to_bits(run_dense(p))
    if m <= 128:
        ref16, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
        compare(g, ref16, what=f"dense {m}x{n}x{k}")
    else:
        rows, cols = sample_positions(m, n, seed=m + n + k, n_rows_full=8)
        ref16, _ = oracle.gemm_fp8_nt_at(p.A, 0, p.sA, p.B, 0, p.sB, rows, cols)
        compare(g[rows, cols], ref16, what=f"dense {m}x{n}x{k} (sampled)")


@pytest.mark.parametrize("m,n,k,b_fmt", wl.large_dense_shapes())
def test_large_square_loguniform_scales(m, n, k, b_fmt):
    """8192^3 (and the K-tail k = 8576, and E5M2 B) with scales drawn
    log-uniform in [2^-8, 2^8] to stress the FP32 promotion."""
    p = wl.dense(m, n, k, seed=wl.seed_for(4, int(k != 8192) + 2 * b_fmt), b_fmt=b_fmt, scales="loguniform")
    g = d_to_bits(run_dense(p))
    rows, cols = sample_positions(m, n, seed=k + b_fmt, n_rows_full=4, boundary_tiles=True)
    ref16, _ = oracle.gemm_fp8_nt_at(p.A, 0, p.sA, p.B, b_fmt, p.sB, rows, cols)
    compare(g[rows, cols], ref16, what=f"dense {m}x{n}x{k} b_fmt={b_fmt} (sampled)")


def test_e5m2_both_operands_small():
    p = wl.dense(130, 264, 384, seed=77, b_fmt=wl.E5M2, a_fmt=wl.E5M2)
    _full_check(p, "dense e5m2 x e5m2")


def test_power_of_two_scale_linearity_bitwise():
    """D(2^e * sA) == 2^e * D(sA) exactly (FP32 promotion is exact under
    power-of-two scaling barring overflow/underflow)."""
    p = wl.dense(256, 512, 640, seed=31)
    base = bits_to_f32(d_to_bits(run_dense(p)))
    for e in (-4, 3):
        q = wl.Dense(p.m, p.n, p.k, p.A, p.sA * np.float32(2.0 ** e), p.B, p.sB)
        out = bits_to_f32(d_to_bits(run_dense(q)))
        assert np.array_equal(out, base * np.float32(2.0 ** e))


def test_zero_scale_block_vanishes():
    p = wl.dense(128, 256, 384, seed=32)
    sA = p.sA.copy()
    sA[:, 1] = 0
    A2 = p.A.copy()
    A2[:, 128:256] = 0
    a = d_to_bits(run_dense(wl.Dense(p.m, p.n, p.k, p.A, sA, p.B, p.sB)))
    b = d_to_bits(run_dense(wl.Dense(p.m, p.n, p.k, A2, p.sA, p.B, p.sB)))
    assert np.array_equal(a, b)
    z = d_to_bits(run_dense(wl.Dense(p.m, p.n, p.k, p.A, np.zeros_like(p.sA), p.B, p.sB)))
    assert np.all((z & 0x7FFF) == 0)


def test_output_guard_bands_untouched():
    """D inside a larger buffer: the bytes before and after D stay as they were."""
    p = wl.dense(100, 264, 256, seed=33)
    guard = 4096
    buf = torch.full((guard + p.m * p.n + guard,), 0x5A5A, dtype=torch.int16, device="cuda")
    D = buf[guard:guard + p.m * p.n].view(torch.bfloat16).view(p.m, p.n)
    run_dense(p, D=D)
    host = buf.cpu().numpy()
    assert np.all(host[:guard] == 0x5A5A) and np.all(host[-guard:] == 0x5A5A)
    ref16, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(d_to_bits(D), ref16, what="guarded D")


def test_repeatable_bitwise():
    p = wl.dense(512, 1024, 2048, seed=34)
    a = d_to_bits(run_dense(p))
    for _ in range(5):
        assert np.array_equal(a, d_to_bits(run_dense(p)))


@pytest.fixture
def plan_override():
    import moe_grouped_gemm_nt_gb300 as fg

    yield fg.fg_set_config_override
    fg.fg_set_config_override(0, 0)


@pytest.mark.parametrize("bn,split", [(256, 1), (128, 1), (256, 2), (256, 3), (128, 4), (128, 5), (256, 8),
                                      (128, 8)])
@pytest.mark.parametrize("m,n,k", [(130, 520, 1280), (64, 2112, 1024), (1, 264, 400)])
def test_forced_plans_match_oracle(plan_override, bn, split, m, n, k):
    """Every tile plan (tile width x split-K cluster size, including ranks with
    no K blocks when split > K blocks) gives the oracle's result."""
    plan_override(bn, split)
    p = wl.dense(m, n, k, seed=7000 + m + n + k)
    _full_check(p, f"dense {m}x{n}x{k} bn={bn} split={split}")


def test_split_plans_agree_and_repeat(plan_override):
    """Split-K reduces in a fixed rank order: repeated calls are bitwise equal."""
    p = wl.dense(128, 4096, 7168, seed=71)
    plan_override(128, 4)
    a = d_to_bits(run_dense(p))
    for _ in range(3):
        assert np.array_equal(a, d_to_bits(run_dense(p)))
    plan_override(256, 1)
    b = d_to_bits(run_dense(p))
    ref16, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(a, ref16, what="split 4")
    compare(b, ref16, what="persistent")


def test_programmatic_launch_keeps_stream_order():
    """Back-to-back calls on one stream, with programmatic dependent launch on:
    a call that overwrites the previous call's output (write after write), and a
    call whose inputs were just written by the previous kernel (read after
    write), give the same bits as with the launches fully serialized."""
    import moe_grouped_gemm_nt_gb300 as fg
    from gpu_common import dev, fp8_dtype

    p1 = wl.dense(128, 4096, 7168, seed=81)   # split-K plan
    p2 = wl.dense(128, 4096, 7168, seed=82)
    p3 = wl.dense(1024, 2048, 2048, seed=83)  # persistent plan
    def args(p):
        return (dev(p.A, fp8_dtype(0)), fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.B, fp8_dtype(0)), dev(p.sB))
    a1, a2, a3 = args(p1), args(p2), args(p3)
    results = {}
    for pdl in (False, True):
        fg.fg_set_programmatic_launch(pdl)
        try:
            D = torch.empty((128, 4096), dtype=torch.bfloat16, device="cuda")
            A3 = torch.empty_like(a3[0])
            D3 = torch.empty((1024, 2048), dtype=torch.bfloat16, device="cuda")
            for _ in range(3):
                fg.fg_gemm_fp8_nt(*a1, D)
                fg.fg_gemm_fp8_nt(*a2, D)          # must land after the first
                A3.copy_(a3[0])                     # written right before the next call reads it
                fg.fg_gemm_fp8_nt(A3, a3[1], a3[2], a3[3], D3)
                fg.fg_gemm_fp8_nt(*a1, D)
            torch.cuda.synchronize()
            results[pdl] = (d_to_bits(D), d_to_bits(D3))
        finally:
            fg.fg_set_programmatic_launch(True)
    assert np.array_equal(results[False][0], results[True][0])
    assert np.array_equal(results[False][1], results[True][1])
    ref1, _ = oracle.gemm_fp8_nt(p1.A, 0, p1.sA, p1.B, 0, p1.sB, want_f64=False)
    compare(results[True][0], ref1, what="last writer wins")


# ------------------------------------------------------------- CTA pairs

@pytest.fixture
def pair_mode():
    import moe_grouped_gemm_nt_gb300 as fg

    yield fg.fg_set_pair_mode
    fg.fg_set_pair_mode(-1)


@pytest.mark.parametrize("m,n,k", [(256, 512, 640), (300, 264, 1040), (384, 520, 384), (1, 256, 128),
                                   (640, 2112, 272), (1030, 1800, 1536)])
def test_pair_tiles_match_oracle(pair_mode, m, n, k):
    """256 x 256 tiles on CTA pairs (forced for every persistent 256-wide plan,
    including m < 256 where the odd CTA's half is empty): full comparison,
    partial M, N and K tiles included."""
    import moe_grouped_gemm_nt_gb300 as fg

    pair_mode(1)
    bn, split, pair = fg.fg_query_dense_plan_ex(m, n, k)
    p = wl.dense(m, n, k, seed=9100 + m + n + k)
    _full_check(p, f"dense pair {m}x{n}x{k} (plan {bn},{split},{pair})")


def test_pair_and_single_cta_tiles_agree(pair_mode):
    """The same problem on CTA pairs and on one-CTA tiles: both within the
    oracle tolerance, and repeated pair calls bitwise equal."""
    p = wl.dense(1024, 2048, 2048, seed=9201)
    ref16, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    pair_mode(1)
    a = d_to_bits(run_dense(p))
    assert np.array_equal(a, d_to_bits(run_dense(p)))
    pair_mode(0)
    b = d_to_bits(run_dense(p))
    compare(a, ref16, what="pair")
    compare(b, ref16, what="single")


def test_pair_plan_query():
    import moe_grouped_gemm_nt_gb300 as fg

    assert fg.fg_query_dense_plan_ex(4096, 7168, 2048)[2] == 1
    assert fg.fg_query_dense_plan_ex(128, 7168, 2048)[2] == 0
    # BF16 pair tiles of at most 56 K blocks store through the eleventh warp
    assert fg.fg_query_plan(0, 4096, 1, 7168, 2048)[2:] == (1, 0, 1)
    assert fg.fg_query_plan(0, 4096, 1, 4096, 7168)[2:] == (1, 0, 1)
    assert fg.fg_query_plan(0, 4096, 1, 7168, 7296)[2:] == (1, 0, 0)
    assert fg.fg_query_plan(0, 4096, 1, 7168, 16384)[2:] == (1, 0, 0)


@pytest.mark.parametrize("m,n,k", [(640, 2112, 1536), (300, 520, 2048), (1030, 1800, 640), (512, 768, 4096)])
def test_pair_deferred_stores_are_bitwise_the_same(pair_mode, m, n, k):
    """Staging a whole tile and storing it from the eleventh warp changes only
    who issues the TMA stores: the bits equal those of the promotion warps'
    own stores, dense and masked, short and long K."""
    import moe_grouped_gemm_nt_gb300 as fg
    from gpu_common import run_masked

    pair_mode(1)
    p = wl.dense(m, n, k, seed=9150 + m + k)
    q = wl.masked(3, 512, n=n, k=k, seed=9160 + k, masked_m=[0, 300, 512])
    outs = []
    try:
        for mode in (0, 1):
            assert fg.lib().fg_debug_set_pair_defer(mode) == 0
            outs.append((d_to_bits(run_dense(p)), d_to_bits(run_masked(q))))
    finally:
        fg.lib().fg_debug_set_pair_defer(-1)
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    ref16, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(outs[1][0], ref16, what=f"deferred stores {m}x{n}x{k}")


@pytest.mark.parametrize("mode,bn,split", [("pair", 0, 0), ("one_cta", 256, 1), ("split", 128, 4)])
def test_repeat_20x_bitwise(pair_mode, plan_override, mode, bn, split):
    """Twenty identical calls give identical bits (a race in a pipeline, a
    barrier phase or the split-K exchange would show up as run-to-run noise)."""
    if mode == "pair":
        pair_mode(1)
    else:
        pair_mode(0)
        plan_override(bn, split)
    p = wl.dense(768 if mode != "split" else 128, 2112, 3072, seed=9300 + bn + split)
    first = d_to_bits(run_dense(p))
    for _ in range(19):
        assert np.array_equal(first, d_to_bits(run_dense(p))), mode
    ref16, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    compare(first, ref16, what=f"repeat {mode}")


@pytest.mark.parametrize("m", [640, 128])
@pytest.mark.parametrize("num_sms", [1, 2, 16, 77])
def test_sm_limit(pair_mode, num_sms, m):
    """fg_set_num_sms caps the grid (persistent one-CTA and CTA-pair tiles;
    split-K plans only where they fit the limit); the results stay exact."""
    import moe_grouped_gemm_nt_gb300 as fg

    p = wl.dense(m, 1040, 1024, seed=9400 + num_sms + m)
    ref16, _ = oracle.gemm_fp8_nt(p.A, 0, p.sA, p.B, 0, p.sB, want_f64=False)
    fg.fg_set_num_sms(num_sms)
    try:
        for mode in (0, 1):
            pair_mode(mode)
            compare(d_to_bits(run_dense(p)), ref16, what=f"sms={num_sms} pair={mode}")
    finally:
        fg.fg_set_num_sms(0)
