"""GPU parity of the K-grouped GEMM (groups as 128-aligned segments of K, the
MoE weight-gradient contraction) against the CPU oracle, through the C ABI:
element-wise values within the tolerance for BF16 and FP32 output, empty
segments give zeros, each group equals a dense call on its K slice, the
device-side segment lengths are graph-replayable, bad lengths are reported,
and the workload-sized case on sampled outputs (every element of the corner
and boundary tiles of the first and the last group's output plane, random and
corner elements of every tile of the others)."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_nt_gb300 as fg
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_common import (ELEM_REL, AGG_REL, check_status, compare, d_to_bits, dev, fp8_dtype,  # noqa: E402
                        run_dense, sample_positions)


def _run(p, ks, f32=False, b_fmt=0):
    A, B = dev(p.A, fp8_dtype(0)), dev(p.B, fp8_dtype(b_fmt))
    sA, sB = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB)
    G = len(ks)
    dt = torch.float32 if f32 else torch.bfloat16
    D = torch.full((G, p.m, p.n), float("nan"), dtype=dt, device="cuda")
    f = fg.fg_k_grouped_gemm_fp8_nt_f32out if f32 else fg.fg_k_grouped_gemm_fp8_nt
    f(A, sA, B, sB, D, dev(np.asarray(ks, np.int32)))
    torch.cuda.synchronize()
    check_status()
    return D


def _compare_f32(got, ref64, what):
    g = got.astype(np.float64)
    assert np.all(np.isfinite(g)), what
    tol = ELEM_REL * float(np.max(np.abs(ref64))) + 1e-30
    assert np.max(np.abs(g - ref64)) <= tol, what
    nr = float(np.linalg.norm(ref64))
    if nr > 0:
        assert float(np.linalg.norm(g - ref64)) / nr <= AGG_REL, what


PLANS = ["auto", "one_cta_256", "cta_pair", "cta_pair_deferred"]


@pytest.fixture(params=PLANS)
def plan(request):
    """The tile plans of the K-grouped call: the automatic choice, one-CTA
    128 x 256 tiles, and 256 x 256 tiles on CTA pairs with the promotion
    warps storing or with the store warp (forced even where M < 256)."""
    name = request.param
    if name != "auto":
        fg.fg_set_config_override(256, 1)
        fg.fg_set_pair_mode(0 if name == "one_cta_256" else 1)
        fg.lib().fg_debug_set_pair_defer(1 if name == "cta_pair_deferred" else 0)
    yield name
    fg.fg_set_config_override(0, 0)
    fg.fg_set_pair_mode(-1)
    fg.lib().fg_debug_set_pair_defer(-1)


@pytest.mark.parametrize("M,N,ks,K", [
    (200, 264, [128, 0, 256, 384], 896),      # ragged M and N, an empty group, 128 unused K columns
    (128, 256, [512], 512),
    (1, 8, [128, 128], 256),
    (300, 520, [0, 0, 1024], 1040),           # K not a multiple of 128 (the tail is unused)
    (257, 2112, [128] * 9, 1152),             # nine groups, the sweep's ragged N
])
@pytest.mark.parametrize("f32", [False, True])
def test_k_grouped_small_full(M, N, ks, K, f32, plan):
    p = wl.k_grouped(M, N, ks, seed=M + N + K + len(ks), K=K)
    D = _run(p, ks, f32)
    ref16, ref64 = oracle.k_grouped(p.A, 0, p.sA, p.B, 0, p.sB, np.array(ks, np.int32))
    for g, kg in enumerate(ks):
        if kg == 0:
            assert torch.count_nonzero(D[g]).item() == 0, f"group {g}: empty segment must give zeros"
    if f32:
        _compare_f32(D.cpu().numpy(), ref64, f"k-grouped f32 {M}x{N} {ks}")
    else:
        compare(d_to_bits(D), ref16, what=f"k-grouped {M}x{N} {ks}")


def test_k_grouped_f32_rounds_to_the_bf16_call():
    p = wl.k_grouped(256, 512, [256, 384], seed=71)
    d32 = _run(p, [256, 384], f32=True)
    d16 = _run(p, [256, 384])
    assert torch.equal(d32.to(torch.bfloat16).view(torch.int16), d16.view(torch.int16))


def test_k_grouped_each_group_equals_dense_on_its_slice():
    """Group g equals the dense call on the K slice of A, B and the scales,
    bitwise when both use the same tile plan (128 x 256 persistent)."""
    ks = [256, 128, 384]
    p = wl.k_grouped(384, 768, ks, seed=72)
    fg.fg_set_config_override(256, 1)
    try:
        D = d_to_bits(_run(p, ks))
        off = 0
        for g, kg in enumerate(ks):
            b0, b1 = off // 128, (off + kg) // 128
            d = wl.Dense(p.m, p.n, kg, np.ascontiguousarray(p.A[:, off:off + kg]),
                         np.ascontiguousarray(p.sA[:, b0:b1]), np.ascontiguousarray(p.B[:, off:off + kg]),
                         np.ascontiguousarray(p.sB[:, b0:b1]))
            assert np.array_equal(D[g], d_to_bits(run_dense(d))), f"group {g}"
            off += kg
    finally:
        fg.fg_set_config_override(0, 0)


def test_k_grouped_graph_replay_reads_new_segment_lengths(plan):
    """The lengths live on the device: a captured call replayed after they
    change gives the result of the new lengths."""
    p = wl.k_grouped(128, 256, [512], seed=73, K=512)
    A, B = dev(p.A, fp8_dtype(0)), dev(p.B, fp8_dtype(0))
    sA, sB = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB)
    ks = torch.tensor([128, 384], dtype=torch.int32, device="cuda")
    D = torch.empty((2, 128, 256), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    fg.fg_k_grouped_gemm_fp8_nt(A, sA, B, sB, D, ks, stream=s)  # first call on this device outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fg.fg_k_grouped_gemm_fp8_nt(A, sA, B, sB, D, ks, stream=s)
    for new in ([384, 128], [0, 512], [256, 0]):
        ks.copy_(torch.tensor(new, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        check_status()
        ref16, _ = oracle.k_grouped(p.A, 0, p.sA, p.B, 0, p.sB, np.array(new, np.int32))
        compare(d_to_bits(D), ref16, what=f"graph replay {new}")


@pytest.mark.parametrize("ks,detail", [([100, 128], 0), ([128, -128], 1), ([256, 384], 2)])
def test_k_grouped_bad_segment_lengths_are_reported(ks, detail, plan):
    """A length that is not a multiple of 128, a negative one, or lengths that
    sum past K are recorded as FG_ERR_DEVICE_CHECK (detail: the group, or G for
    the sum); nothing faults and the next call is clean."""
    p = wl.k_grouped(128, 256, [512], seed=74, K=512)
    A, B = dev(p.A, fp8_dtype(0)), dev(p.B, fp8_dtype(0))
    sA, sB = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB)
    D = torch.empty((2, 128, 256), dtype=torch.bfloat16, device="cuda")
    fg.fg_k_grouped_gemm_fp8_nt(A, sA, B, sB, D, dev(np.array(ks, np.int32)))
    st, det = fg.fg_get_device_status()
    assert st == 6 and det == detail
    fg.fg_k_grouped_gemm_fp8_nt(A, sA, B, sB, D, dev(np.array([128, 384], np.int32)))
    check_status()


@pytest.mark.parametrize("G,M,N,tokens", wl.k_grouped_shapes()[:2] + wl.k_grouped_short_shapes())
def test_k_grouped_workload(G, M, N, tokens):
    """The weight gradient of the contiguous workload (G experts of 8192 tokens;
    or 32 experts of 512, the short-segment plan on CTA pairs with the store
    warp), M = n, N = k of the forward weight, checked on sampled outputs of
    every group's plane (the first and last planes' corner and boundary tiles
    in full)."""
    ks = [tokens] * G
    shapes = wl.k_grouped_shapes() + wl.k_grouped_short_shapes()
    p = wl.k_grouped(M, N, ks, seed=wl.seed_for(6, shapes.index((G, M, N, tokens))))
    D = d_to_bits(_run(p, ks))
    full = sample_positions(M, N, seed=G + M, n_rows_full=2, boundary_tiles=True)
    light = sample_positions(M, N, seed=G + M + 1, n_rows_full=2)
    picks = [full if g in (0, G - 1) else light for g in range(G)]  # first and last plane in full
    gs = np.concatenate([np.full(pk[0].size, g, np.int64) for g, pk in enumerate(picks)])
    rr = np.concatenate([pk[0] for pk in picks])
    cc = np.concatenate([pk[1] for pk in picks])
    ref16, _ = oracle.k_grouped_at(p.A, 0, p.sA, p.B, 0, p.sB, np.array(ks, np.int32), gs, rr, cc)
    compare(D[gs, rr, cc], ref16, what=f"k-grouped G={G} {M}x{N} (sampled)")


@pytest.mark.parametrize("G,M,N,K,want", [
    (4, 4096, 7168, 4 * 8192, (256, 1, 1, 0, 0)),    # segments of 64 K blocks: CTA pairs, promotion warps store
    (8, 4096, 7168, 8 * 2048, (256, 1, 1, 0, 0)),    # segments of 16: the same
    (8, 4096, 7168, 8 * 1536, (256, 1, 1, 0, 1)),    # segments of 12: CTA pairs with the store warp
    (8, 4096, 2048, 8 * 1024, (256, 1, 1, 0, 1)),    # segments of 8: CTA pairs with the store warp
    (2, 128, 512, 2 * 1024, (128, 1, 0, 0, 0)),      # a few one-CTA tiles: 128 wide
    (8, 200, 4096, 8 * 512, (256, 1, 0, 0, 0)),      # fewer than 256 rows: one-CTA tiles
    (32, 4096, 7168, 32 * 256, (256, 1, 1, 0, 0)),   # segments of 2 K blocks: pairs, promotion warps store
])
def test_k_grouped_plan_query(G, M, N, K, want):
    got = fg.fg_query_plan(3, M, G, N, K)
    assert tuple(got) == want, got


def test_k_grouped_pair_tiles_workload_sampled():
    """CTA-pair tiles with the store warp on a workload-shaped call whose
    segments are short and ragged (an empty one among them), sampled outputs
    of every plane, and the same call on one-CTA tiles agreeing within the
    tolerance on the same samples."""
    ks = [1024, 0, 384, 2048, 128, 896, 1536, 256]
    M, N = 2304, 3072
    p = wl.k_grouped(M, N, ks, seed=75)
    assert fg.fg_query_plan(3, M, len(ks), N, p.k)[2:] == (1, 0, 1)
    D = d_to_bits(_run(p, ks))
    pk = sample_positions(M, N, seed=76, n_rows_full=2, boundary_tiles=True)
    gs = np.repeat(np.arange(len(ks)), pk[0].size)
    rr, cc = np.tile(pk[0], len(ks)), np.tile(pk[1], len(ks))
    ref16, _ = oracle.k_grouped_at(p.A, 0, p.sA, p.B, 0, p.sB, np.array(ks, np.int32), gs, rr, cc)
    compare(D[gs, rr, cc], ref16, what="k-grouped pair tiles (sampled)")
    assert not np.any(D[1]), "empty segment must give zeros"


@pytest.mark.parametrize("plan", ["auto", "one_cta_256", "cta_pair_deferred"])
def test_k_grouped_many_short_segments(plan):
    """128 groups of one or two K blocks each (and some empty ones): every
    role's forward scan over the segment lengths walks all 128 groups, full
    comparison with the oracle."""
    name = plan
    if name != "auto":
        fg.fg_set_config_override(256, 1)
        fg.fg_set_pair_mode(0 if name == "one_cta_256" else 1)
        fg.lib().fg_debug_set_pair_defer(1 if name == "cta_pair_deferred" else 0)
    try:
        rng = wl.rng_for(77)
        ks = (rng.integers(0, 3, size=128) * 128).tolist()
        ks[:3] = [0, 256, 128]
        p = wl.k_grouped(288, 264, ks, seed=78)
        D = _run(p, ks)
    finally:
        fg.fg_set_config_override(0, 0)
        fg.fg_set_pair_mode(-1)
        fg.lib().fg_debug_set_pair_defer(-1)
    ref16, _ = oracle.k_grouped(p.A, 0, p.sA, p.B, 0, p.sB, np.array(ks, np.int32))
    compare(d_to_bits(D), ref16, what=f"k-grouped 128 short segments ({plan})")
