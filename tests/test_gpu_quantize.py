"""GPU parity of the per-token FP8 activation quantizer against the CPU oracle.

The FP8 codes and the scales are integers and floats decided by float32
arithmetic on both sides, so the bar is bit-exactness: every byte of A and
every scale of sA equal the oracle's.  Rows and padding the call must not
touch are pre-filled with sentinels (0x7F is an E4M3 NaN and 0x7F an E5M2 NaN,
which a saturating conversion of finite values never produces) and checked to
survive.  The quantizer then feeds the GEMM kernels, and a CUDA graph replays
the quantize + masked-GEMM pair with new device-side counts."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_nt_gb300 as fg
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_common import SENTINEL, compare, d_to_bits, dev, fp8_dtype  # noqa: E402

A_SENTINEL = 0x7F
SA_SENTINEL_BITS = 0x7FCADBAD  # a quiet-NaN pattern no scale can take (filled through an int32 view)


def _x_device(x, ld_x=None, dtype=torch.bfloat16):
    """float32 [.., rows, k] (bfloat16-valued for a bfloat16 X) -> CUDA tensor of
    `dtype` with row pitch ld_x."""
    *lead, rows, k = x.shape
    ld_x = k if ld_x is None else ld_x
    full = np.zeros((*lead, rows, ld_x), np.float32)
    full[..., :k] = x
    if ld_x > k:
        full[..., k:] = 1.0e30  # columns past k must not reach any group maximum
    t = torch.from_numpy(full).to(dtype).cuda()
    return t[..., :k]


def _run(x, fmt, ld_x=None, masked_m=None, ld_sa=None, dtype=torch.bfloat16):
    *lead, rows, k = x.shape
    kb = (k + 127) // 128
    ld_sa = fg.fg_scales_a_ld(rows) if ld_sa is None else ld_sa
    X = _x_device(x, ld_x, dtype)
    A = torch.full((*lead, rows, k), A_SENTINEL, dtype=torch.uint8, device="cuda")
    sA = torch.full((*lead, kb, ld_sa), SA_SENTINEL_BITS, dtype=torch.int32, device="cuda").view(torch.float32)
    mm = None if masked_m is None else torch.tensor(masked_m, dtype=torch.int32, device="cuda")
    A_out, sA_out = fg.fg_quantize_fp8_per_token(X, A.view(fp8_dtype(fmt)), sA, fmt=fmt, masked_m=mm)
    assert A_out.data_ptr() == A.data_ptr() and sA_out.data_ptr() == sA.data_ptr()
    torch.cuda.synchronize()
    return A.cpu().numpy(), sA.cpu().numpy()


def _check_against_oracle(x, fmt, A, sA, limits=None):
    """Bit-exact A and sA on the valid rows; sentinels everywhere else."""
    xb = x.reshape(-1, *x.shape[-2:])
    A = A.reshape(-1, *A.shape[-2:])
    sA = sA.reshape(-1, *sA.shape[-2:])
    rows = xb.shape[1]
    q, s = oracle.quantize_per_token(xb, fmt)
    for b in range(xb.shape[0]):
        lim = rows if limits is None else limits[b]
        assert np.array_equal(A[b, :lim], q[b, :lim]), f"batch {b}: FP8 codes differ"
        assert np.array_equal(sA[b, :, :lim].view(np.uint32), s[b, :lim].T.copy().view(np.uint32)), \
            f"batch {b}: scales differ"
        assert np.all(A[b, lim:] == A_SENTINEL), f"batch {b}: rows past the count were written"
        assert np.all(sA[b, :, lim:].view(np.uint32) == SA_SENTINEL_BITS), \
            f"batch {b}: scale entries past the valid rows were written"


@pytest.mark.parametrize("fmt", [wl.E4M3, wl.E5M2])
@pytest.mark.parametrize("batches,rows,k,ld_x", [
    (1, 1, 16, 16),
    (1, 31, 112, 112),      # one partial K block, fewer rows than a CTA
    (1, 32, 128, 128),
    (1, 33, 144, 160),      # a 16-wide tail block, one row in a second CTA, wider rows of X
    (1, 100, 1024, 1024),
    (1, 257, 304, 312),
    (3, 70, 256, 264),      # batches
    (2, 1, 128, 136),       # one row per batch
])
def test_quantize_small_bit_exact(fmt, batches, rows, k, ld_x):
    x = wl.activations((batches, rows, k), seed=rows * 7 + k + fmt)
    A, sA = _run(x, fmt, ld_x=ld_x)
    _check_against_oracle(x, fmt, A, sA)


@pytest.mark.parametrize("fmt", [wl.E4M3, wl.E5M2])
def test_quantize_special_values(fmt):
    """Zero rows and groups (scale 1), signed zeros, the largest BF16 values,
    BF16 subnormals (scales that are float32 subnormals), values at the
    saturation edge, and a single nonzero per group."""
    rows, k = 12, 384
    x = wl.activations((rows, k), seed=31)
    bf16_max = float(np.array([0x7F7F0000], np.uint32).view(np.float32)[0])
    tiny = float(np.array([0x00010000], np.uint32).view(np.float32)[0])  # smallest BF16 subnormal
    x[0] = 0.0
    x[1, 128:256] = 0.0
    x[2] = -0.0
    x[3, :] = bf16_max
    x[3, 1::2] = -bf16_max
    x[4, :] = tiny
    x[4, 5] = 7 * tiny
    x[5, :] = 0.0
    x[5, 17] = -3.0
    x[5, 200] = 1.0e-30
    x[6] = np.float32(1.0) + np.arange(k, dtype=np.float32) / 512  # a slow ramp
    x = np.array(torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy())
    A, sA = _run(x, fmt)
    _check_against_oracle(x, fmt, A, sA)


@pytest.mark.parametrize("fmt", [wl.E4M3, wl.E5M2])
def test_quantize_extreme_dynamic_range(fmt):
    """Magnitudes log-uniform over the whole BF16 range (2^-133 .. 2^127) with
    per-group ceilings, so groups have scales from float32 subnormals to 2^119
    and elements from far below to exactly at the group maximum: the
    quotient's rounding (including ties of the FP8 rounding and zeros of
    either sign) must match an IEEE division everywhere."""
    rng = wl.rng_for(2024 + fmt)
    rows, k = 96, 1024
    ceil = rng.uniform(-133, 127, size=(rows, k // 128, 1))
    e = ceil - rng.uniform(0, 60, size=(rows, k // 128, 128))
    x = np.exp2(np.maximum(e, -133)) * rng.choice([-1.0, 1.0], size=e.shape)
    x = x.reshape(rows, k).astype(np.float32)
    x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    A, sA = _run(x, fmt)
    _check_against_oracle(x, fmt, A, sA)


def test_quantize_walks_many_units_per_cta():
    """With the SM limit at 1 each persistent CTA walks hundreds of units."""
    x = wl.activations((2, 300, 2048), seed=16)
    fg.fg_set_num_sms(1)
    try:
        A, sA = _run(x, wl.E5M2, masked_m=[300, 123])
    finally:
        fg.fg_set_num_sms(0)
    _check_against_oracle(x, wl.E5M2, A, sA, limits=[300, 123])


def test_quantize_masked_counts():
    """Rows past each batch's device-side count stay untouched."""
    x = wl.activations((4, 96, 512), seed=8)
    counts = [0, 96, 33, 1]
    A, sA = _run(x, wl.E4M3, masked_m=counts)
    _check_against_oracle(x, wl.E4M3, A, sA, limits=counts)
    st, _ = fg.fg_get_device_status()
    assert st == fg.FG_OK


def test_quantize_masked_counts_out_of_range_are_clamped():
    x = wl.activations((3, 40, 256), seed=9)
    A, sA = _run(x, wl.E4M3, masked_m=[-3, 41, 7])
    _check_against_oracle(x, wl.E4M3, A, sA, limits=[0, 40, 7])
    st, detail = fg.fg_get_device_status()
    assert st == 6 and detail in (0, 1)
    assert fg.fg_get_device_status()[0] == fg.FG_OK  # reading clears it


@pytest.mark.parametrize("pdl", [1, 0])
def test_quantize_with_and_without_programmatic_launch(pdl):
    x = wl.activations((65, 640), seed=10)
    fg.lib().fg_set_programmatic_launch(pdl)
    try:
        A, sA = _run(x, wl.E4M3)
    finally:
        fg.lib().fg_set_programmatic_launch(1)
    _check_against_oracle(x, wl.E4M3, A, sA)


@pytest.mark.parametrize("rows,k", [(4096, 7168), (4096, 16384), (128, 7168), (64, 2048)])
def test_quantize_full_size_bit_exact(rows, k):
    """The activation shapes of the dense sweep, compared in full."""
    x = wl.activations((rows, k), seed=rows + k)
    A, sA = _run(x, wl.E4M3)
    _check_against_oracle(x, wl.E4M3, A, sA)


def test_quantize_then_gemm_matches_oracle():
    """The quantizer's outputs feed the dense GEMM directly (A and MN-major sA)."""
    m, n, k = 300, 512, 640
    x = wl.activations((m, k), seed=12)
    pb = wl.dense(8, n, k, seed=13)  # only its B and sB are used
    X = _x_device(x)
    A, sA = fg.fg_quantize_fp8_per_token(X, fmt=wl.E4M3)
    D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    fg.fg_gemm_fp8_nt(A, sA, dev(pb.B, fp8_dtype(pb.b_fmt)), dev(pb.sB), D)
    torch.cuda.synchronize()
    q, s = oracle.quantize_per_token(x, wl.E4M3)
    ref, _ = oracle.gemm_fp8_nt(q, wl.E4M3, s, pb.B, pb.b_fmt, pb.sB)
    compare(d_to_bits(D), ref, what="quantize + dense GEMM")


def test_graph_replays_quantize_and_masked_gemm_with_new_counts():
    """Quantize + masked GEMM captured once in a CUDA graph: the counts live on
    the device, so replays with new counts need no host knowledge of them."""
    G, M_cap, n, k = 3, 256, 256, 512
    x = wl.activations((G, M_cap, k), seed=14)
    pb = wl.masked(G, M_cap, n=n, k=k, seed=15)  # its B and sB
    X = _x_device(x)
    A = torch.empty((G, M_cap, k), dtype=torch.float8_e4m3fn, device="cuda")
    sA = torch.empty((G, (k + 127) // 128, fg.fg_scales_a_ld(M_cap)), dtype=torch.float32, device="cuda")
    B, sB = dev(pb.B, fp8_dtype(pb.b_fmt)), dev(pb.sB)
    counts = torch.zeros(G, dtype=torch.int32, device="cuda")
    D = torch.empty((G, M_cap, n), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        # warm-up outside the graph (loads both kernels before the capture)
        fg.fg_quantize_fp8_per_token(X, A, sA, fmt=wl.E4M3, masked_m=counts, stream=s)
        fg.fg_grouped_gemm_fp8_masked(A, sA, B, sB, D, counts, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fg.fg_quantize_fp8_per_token(X, A, sA, fmt=wl.E4M3, masked_m=counts, stream=s)
            fg.fg_grouped_gemm_fp8_masked(A, sA, B, sB, D, counts, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    q, sc = oracle.quantize_per_token(x, wl.E4M3)
    for cnt in ([5, 256, 130], [0, 1, 255]):
        D.view(torch.int16).fill_(int(np.array(SENTINEL, np.uint16).view(np.int16)))
        counts.copy_(torch.tensor(cnt, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        got = d_to_bits(D)
        init = np.full((G, M_cap, n), SENTINEL, np.uint16)
        ref, _ = oracle.grouped_masked(q, wl.E4M3, sc, pb.B, pb.b_fmt, pb.sB, np.array(cnt, np.int32), init)
        for gi in range(G):
            c = cnt[gi]
            assert np.all(got[gi, c:] == SENTINEL)
            if c:
                compare(got[gi, :c], ref[gi, :c], what=f"graph replay group {gi}")
    assert fg.fg_get_device_status()[0] == fg.FG_OK


@pytest.mark.parametrize("fmt", [wl.E4M3, wl.E5M2])
def test_quantize_exact_ties(fmt):
    """Rows whose quotients x / s land exactly on FP8 midpoints (ties to even),
    with scales s = odd * 2^j whose reciprocals are inexact in FP32: a quotient
    that is not the correctly rounded one breaks such a tie.  Each row holds
    amax = fmax * s (so s is exact) and x = M * s for midpoints M, all exact in
    BF16; the fast division path (s >= 2^-40) and the IEEE fallback are both
    exercised."""
    t = oracle.decode_table(fmt)
    fmax = 448.0 if fmt == wl.E4M3 else 57344.0
    vals = sorted({float(v) for v in t[:128] if np.isfinite(v) and v >= 0})
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    rows = []
    for odd in (3, 5, 7, 11, 13, 25, 49):
        for j in (-60, -20, -3, 0, 7, 20):
            s = odd * 2.0 ** j
            amax = fmax * s
            xs = [m * s for m in mids]
            cand = np.array([amax] + xs + [-x for x in xs], np.float64).astype(np.float32)
            exact = torch.from_numpy(cand).to(torch.bfloat16).to(torch.float32).numpy() == cand
            if not exact[0]:
                continue
            row = cand[exact][:128]
            rows.append(np.pad(row, (0, 128 - row.size)))
    x = np.stack(rows).astype(np.float32)
    A, sA = _run(x, fmt)
    _check_against_oracle(x, fmt, A, sA)


# ------------------------------------------------------------ FP32 activations
# fg_quantize_fp8_per_token_f32in: the same contract on float32 X, whose values
# carry full 24-bit significands and reach the float32 extremes.

def _f32_activations(shape, seed):
    """Seeded float32 activations that are not bfloat16 values (random low
    significand bits), with the magnitude mix of the BF16 workload."""
    x = wl.activations(shape, seed=seed).astype(np.float32)
    jitter = wl.rng_for(seed + 1).uniform(-1, 1, size=x.shape).astype(np.float32)
    return (x * (np.float32(1) + jitter * np.float32(2.0 ** -9))).astype(np.float32)


@pytest.mark.parametrize("fmt", [wl.E4M3, wl.E5M2])
@pytest.mark.parametrize("batches,rows,k,ld_x", [
    (1, 1, 16, 16),
    (1, 31, 112, 116),      # one partial K block, a row pitch of 116 floats
    (1, 33, 144, 160),
    (1, 257, 304, 304),
    (3, 70, 256, 260),      # batches
    (2, 1, 128, 132),       # one row per batch
])
def test_quantize_f32_input_bit_exact(fmt, batches, rows, k, ld_x):
    x = _f32_activations((batches, rows, k), seed=rows * 11 + k + fmt)
    assert not np.array_equal(x, torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy())
    A, sA = _run(x, fmt, ld_x=ld_x, dtype=torch.float32)
    _check_against_oracle(x, fmt, A, sA)


@pytest.mark.parametrize("fmt", [wl.E4M3, wl.E5M2])
def test_quantize_f32_input_extremes(fmt):
    """Zero groups, signed zeros, the largest float32 values (scale amax / fmax
    stays finite), float32 subnormals down to 2^-149 (scales in the subnormal
    range: the IEEE-division fallback), magnitudes log-uniform over the whole
    float32 range, and quotients on exact FP8 midpoints of full-precision
    scales."""
    rng = wl.rng_for(4040 + fmt)
    rows, k = 64, 512
    ceil = rng.uniform(-149, 127, size=(rows, k // 128, 1))
    e = ceil - rng.uniform(0, 40, size=(rows, k // 128, 128))
    x = (np.exp2(np.maximum(e, -149)) * rng.choice([-1.0, 1.0], size=e.shape)).reshape(rows, k).astype(np.float32)
    fmax32 = np.float32(np.finfo(np.float32).max)
    x[0] = 0.0
    x[1] = -0.0
    x[2, :] = fmax32
    x[2, 1::2] = -fmax32
    x[3, :] = np.float32(2.0 ** -149)
    x[3, 7] = np.float32(5 * 2.0 ** -149)
    # quotients on FP8 midpoints: x = mid * s with scales of 19 significant
    # bits whose reciprocals are inexact (mid has at most 5, fmax 3 bits, so
    # mid * s and amax = fmax * s are exact float32 values and amax / fmax = s)
    t = oracle.decode_table(fmt)
    fm = 448.0 if fmt == wl.E4M3 else 57344.0
    vals = sorted({float(v) for v in t[:128] if np.isfinite(v) and v >= 0})
    mids = np.array([(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])], np.float64)
    for i, sc in enumerate([1.0 + 2.0 ** -18, 3.0 * (1 - 2.0 ** -17), (2.0 ** 19 - 1) * 2.0 ** -25]):
        row = np.resize(mids, 128) * sc
        row[0] = fm * sc  # the group maximum
        assert np.all(row.astype(np.float32).astype(np.float64) == row)
        x[4 + i, :128] = row.astype(np.float32)
    A, sA = _run(x, fmt, dtype=torch.float32)
    _check_against_oracle(x, fmt, A, sA)


def test_quantize_f32_input_masked_counts():
    x = _f32_activations((4, 96, 512), seed=81)
    counts = [0, 96, 33, 1]
    A, sA = _run(x, wl.E5M2, masked_m=counts, dtype=torch.float32)
    _check_against_oracle(x, wl.E5M2, A, sA, limits=counts)
    assert fg.fg_get_device_status()[0] == fg.FG_OK


@pytest.mark.parametrize("rows,k", [(4096, 7168), (64, 2048)])
def test_quantize_f32_input_full_size_bit_exact(rows, k):
    x = _f32_activations((rows, k), seed=rows + k + 3)
    A, sA = _run(x, wl.E4M3, dtype=torch.float32)
    _check_against_oracle(x, wl.E4M3, A, sA)


def test_graph_replays_f32_quantize_and_masked_gemm_with_new_counts():
    """FP32-input quantize + masked GEMM captured once in a CUDA graph and
    replayed with new device-side counts."""
    G, M_cap, n, k = 2, 256, 264, 384
    x = _f32_activations((G, M_cap, k), seed=84)
    pb = wl.masked(G, M_cap, n=n, k=k, seed=85)  # its B and sB
    X = _x_device(x, dtype=torch.float32)
    A = torch.empty((G, M_cap, k), dtype=torch.float8_e4m3fn, device="cuda")
    sA = torch.empty((G, (k + 127) // 128, fg.fg_scales_a_ld(M_cap)), dtype=torch.float32, device="cuda")
    B, sB = dev(pb.B, fp8_dtype(pb.b_fmt)), dev(pb.sB)
    counts = torch.zeros(G, dtype=torch.int32, device="cuda")
    D = torch.empty((G, M_cap, n), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fg.fg_quantize_fp8_per_token(X, A, sA, fmt=wl.E4M3, masked_m=counts, stream=s)
        fg.fg_grouped_gemm_fp8_masked(A, sA, B, sB, D, counts, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fg.fg_quantize_fp8_per_token(X, A, sA, fmt=wl.E4M3, masked_m=counts, stream=s)
            fg.fg_grouped_gemm_fp8_masked(A, sA, B, sB, D, counts, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    q, sc = oracle.quantize_per_token(x, wl.E4M3)
    for cnt in ([256, 7], [0, 129]):
        D.view(torch.int16).fill_(int(np.array(SENTINEL, np.uint16).view(np.int16)))
        counts.copy_(torch.tensor(cnt, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        got = d_to_bits(D)
        init = np.full((G, M_cap, n), SENTINEL, np.uint16)
        ref, _ = oracle.grouped_masked(q, wl.E4M3, sc, pb.B, pb.b_fmt, pb.sB, np.array(cnt, np.int32), init)
        for gi in range(G):
            c = cnt[gi]
            assert np.all(got[gi, c:] == SENTINEL)
            if c:
                compare(got[gi, :c], ref[gi, :c], what=f"FP32 quantize graph replay group {gi}")
    assert fg.fg_get_device_status()[0] == fg.FG_OK


def test_quantize_f32_input_then_gemm_matches_oracle():
    m, n, k = 300, 512, 640
    x = _f32_activations((m, k), seed=82)
    pb = wl.dense(8, n, k, seed=83)  # only its B and sB are used
    A, sA = fg.fg_quantize_fp8_per_token(_x_device(x, dtype=torch.float32), fmt=wl.E4M3)
    D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    fg.fg_gemm_fp8_nt(A, sA, dev(pb.B, fp8_dtype(pb.b_fmt)), dev(pb.sB), D)
    torch.cuda.synchronize()
    q, s = oracle.quantize_per_token(x, wl.E4M3)
    ref, _ = oracle.gemm_fp8_nt(q, wl.E4M3, s, pb.B, pb.b_fmt, pb.sB)
    compare(d_to_bits(D), ref, what="quantize (FP32 input) + dense GEMM")

