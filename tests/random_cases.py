"""Seeded random calls of the four GEMM layouts, shared by the randomized
parity sweeps of the release library and of the FG_DEBUG build: each draw
picks the shape (ragged in every dimension), the FP8 formats of A and B, the
output type and a tile plan forced through the process-wide
knobs, runs the call through the C ABI and compares every output element with
the CPU oracle; D starts filled with a sentinel inside a buffer with sentinel
guard bands before and after it, the rows a grouped call must leave untouched
are checked bit for bit, and so are the guard bands."""
import numpy as np
import torch

import moe_grouped_gemm_nt_gb300 as fg
import oracle
import workloads as wl
from gpu_common import SENTINEL, check_status, compare, d_to_bits, dev, fp8_dtype

LAYOUTS = ("dense", "contiguous", "masked", "k_grouped")
SENT32 = 0x7FCADBAD  # float32 NaN pattern the kernels never write


def reset_knobs():
    fg.fg_set_num_sms(0)
    fg.fg_set_config_override(0, 0)
    fg.fg_set_pair_mode(-1)
    fg.fg_set_swap_mode(-1)
    fg.lib().fg_debug_set_pair_defer(-1)


def _draw_plan(rng, layout, rows, k):
    """(block_n, split_k, pair_mode, defer_mode, swap_mode); 0 / -1 = automatic."""
    max_split = max(1, min(8, -(-k // 128)))
    opts = [(0, 0, -1, -1, -1), (128, 1, 0, -1, 0), (256, 1, 0, -1, 0)]
    if layout in ("dense", "contiguous", "masked") and max_split > 1:
        s = int(rng.integers(2, max_split + 1))
        opts += [(128, s, 0, -1, 0), (256, s, 0, -1, 0)]
    opts += [(256, 1, 1, 0, 0), (256, 1, 1, 1, 0)]
    if layout in ("dense", "masked") and rows <= 256:
        opts += [(0, 0, -1, -1, 1), (0, int(rng.integers(1, max_split + 1)), -1, -1, 1)]
    return opts[int(rng.integers(len(opts)))]


def _apply(plan, sms):
    bn, split, pair, defer, swap = plan
    fg.fg_set_num_sms(sms)
    fg.fg_set_config_override(bn, split)
    fg.fg_set_pair_mode(pair)
    fg.lib().fg_debug_set_pair_defer(defer)
    fg.fg_set_swap_mode(swap)


GUARD = 4096  # canary elements on each side of D


def _empty(shape, f32):
    """D filled with the sentinel, inside a buffer whose GUARD elements before
    and after it hold the sentinel too (checked by _guards_intact)."""
    n = int(np.prod(shape))
    if f32:
        buf = torch.full((GUARD + n + GUARD,), SENT32, dtype=torch.int32, device="cuda")
        return buf[GUARD:GUARD + n].view(torch.float32).view(shape), buf
    buf = torch.full((GUARD + n + GUARD,), -1, dtype=torch.int16, device="cuda")
    return buf[GUARD:GUARD + n].view(torch.bfloat16).view(shape), buf


def _guards_intact(buf, f32):
    host = buf.cpu().numpy()
    want = SENT32 if f32 else -1
    return bool(np.all(host[:GUARD] == want) and np.all(host[-GUARD:] == want))


def _check(D, f32, ref16, ref64, written, what):
    """Written elements within the parity bar (FP32 output: against the FP64
    result), the others still the sentinel."""
    if f32:
        got = D.cpu().numpy()
        raw = got.view(np.uint32)
        assert np.all(raw[~written] == SENT32), f"{what}: untouched elements were written"
        g = got[written].astype(np.float64)
        r = ref64[written]
        assert np.all(np.isfinite(g)), f"{what}: non-finite output"
        m = float(np.max(np.abs(r))) if r.size else 0.0
        assert np.all(np.abs(g - r) <= 1e-2 * m), f"{what}: FP32 output out of tolerance"
        nr = float(np.linalg.norm(r))
        if nr > 0:
            assert float(np.linalg.norm(g - r)) / nr <= 1e-3, f"{what}: FP32 aggregate error"
    else:
        got = d_to_bits(D)
        assert np.all(got[~written] == SENTINEL), f"{what}: untouched elements were written"
        if written.any():
            compare(got[written], ref16[written], what=what)


def random_case(case, rng_base, seed_base):
    """One seeded random call (layout chosen by case % 4), checked against the
    oracle.  Returns False when the draw holds no rows (nothing to check)."""
    rng = np.random.default_rng(rng_base + case)
    layout = LAYOUTS[case % len(LAYOUTS)]
    b_fmt = wl.E5M2 if rng.random() < 0.3 else wl.E4M3
    a_fmt = wl.E5M2 if rng.random() < 0.2 else wl.E4M3
    f32 = bool(rng.random() < 0.3)
    n = 8 * int(rng.integers(1, 161))
    seed = wl.seed_for(9, seed_base + case)
    # persistent CTAs: all SMs, or few, so that each CTA (or CTA pair) walks many
    # tiles of the ragged problem and carries its rings and scans across them
    sms = int(rng.choice([0, 0, 2, 3, 8]))
    sfx = "_f32out" if f32 else ""

    if layout == "dense":
        m, k = int(rng.integers(1, 1101)), 16 * int(rng.integers(1, 151))
        p = wl.dense(m, n, k, seed=seed, b_fmt=b_fmt, a_fmt=a_fmt)
        plan = _draw_plan(rng, layout, m, k)
        _apply(plan, sms)
        D, buf = _empty((m, n), f32)
        getattr(fg, "fg_gemm_fp8_nt" + sfx)(dev(p.A, fp8_dtype(a_fmt)), fg.fg_scales_a_to_mn_major(dev(p.sA)),
                                            dev(p.B, fp8_dtype(b_fmt)), dev(p.sB), D)
        ref16, ref64 = oracle.gemm_fp8_nt(p.A, a_fmt, p.sA, p.B, b_fmt, p.sB, want_f64=f32)
        written = np.ones((m, n), bool)
    elif layout == "contiguous":
        G = int(rng.integers(1, 6))
        rows = [int(rng.integers(0, 301)) for _ in range(G)]
        k = 16 * int(rng.integers(1, 76))
        p = wl.contiguous(rows, n=n, k=k, seed=seed, b_fmt=b_fmt, a_fmt=a_fmt)
        if p.M == 0:
            return False
        plan = _draw_plan(rng, layout, p.M, k)
        _apply(plan, sms)
        D, buf = _empty((p.M, n), f32)
        getattr(fg, "fg_grouped_gemm_fp8_contiguous" + sfx)(
            dev(p.A, fp8_dtype(p.a_fmt)), fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.B, fp8_dtype(b_fmt)),
            dev(p.sB), D, dev(p.m_indices))
        init = np.full((p.M, n), SENTINEL, np.uint16)
        ref16, ref64 = oracle.grouped_contiguous(p.A, p.a_fmt, p.sA, p.B, b_fmt, p.sB, p.m_indices, init,
                                                 want_f64=f32)
        written = np.repeat((p.m_indices >= 0)[:, None], n, axis=1)
    elif layout == "masked":
        G, M_cap = int(rng.integers(1, 6)), int(rng.integers(1, 401))
        k = 16 * int(rng.integers(1, 76))
        counts = [int(rng.choice([0, M_cap, int(rng.integers(0, M_cap + 1))])) for _ in range(G)]
        p = wl.masked(G, M_cap, n=n, k=k, seed=seed, masked_m=counts, b_fmt=b_fmt, a_fmt=a_fmt)
        plan = _draw_plan(rng, layout, M_cap, k)
        _apply(plan, sms)
        D, buf = _empty((G, M_cap, n), f32)
        getattr(fg, "fg_grouped_gemm_fp8_masked" + sfx)(
            dev(p.A, fp8_dtype(p.a_fmt)), fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.B, fp8_dtype(b_fmt)),
            dev(p.sB), D, dev(p.masked_m))
        init = np.full((G, M_cap, n), SENTINEL, np.uint16)
        ref16, ref64 = oracle.grouped_masked(p.A, p.a_fmt, p.sA, p.B, b_fmt, p.sB, p.masked_m, init, want_f64=f32)
        written = np.repeat((np.arange(M_cap)[None, :] < p.masked_m[:, None])[:, :, None], n, axis=2)
    else:
        G, M = int(rng.integers(1, 7)), int(rng.integers(1, 601))
        ks = [128 * int(rng.integers(0, 7)) for _ in range(G)]
        K = sum(ks) + 16 * int(rng.integers(0 if sum(ks) else 1, 11))
        p = wl.k_grouped(M, n, ks, seed=seed, b_fmt=b_fmt, K=K, a_fmt=a_fmt)
        plan = _draw_plan(rng, layout, M, K)
        _apply(plan, sms)
        D, buf = _empty((G, M, n), f32)
        getattr(fg, "fg_k_grouped_gemm_fp8_nt" + sfx)(
            dev(p.A, fp8_dtype(p.a_fmt)), fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.B, fp8_dtype(b_fmt)),
            dev(p.sB), D, dev(np.array(ks, np.int32)))
        ref16, ref64 = oracle.k_grouped(p.A, p.a_fmt, p.sA, p.B, b_fmt, p.sB, np.array(ks, np.int32), want_f64=f32)
        written = np.ones((G, M, n), bool)
    torch.cuda.synchronize()
    check_status()
    assert _guards_intact(buf, f32), f"case {case}: bytes outside D were written"
    what = (f"case {case}: {layout} {tuple(D.shape)} k={p.k} A/B fmt {a_fmt}/{b_fmt} {'f32' if f32 else 'bf16'} plan {plan} "
            f"sms {sms}")
    _check(D, f32, ref16, ref64, written, what)
    return True
