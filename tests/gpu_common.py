"""Helpers shared by the GPU tests: move generated problems to the device, run
the library through its C ABI binding and compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import moe_grouped_gemm_nt_gb300 as fg
import oracle
import workloads as wl

SENTINEL = 0xFFFF  # a BF16 NaN pattern the kernels never write (they write 0x7FC0-style NaNs at most)

# tolerance of the parity bar: per element |d| <= 1e-2 * max|ref| + 1 ulp_bf16(ref),
# aggregate ||gpu - ref||_F / ||ref||_F <= 1e-3 (ref = oracle result rounded to BF16)
ELEM_REL = 1e-2
AGG_REL = 1e-3


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def bf16_ulp(x32: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 at each (bfloat16-valued) float32 number."""
    a = np.abs(x32.astype(np.float32))
    sp = np.spacing(a) * np.float32(65536.0)
    return np.maximum(sp, np.float32(2.0 ** -133))


def compare(gpu_bits: np.ndarray, ref_bits: np.ndarray, scale_ref: float | None = None, what: str = ""):
    """Assert the parity bar; returns (max_abs_err, aggregate_rel_err)."""
    g = bits_to_f32(gpu_bits).astype(np.float64)
    r = bits_to_f32(ref_bits).astype(np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    m = float(np.max(np.abs(r))) if scale_ref is None else float(scale_ref)
    d = np.abs(g - r)
    tol = ELEM_REL * m + bf16_ulp(r.astype(np.float32)).astype(np.float64)
    bad = d > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; first at "
                             f"{tuple(i)}: gpu={g[tuple(i)]} ref={r[tuple(i)]} tol={tol[tuple(i)]}")
    nr = float(np.linalg.norm(r))
    agg = float(np.linalg.norm(g - r)) / nr if nr > 0 else float(np.linalg.norm(g))
    assert agg <= AGG_REL, f"{what}: aggregate relative error {agg:.3e} > {AGG_REL}"
    return float(d.max()), agg


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def d_to_bits(D: torch.Tensor) -> np.ndarray:
    return D.view(torch.int16).cpu().numpy().view(np.uint16)


def fp8_dtype(fmt):
    return torch.float8_e4m3fn if fmt == wl.E4M3 else torch.float8_e5m2


def check_status():
    st, detail = fg.fg_get_device_status()
    assert st == fg.FG_OK, f"device status {fg.STATUS_NAMES.get(st, st)} detail={detail:#x}"


def run_dense(p: wl.Dense, D=None):
    A = dev(p.A, fp8_dtype(p.a_fmt))
    B = dev(p.B, fp8_dtype(p.b_fmt))
    sA = fg.fg_scales_a_to_mn_major(dev(p.sA))
    sB = dev(p.sB)
    if D is None:
        D = torch.empty((p.m, p.n), dtype=torch.bfloat16, device="cuda")
    fg.fg_gemm_fp8_nt(A, sA, B, sB, D)
    torch.cuda.synchronize()
    check_status()
    return D


def run_contiguous(p: wl.Contiguous, D=None):
    A = dev(p.A, fp8_dtype(p.a_fmt))
    B = dev(p.B, fp8_dtype(p.b_fmt))
    sA = fg.fg_scales_a_to_mn_major(dev(p.sA))
    sB = dev(p.sB)
    mi = dev(p.m_indices)
    if D is None:
        D = torch.full((p.M, p.n), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fg.fg_grouped_gemm_fp8_contiguous(A, sA, B, sB, D, mi)
    torch.cuda.synchronize()
    check_status()
    return D


def run_masked(p: wl.Masked, D=None):
    A = dev(p.A, fp8_dtype(p.a_fmt))
    B = dev(p.B, fp8_dtype(p.b_fmt))
    sA = fg.fg_scales_a_to_mn_major(dev(p.sA))
    sB = dev(p.sB)
    mm = dev(p.masked_m)
    if D is None:
        D = torch.full((p.G, p.M_cap, p.n), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fg.fg_grouped_gemm_fp8_masked(A, sA, B, sB, D, mm)
    torch.cuda.synchronize()
    check_status()
    return D


def sample_positions(rows: int, cols: int, seed: int, block_m=128, block_n=256, n_rows_full=16,
                     per_tile=1, boundary_tiles=False):
    """Sampled output positions for large problems: `per_tile` random elements of
    every 128 x 256 output tile, the four corners of every tile, and every
    column of `n_rows_full` random rows (including the first and the last).
    With `boundary_tiles`, also every element of the four corner tiles and of
    the boundary tiles (the last 128-row block across all columns and the
    last 256-column block across all rows), each position once."""
    rng = np.random.default_rng(seed)
    rr, cc = [], []
    for t0 in range(0, rows, block_m):
        t1 = min(t0 + block_m, rows)
        for c0 in range(0, cols, block_n):
            c1 = min(c0 + block_n, cols)
            rr += list(rng.integers(t0, t1, per_tile)) + [t0, t0, t1 - 1, t1 - 1]
            cc += list(rng.integers(c0, c1, per_tile)) + [c0, c1 - 1, c0, c1 - 1]
    full = np.unique(np.concatenate([[0, rows - 1], rng.integers(0, rows, n_rows_full)]))
    for r in full:
        rr += [int(r)] * cols
        cc += list(range(cols))
    r = np.array(rr, np.int64)
    c = np.array(cc, np.int64)
    if boundary_tiles:
        lm0 = (rows - 1) // block_m * block_m   # first row of the last 128-row block
        ln0 = (cols - 1) // block_n * block_n   # first column of the last 256-column block
        blocks = [
            (0, min(block_m, rows), 0, min(block_n, cols)),   # top-left corner tile
            (0, min(block_m, rows), ln0, cols),               # top-right corner tile
            (lm0, rows, 0, cols),                              # last row block: bottom corners and edge
            (0, rows, ln0, cols),                              # last column block: right corners and edge
        ]
        for (a0, a1, b0, b1) in blocks:
            gr, gc = np.meshgrid(np.arange(a0, a1, dtype=np.int64), np.arange(b0, b1, dtype=np.int64),
                                 indexing="ij")
            r = np.concatenate([r, gr.ravel()])
            c = np.concatenate([c, gc.ravel()])
        lin = np.unique(r * cols + c)
        r, c = lin // cols, lin % cols
    return r, c
