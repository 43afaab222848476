"""Seeded synthetic inputs for the FP8 NT GEMM and its two grouped layouts.

This module is shared by the tests, ``bench.py`` and the smoke entry.  It holds
no arithmetic of the GEMM itself: it draws seeded N(0,1) values, quantizes them
to FP8 the way the input recipe asks (one FP32 scale ``amax / fp8_max`` per
1x128 row group of the LHS and per 128x128 block of the RHS, as in the page
"DeepSeek开源周第三天DeepGEMM", section "基本用法", with maxima 448 for E4M3 and
57344 for E5M2 from "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践", section 3.1), builds the
grouped index tensors, and rearranges scale tensors between layouts.

FP8 encoding uses torch's float8 conversions (round to nearest even) after
clipping to the finite range, i.e. saturating.  All randomness comes from
numpy's PCG64 with an explicit seed.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

E4M3 = 0
E5M2 = 1
FP8_MAX = {E4M3: 448.0, E5M2: 57344.0}
KBLOCK = 128
NBLOCK = 128
MBLOCK_ALIGN = 128  # row alignment of contiguous-layout segments


def cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


def round_up(a: int, b: int) -> int:
    return cdiv(a, b) * b


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def encode_fp8(x: np.ndarray, fmt: int) -> np.ndarray:
    """float32 -> FP8 bytes, round to nearest even, saturating at +-max."""
    import torch

    lim = np.float32(FP8_MAX[fmt])
    x = np.clip(np.ascontiguousarray(x, dtype=np.float32), -lim, lim)
    dt = torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2
    return torch.from_numpy(x).to(dt).view(torch.uint8).numpy()


def _amax_scale(amax: np.ndarray, fmt: int) -> np.ndarray:
    s = (amax.astype(np.float32) / np.float32(FP8_MAX[fmt])).astype(np.float32)
    # an all-zero group gets scale 1 (its payload is all zeros), never 0
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def quantize_rows(x: np.ndarray, fmt: int = E4M3):
    """Per 1x128 row-group quantization of x [..., rows, k].
    Returns (q uint8 [..., rows, k], s float32 [..., rows, ceil(k/128)])."""
    *lead, rows, k = x.shape
    kb = cdiv(k, KBLOCK)
    xp = x if k == kb * KBLOCK else np.concatenate(
        [x, np.zeros((*lead, rows, kb * KBLOCK - k), np.float32)], axis=-1)
    xb = xp.reshape(*lead, rows, kb, KBLOCK)
    s = _amax_scale(np.abs(xb).max(axis=-1), fmt)
    q = encode_fp8(xb / s[..., None], fmt).reshape(*lead, rows, kb * KBLOCK)[..., :k]
    return np.ascontiguousarray(q), s


def quantize_blocks(x: np.ndarray, fmt: int = E4M3):
    """Per 128x128 block quantization of x [..., n, k].
    Returns (q uint8 [..., n, k], s float32 [..., ceil(n/128), ceil(k/128)])."""
    *lead, n, k = x.shape
    nb, kb = cdiv(n, NBLOCK), cdiv(k, KBLOCK)
    xp = np.zeros((*lead, nb * NBLOCK, kb * KBLOCK), np.float32)
    xp[..., :n, :k] = x
    xb = xp.reshape(*lead, nb, NBLOCK, kb, KBLOCK)
    s = _amax_scale(np.abs(xb).max(axis=(-3, -1)), fmt)
    q = encode_fp8(xb / s[..., :, None, :, None], fmt).reshape(*lead, nb * NBLOCK, kb * KBLOCK)
    return np.ascontiguousarray(q[..., :n, :k]), s


def scales_ld(rows: int) -> int:
    """Leading dimension of an MN-major LHS scale matrix: rows rounded up to 4
    so that each K-block's column of scales starts on a 16-byte boundary."""
    return round_up(max(rows, 1), 4)


def scales_mn_major(s_rows: np.ndarray, ld: Optional[int] = None) -> np.ndarray:
    """[..., rows, KB] row-major -> [..., KB, ld] (MN-major, padded with zeros)."""
    *lead, rows, kb = s_rows.shape
    ld = scales_ld(rows) if ld is None else ld
    out = np.zeros((*lead, kb, ld), np.float32)
    out[..., :, :rows] = np.swapaxes(s_rows, -1, -2)
    return out


def _normal(rng, shape, chunk_rows=4096):
    """Seeded N(0,1) float32, drawn in row chunks to bound peak memory."""
    shape = tuple(shape)
    out = np.empty(shape, np.float32)
    flat = out.reshape(-1, shape[-1])
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(r0 + chunk_rows, flat.shape[0])
        flat[r0:r1] = rng.standard_normal((r1 - r0, shape[-1]), dtype=np.float32)
    return out


def _quant_rows_chunked(rng, lead_rows, k, fmt, chunk_rows=8192):
    """Draw and quantize a [lead_rows, k] LHS in chunks (memory-bounded)."""
    q = np.empty((lead_rows, k), np.uint8)
    s = np.empty((lead_rows, cdiv(k, KBLOCK)), np.float32)
    for r0 in range(0, lead_rows, chunk_rows):
        r1 = min(r0 + chunk_rows, lead_rows)
        x = rng.standard_normal((r1 - r0, k), dtype=np.float32)
        q[r0:r1], s[r0:r1] = quantize_rows(x, fmt)
    return q, s


def _quant_blocks_chunked(rng, n, k, fmt, chunk_rows=8192):
    """Draw and quantize one [n, k] RHS in 128-row-aligned chunks."""
    q = np.empty((n, k), np.uint8)
    s = np.empty((cdiv(n, NBLOCK), cdiv(k, KBLOCK)), np.float32)
    for r0 in range(0, n, chunk_rows):
        r1 = min(r0 + chunk_rows, n)
        x = rng.standard_normal((r1 - r0, k), dtype=np.float32)
        q[r0:r1], s[r0 // NBLOCK: cdiv(r1, NBLOCK)] = quantize_blocks(x, fmt)
    return q, s


def _loguniform_scales(rng, shape, lo_exp=-8.0, hi_exp=8.0):
    e = rng.uniform(lo_exp, hi_exp, size=shape)
    return np.exp2(e).astype(np.float32)


# ------------------------------------------------------------------ problems


@dataclass
class Dense:
    m: int
    n: int
    k: int
    A: np.ndarray          # [m, k] uint8
    sA: np.ndarray         # [m, KB] float32 (row-major, the logical layout)
    B: np.ndarray          # [n, k] uint8
    sB: np.ndarray         # [NB, KB] float32
    a_fmt: int = E4M3
    b_fmt: int = E4M3
    seed: int = 0

    @property
    def flops(self) -> float:
        return 2.0 * self.m * self.n * self.k

    @property
    def bytes(self) -> int:
        """Algorithmic HBM bytes: A + B + scales + D, each touched once."""
        return (self.m * self.k + self.n * self.k + self.sA.size * 4 + self.sB.size * 4
                + self.m * self.n * 2)


def dense(m, n, k, seed, b_fmt=E4M3, a_fmt=E4M3, scales="amax") -> Dense:
    """Dense NT problem.  scales="amax": scale = amax/max per group/block.
    scales="loguniform": the FP8 payload is quantized the same way, but the
    stored scales are replaced by independent draws 2^U(-8,8)."""
    rng = rng_for(seed)
    A, sA = _quant_rows_chunked(rng, m, k, a_fmt)
    B, sB = _quant_blocks_chunked(rng, n, k, b_fmt)
    if scales == "loguniform":
        sA = _loguniform_scales(rng, sA.shape)
        sB = _loguniform_scales(rng, sB.shape)
    elif scales != "amax":
        raise ValueError(scales)
    return Dense(m, n, k, A, sA, B, sB, a_fmt, b_fmt, seed)


@dataclass
class Contiguous:
    M: int
    n: int
    k: int
    G: int
    A: np.ndarray          # [M, k]
    sA: np.ndarray         # [M, KB]
    B: np.ndarray          # [G, n, k]
    sB: np.ndarray         # [G, NB, KB]
    m_indices: np.ndarray  # [M] int32, -1 on padding rows
    group_rows: List[int] = field(default_factory=list)
    a_fmt: int = E4M3
    b_fmt: int = E4M3
    seed: int = 0

    @property
    def valid_rows(self) -> int:
        return int((self.m_indices >= 0).sum())

    @property
    def flops(self) -> float:
        return 2.0 * self.valid_rows * self.n * self.k

    @property
    def bytes(self) -> int:
        used = len({int(g) for g in np.unique(self.m_indices) if g >= 0})
        nb, kb = cdiv(self.n, NBLOCK), cdiv(self.k, KBLOCK)
        return (self.M * self.k + used * self.n * self.k + self.M * kb * 4
                + used * nb * kb * 4 + self.valid_rows * self.n * 2 + self.M * 4)


def contiguous(group_rows, n, k, seed, b_fmt=E4M3, align=MBLOCK_ALIGN, a_fmt=E4M3) -> Contiguous:
    """Contiguous layout: group g contributes group_rows[g] rows, each segment
    padded with -1 rows to a multiple of `align`, segments concatenated on M."""
    rng = rng_for(seed)
    G = len(group_rows)
    seg = [round_up(r, align) for r in group_rows]
    M = int(sum(seg))
    m_indices = np.full(M, -1, np.int32)
    r0 = 0
    for g, (r, s) in enumerate(zip(group_rows, seg)):
        m_indices[r0:r0 + r] = g
        r0 += s
    A, sA = _quant_rows_chunked(rng, M, k, a_fmt) if M > 0 else (
        np.zeros((0, k), np.uint8), np.zeros((0, cdiv(k, KBLOCK)), np.float32))
    B = np.empty((G, n, k), np.uint8)
    sB = np.empty((G, cdiv(n, NBLOCK), cdiv(k, KBLOCK)), np.float32)
    for g in range(G):
        B[g], sB[g] = _quant_blocks_chunked(rng, n, k, b_fmt)
    return Contiguous(M, n, k, G, A, sA, B, sB, m_indices, list(group_rows), a_fmt, b_fmt, seed)


@dataclass
class Masked:
    G: int
    M_cap: int
    n: int
    k: int
    A: np.ndarray          # [G, M_cap, k]
    sA: np.ndarray         # [G, M_cap, KB]
    B: np.ndarray          # [G, n, k]
    sB: np.ndarray         # [G, NB, KB]
    masked_m: np.ndarray   # [G] int32
    a_fmt: int = E4M3
    b_fmt: int = E4M3
    seed: int = 0

    @property
    def valid_rows(self) -> int:
        return int(np.clip(self.masked_m, 0, self.M_cap).sum())

    @property
    def flops(self) -> float:
        return 2.0 * self.valid_rows * self.n * self.k

    @property
    def bytes(self) -> int:
        """Valid rows of A/sA/D, B and sB of every group with rows, counts."""
        nb, kb = cdiv(self.n, NBLOCK), cdiv(self.k, KBLOCK)
        used = int((self.masked_m > 0).sum())
        v = self.valid_rows
        return (v * self.k + used * self.n * self.k + v * kb * 4 + used * nb * kb * 4
                + v * self.n * 2 + self.G * 4)


def masked(G, M_cap, n, k, seed, masked_m=None, b_fmt=E4M3, a_fmt=E4M3) -> Masked:
    """Masked layout: fixed capacity M_cap per group; valid-row counts drawn
    uniformly from [0, M_cap] (inclusive) unless given."""
    rng = rng_for(seed)
    if masked_m is None:
        masked_m = rng.integers(0, M_cap, size=G, endpoint=True)
    masked_m = np.asarray(masked_m, np.int32)
    A, sA = _quant_rows_chunked(rng, G * M_cap, k, a_fmt)
    B = np.empty((G, n, k), np.uint8)
    sB = np.empty((G, cdiv(n, NBLOCK), cdiv(k, KBLOCK)), np.float32)
    for g in range(G):
        B[g], sB[g] = _quant_blocks_chunked(rng, n, k, b_fmt)
    return Masked(G, M_cap, n, k, A.reshape(G, M_cap, k), sA.reshape(G, M_cap, -1),
                  B, sB, masked_m, a_fmt, b_fmt, seed)


# ------------------------------------------------- the five named workloads

# (n, k) weight shapes of the dense sweep and of the grouped layouts
DENSE_SWEEP_NK = [(2112, 7168), (24576, 1536), (7168, 16384), (4096, 7168), (7168, 2048)]
DENSE_SWEEP_M = [64, 128, 4096]
GROUPED_NK = [(4096, 7168), (7168, 2048)]
CONTIGUOUS_G = [4, 8]
CONTIGUOUS_ROWS_PER_GROUP = 8192
MASKED_G = [1, 2, 4, 16]
MASKED_M_CAP = 256


def seed_for(config_id: int, variant: int = 0) -> int:
    """Seed recipe: 1000 + workload number + 100 * variant."""
    return 1000 + config_id + 100 * variant


def small_dense(seed=None) -> Dense:
    """Dense 128 x 256 x 512 (workload 0)."""
    return dense(128, 256, 512, seed_for(0) if seed is None else seed)


def dense_sweep_shapes():
    """(m, n, k) of the dense sweep (workload 1), in a fixed order."""
    return [(m, n, k) for (n, k) in DENSE_SWEEP_NK for m in DENSE_SWEEP_M]


def contiguous_shapes():
    return [(G, n, k) for G in CONTIGUOUS_G for (n, k) in GROUPED_NK]


def masked_shapes():
    return [(G, n, k) for G in MASKED_G for (n, k) in GROUPED_NK]


def large_dense_shapes():
    """(m, n, k, b_fmt) of workload 4: 8192^3, the K-tail case, the E5M2-B case."""
    return [(8192, 8192, 8192, E4M3), (8192, 8192, 8192 + 128 * 3, E4M3),
            (8192, 8192, 8192, E5M2)]


def activations(shape, seed: int, outlier_frac: float = 0.01, outlier_gain: float = 32.0,
                chunk_rows: int = 4096) -> np.ndarray:
    """Seeded BF16 activations [..., rows, k], returned as float32 numpy values
    that are exactly bfloat16 (rounded to nearest even by torch).

    Recipe: N(0,1) entries; each row scaled by 2^u with u uniform in [-6, 6]
    (tokens of different magnitude); a fixed random ~1% of the columns (outlier
    channels) multiplied by `outlier_gain`.  Drawn in row chunks to bound peak
    memory."""
    import torch

    shape = tuple(shape)
    rng = rng_for(seed)
    k = shape[-1]
    out = _normal(rng, shape, chunk_rows)
    flat = out.reshape(-1, k)
    rows_total = flat.shape[0]
    gain = np.exp2(rng.uniform(-6.0, 6.0, size=(rows_total, 1))).astype(np.float32)
    cols = np.ones(k, np.float32)
    cols[rng.random(k) < outlier_frac] = np.float32(outlier_gain)
    for r0 in range(0, rows_total, chunk_rows):
        r1 = min(r0 + chunk_rows, rows_total)
        blk = flat[r0:r1] * gain[r0:r1] * cols
        flat[r0:r1] = torch.from_numpy(blk).to(torch.bfloat16).to(torch.float32).numpy()
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Bit patterns (uint16) of float32 values that are exactly bfloat16."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert not np.any(u & 0xFFFF), "values are not bfloat16"
    return (u >> 16).astype(np.uint16)


# K-grouped layout (the weight gradient of the contiguous workload): for each
# (n, k) weight shape, G experts of 8192 tokens; the gradient of B[g] [n][k]
# contracts the output gradient [tokens][n] with the activations [tokens][k]
# over the group's tokens, i.e. M = n, N = k, one 8192-long K segment per group.
KGROUPED_G = [4, 8]
KGROUPED_TOKENS_PER_GROUP = CONTIGUOUS_ROWS_PER_GROUP


def k_grouped_shapes():
    """(G, M, N, tokens per group) of the K-grouped workload."""
    return [(G, n, k, KGROUPED_TOKENS_PER_GROUP) for G in KGROUPED_G for (n, k) in GROUPED_NK]


# short segments: many experts with few tokens each (the CTA-pair plan with the store warp)
KGROUPED_SHORT_G = 32
KGROUPED_SHORT_TOKENS = 512


def k_grouped_short_shapes():
    """(G, M, N, tokens per group) of the short-segment K-grouped figures."""
    return [(KGROUPED_SHORT_G, n, k, KGROUPED_SHORT_TOKENS) for (n, k) in GROUPED_NK]


def k_grouped(M, N, k_sizes, seed, b_fmt=E4M3, K=None, a_fmt=E4M3) -> Dense:
    """Operands of a K-grouped problem: A [M][K], B [N][K] with the NT GEMM's
    scaling (1 x 128 LHS groups, 128 x 128 RHS blocks), K = sum of the segment
    lengths unless given.  Returns a Dense holding them (m = M, n = N, k = K)."""
    total = int(np.sum(k_sizes))
    return dense(M, N, total if K is None else K, seed, b_fmt=b_fmt, a_fmt=a_fmt)
