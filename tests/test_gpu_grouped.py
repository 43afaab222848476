"""GPU parity of the two MoE grouped layouts against the CPU oracle.

Checks, through the C ABI: element-wise values of written rows within the
tolerance, bit-exactness of which rows are written (D is pre-filled with a
sentinel pattern the kernels never produce), agreement with per-group dense
calls (bitwise: same tile arithmetic), and the full-size workloads on sampled
outputs."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_nt_gb300 as fg
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_common import (SENTINEL, compare, d_to_bits, dev, fp8_dtype, run_contiguous, run_dense,  # noqa: E402
                        run_masked, sample_positions)


# ------------------------------------------------------------- contiguous

@pytest.mark.parametrize("group_rows,n,k", [
    ([100, 0, 300, 5, 128], 264, 400),
    ([128], 256, 128),
    ([1, 1, 1], 8, 16),
    ([513, 77], 2112, 256),
    ([0, 0, 0], 64, 128),
])
def test_contiguous_small_full(group_rows, n, k):
    p = wl.contiguous(group_rows, n=n, k=k, seed=sum(group_rows) + n + k)
    if p.M == 0:
        pytest.skip("no rows")
    got = d_to_bits(run_contiguous(p))
    init = np.full((p.M, p.n), SENTINEL, np.uint16)
    ref, _ = oracle.grouped_contiguous(p.A, 0, p.sA, p.B, 0, p.sB, p.m_indices, init)
    pad = p.m_indices < 0
    assert np.array_equal(got[pad], ref[pad]), "padding rows were written"
    if (~pad).any():
        compare(got[~pad], ref[~pad], what=f"contiguous {group_rows}")


def test_contiguous_all_padding_is_noop():
    p = wl.contiguous([0, 0], n=64, k=128, seed=3)
    assert p.M == 0
    p = wl.contiguous([5], n=64, k=128, seed=3)
    mi = np.full_like(p.m_indices, -1)
    q = wl.Contiguous(p.M, p.n, p.k, p.G, p.A, p.sA, p.B, p.sB, mi)
    got = d_to_bits(run_contiguous(q))
    assert np.all(got == SENTINEL)


@pytest.fixture
def persistent_dense_plan():
    """Dense calls use the grouped kernels' tile plan (128 x 256, no split-K),
    so that per-group dense results have the same FP32 summation order."""
    fg.fg_set_config_override(256, 1)
    yield
    fg.fg_set_config_override(0, 0)


def test_contiguous_equals_per_group_dense_bitwise(persistent_dense_plan):
    p = wl.contiguous([256, 384, 128], n=512, k=768, seed=41)
    got = d_to_bits(run_contiguous(p))
    for g in range(p.G):
        rows = np.nonzero(p.m_indices == g)[0]
        d = wl.Dense(rows.size, p.n, p.k, p.A[rows], p.sA[rows], p.B[g], p.sB[g])
        assert np.array_equal(got[rows], d_to_bits(run_dense(d))), f"group {g}"


def test_contiguous_bad_group_id_reports_device_check():
    p = wl.contiguous([128, 128], n=64, k=128, seed=42)
    mi = p.m_indices.copy()
    mi[128:] = 7  # not a group: the tile is skipped and the call reports it
    A = dev(p.A, fp8_dtype(0))
    D = torch.full((p.M, p.n), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fg.fg_grouped_gemm_fp8_contiguous(A, fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.B, fp8_dtype(0)),
                                      dev(p.sB), D, dev(mi))
    st, detail = fg.fg_get_device_status()
    assert st == 6 and detail == 1 * 1  # tile index 1 (N blocks: 1)
    got = d_to_bits(D)
    assert np.all(got[128:] == SENTINEL)
    init = np.full((p.M, p.n), SENTINEL, np.uint16)
    ref, _ = oracle.grouped_contiguous(p.A, 0, p.sA, p.B, 0, p.sB, mi, init)
    compare(got[:128], ref[:128], what="valid part")


@pytest.mark.parametrize("case", ["foreign_id_in_tile", "id_in_skipped_block"])
def test_contiguous_misaligned_segments_report_device_check(case):
    """Rows that break the 128-row segment contract are never written and the
    call reports FG_ERR_DEVICE_CHECK with the offending row: a row of another
    group inside a tile, or a group id inside a block whose first row is -1."""
    p = wl.contiguous([128, 100], n=64, k=256, seed=43)
    mi = p.m_indices.copy()
    if case == "foreign_id_in_tile":
        bad = 5
        mi[bad] = 1          # tile 0 belongs to group 0
    else:
        mi[128:] = -1
        bad = 130
        mi[bad] = 1          # the block starting at row 128 is skipped
    D = torch.full((p.M, p.n), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fg.fg_grouped_gemm_fp8_contiguous(dev(p.A, fp8_dtype(0)), fg.fg_scales_a_to_mn_major(dev(p.sA)),
                                      dev(p.B, fp8_dtype(0)), dev(p.sB), D, dev(mi))
    st, detail = fg.fg_get_device_status()
    assert st == 6 and detail == bad
    got = d_to_bits(D)
    assert np.all(got[bad] == SENTINEL)
    init = np.full((p.M, p.n), SENTINEL, np.uint16)
    mi_ref = mi.copy()
    mi_ref[bad] = -1  # what the kernel writes: the contract-breaking row stays untouched
    ref, _ = oracle.grouped_contiguous(p.A, 0, p.sA, p.B, 0, p.sB, mi_ref, init)
    written = mi_ref >= 0
    assert np.array_equal(got[~written], ref[~written])
    compare(got[written], ref[written], what=f"contiguous {case}")


@pytest.mark.parametrize("G,n,k", wl.contiguous_shapes())
def test_contiguous_workload(G, n, k):
    """G groups of 8192 rows, (n,k) weight shapes, sampled outputs."""
    p = wl.contiguous([wl.CONTIGUOUS_ROWS_PER_GROUP] * G, n=n, k=k,
                      seed=wl.seed_for(2, wl.contiguous_shapes().index((G, n, k))))
    got = d_to_bits(run_contiguous(p))
    rows, cols = sample_positions(p.M, n, seed=G + n, n_rows_full=8, boundary_tiles=True)
    ref, _ = oracle.grouped_contiguous_at(p.A, 0, p.sA, p.B, 0, p.sB, p.m_indices, rows, cols)
    compare(got[rows, cols], ref, what=f"contiguous G={G} n={n} k={k} (sampled)")


# ----------------------------------------------------------------- masked

@pytest.mark.parametrize("counts,M_cap,n,k", [
    ([0, 1, 127, 128, 129, 256], 256, 264, 400),
    ([37], 96, 128, 256),
    ([0, 0], 128, 64, 128),
    ([300, -4], 256, 256, 256),   # out-of-range counts are clamped (and reported)
    ([200, 64, 3], 200, 2112, 128),
])
def test_masked_small_full(counts, M_cap, n, k):
    p = wl.masked(len(counts), M_cap, n=n, k=k, seed=M_cap + n + k, masked_m=counts)
    got = d_to_bits(run_masked_allow_check(p, expect_check=any(c < 0 or c > M_cap for c in counts)))
    init = np.full((p.G, p.M_cap, p.n), SENTINEL, np.uint16)
    ref, _ = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, init)
    valid = np.arange(M_cap)[None, :] < np.clip(p.masked_m, 0, M_cap)[:, None]
    assert np.array_equal(got[~valid], ref[~valid]), "rows past the count were written"
    if valid.any():
        compare(got[valid], ref[valid], what=f"masked {counts}")


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("counts,M_cap", [([0, 1, 255, 256, 257, 384, 512], 512), ([130, 300], 384)])
def test_masked_pair_tiles(counts, M_cap, pair):
    """Masked layout on CTA pairs (256-row blocks inside a group) and on
    one-CTA tiles: rows past each count untouched, the rest within tolerance."""
    fg.fg_set_pair_mode(pair)
    try:
        p = wl.masked(len(counts), M_cap, n=520, k=384, seed=M_cap + 11 * pair, masked_m=counts)
        got = d_to_bits(run_masked(p))
    finally:
        fg.fg_set_pair_mode(-1)
    init = np.full((p.G, p.M_cap, p.n), SENTINEL, np.uint16)
    ref, _ = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, init)
    valid = np.arange(M_cap)[None, :] < np.clip(p.masked_m, 0, M_cap)[:, None]
    assert np.array_equal(got[~valid], ref[~valid]), "rows past the count were written"
    compare(got[valid], ref[valid], what=f"masked pair={pair} {counts}")


@pytest.mark.parametrize("defer", [0, 1])
@pytest.mark.parametrize("group_rows,n,k", [
    ([100, 0, 300, 5, 128], 264, 1040),  # odd block counts: pair tiles across two groups
    ([256, 512, 128], 520, 640),         # groups on 256-row boundaries, the last block alone
    ([1, 1, 1], 64, 256),                # every pair tile holds two groups (or one and past M)
    ([513, 77], 2112, 384),              # ragged rows and a partial column block
    ([128], 256, 128),                   # one block: the second CTA's half past M
])
def test_contiguous_pair_tiles(group_rows, n, k, defer):
    """Contiguous layout on CTA pairs (forced): a pair tile whose two 128-row
    blocks belong to different groups runs once per group, each pass storing
    only its group's rows; padding rows stay untouched, the rest within the
    tolerance of the oracle, with the store warp or the promotion warps
    storing."""
    fg.fg_set_config_override(256, 1)
    fg.fg_set_pair_mode(1)
    fg.lib().fg_debug_set_pair_defer(defer)
    try:
        p = wl.contiguous(group_rows, n=n, k=k, seed=sum(group_rows) + n + k + 7 * defer)
        assert tuple(fg.fg_query_plan(1, p.M, p.G, n, k)[2:]) == (1, 0, defer)
        got = d_to_bits(run_contiguous(p))
    finally:
        fg.fg_set_config_override(0, 0)
        fg.fg_set_pair_mode(-1)
        fg.lib().fg_debug_set_pair_defer(-1)
    init = np.full((p.M, p.n), SENTINEL, np.uint16)
    ref, _ = oracle.grouped_contiguous(p.A, 0, p.sA, p.B, 0, p.sB, p.m_indices, init)
    pad = p.m_indices < 0
    assert np.array_equal(got[pad], ref[pad]), "padding rows were written"
    compare(got[~pad], ref[~pad], what=f"contiguous pairs {group_rows} defer={defer}")


def run_masked_allow_check(p, expect_check):
    if not expect_check:
        return run_masked(p)
    A = dev(p.A, fp8_dtype(0))
    D = torch.full((p.G, p.M_cap, p.n), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fg.fg_grouped_gemm_fp8_masked(A, fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.B, fp8_dtype(0)),
                                  dev(p.sB), D, dev(p.masked_m))
    st, _ = fg.fg_get_device_status()
    assert st == 6
    return D


def test_masked_equals_per_group_dense_bitwise(persistent_dense_plan):
    p = wl.masked(3, 256, n=512, k=640, seed=43, masked_m=[256, 100, 129])
    got = d_to_bits(run_masked(p))
    for g in range(p.G):
        v = int(p.masked_m[g])
        d = wl.Dense(v, p.n, p.k, p.A[g, :v], p.sA[g, :v], p.B[g], p.sB[g])
        assert np.array_equal(got[g, :v], d_to_bits(run_dense(d))), f"group {g}"


def test_masked_counts_read_on_device_only():
    """The same launch serves new counts written on the device (graph-style use)."""
    p = wl.masked(2, 256, n=256, k=256, seed=44, masked_m=[256, 256])
    A, B = dev(p.A, fp8_dtype(0)), dev(p.B, fp8_dtype(0))
    sA, sB = fg.fg_scales_a_to_mn_major(dev(p.sA)), dev(p.sB)
    mm = dev(np.array([10, 0], np.int32))
    D = torch.full((2, 256, 256), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fg.fg_grouped_gemm_fp8_masked(A, sA, B, sB, D, mm)  # warm-up outside the graph
        torch.cuda.synchronize()
        D.view(torch.int16).fill_(-1)
        with torch.cuda.graph(g, stream=s):
            fg.fg_grouped_gemm_fp8_masked(A, sA, B, sB, D, mm)
    for counts in ([10, 0], [0, 200], [256, 1]):
        D.view(torch.int16).fill_(-1)
        mm.copy_(torch.tensor(counts, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        got = d_to_bits(D)
        q = wl.Masked(p.G, p.M_cap, p.n, p.k, p.A, p.sA, p.B, p.sB, np.array(counts, np.int32))
        init = np.full((2, 256, 256), SENTINEL, np.uint16)
        ref, _ = oracle.grouped_masked(q.A, 0, q.sA, q.B, 0, q.sB, q.masked_m, init)
        valid = np.arange(256)[None, :] < np.array(counts)[:, None]
        assert np.array_equal(got[~valid], ref[~valid])
        compare(got[valid], ref[valid], what=f"graph replay {counts}")
    st, _ = fg.fg_get_device_status()
    assert st == 0


@pytest.mark.parametrize("plan", ["auto", "one_cta_128", "split3_256", "pair"])
def test_masked_many_groups(plan):
    """128 groups (the expert counts of large MoE layers): every tile walks the
    device-side counts of all groups to find its own; counts 0 and M_cap among
    them, rows past each count untouched, the rest against the oracle."""
    bn, split, pair = {"auto": (0, 0, -1), "one_cta_128": (128, 1, 0), "split3_256": (256, 3, 0),
                       "pair": (256, 1, 1)}[plan]
    G, M_cap = 128, 192
    counts = wl.rng_for(71).integers(0, M_cap, size=G, endpoint=True)
    counts[:4] = [0, M_cap, 1, 128]
    p = wl.masked(G, M_cap, n=264, k=384, seed=72, masked_m=counts)
    fg.fg_set_config_override(bn, split)
    fg.fg_set_pair_mode(pair)
    try:
        got = d_to_bits(run_masked(p))
    finally:
        fg.fg_set_config_override(0, 0)
        fg.fg_set_pair_mode(-1)
    init = np.full((p.G, p.M_cap, p.n), SENTINEL, np.uint16)
    ref, _ = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, init)
    valid = np.arange(M_cap)[None, :] < p.masked_m[:, None]
    assert np.array_equal(got[~valid], ref[~valid]), "rows past the count were written"
    compare(got[valid], ref[valid], what=f"masked G=128 ({plan})")


@pytest.mark.parametrize("G,n,k", wl.masked_shapes())
def test_masked_workload(G, n, k):
    """G groups of capacity 256 with seeded uniform counts; rows past the counts
    are checked bitwise in full, written rows on samples."""
    p = wl.masked(G, wl.MASKED_M_CAP, n=n, k=k, seed=wl.seed_for(3, wl.masked_shapes().index((G, n, k))))
    got = d_to_bits(run_masked(p))
    valid = np.arange(p.M_cap)[None, :] < p.masked_m[:, None]
    assert np.all(got[~valid] == SENTINEL), "rows past the count were written"
    gg, rr = np.nonzero(valid)
    if gg.size == 0:
        return
    rng = np.random.default_rng(G + n)
    pick = rng.choice(gg.size, size=min(gg.size, 4096), replace=False)
    cols = rng.integers(0, n, size=pick.size)
    # plus every column of the last valid row of each group
    extra_g, extra_r, extra_c = [], [], []
    for g in range(G):
        if p.masked_m[g] > 0:
            extra_g += [g] * n
            extra_r += [int(p.masked_m[g]) - 1] * n
            extra_c += list(range(n))
    G_ = np.concatenate([gg[pick], extra_g]).astype(np.int64)
    R_ = np.concatenate([rr[pick], extra_r]).astype(np.int64)
    C_ = np.concatenate([cols, extra_c]).astype(np.int64)
    ref, _ = oracle.grouped_masked_at(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, G_, R_, C_)
    compare(got[G_, R_, C_], ref, what=f"masked G={G} n={n} k={k} (sampled)")


@pytest.mark.parametrize("bn,split", [(256, 2), (128, 3), (256, 5), (128, 8)])
def test_grouped_split_plans_match_oracle(bn, split):
    """Split-K clusters on the grouped layouts: tiles past the device-side
    counts, padding tiles and untouched rows behave as in the persistent walk."""
    fg.fg_set_config_override(bn, split)
    try:
        p = wl.masked(6, 256, n=264, k=1040, seed=61, masked_m=[0, 1, 127, 128, 129, 256])
        got = d_to_bits(run_masked(p))
        init = np.full((p.G, p.M_cap, p.n), SENTINEL, np.uint16)
        ref, _ = oracle.grouped_masked(p.A, 0, p.sA, p.B, 0, p.sB, p.masked_m, init)
        valid = np.arange(p.M_cap)[None, :] < p.masked_m[:, None]
        assert np.array_equal(got[~valid], ref[~valid])
        compare(got[valid], ref[valid], what=f"masked split bn={bn} s={split}")

        c = wl.contiguous([100, 0, 300, 5, 128], n=264, k=1040, seed=62)
        got = d_to_bits(run_contiguous(c))
        init = np.full((c.M, c.n), SENTINEL, np.uint16)
        ref, _ = oracle.grouped_contiguous(c.A, 0, c.sA, c.B, 0, c.sB, c.m_indices, init)
        pad = c.m_indices < 0
        assert np.array_equal(got[pad], ref[pad])
        compare(got[~pad], ref[~pad], what=f"contiguous split bn={bn} s={split}")
    finally:
        fg.fg_set_config_override(0, 0)
