"""Host-side checks of the seeded input generators and of the separation
between the oracle, the generators and the CUDA library (no GPU needed)."""
import ast
import os

import numpy as np
import pytest

import oracle
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_rows_quantization_recipe():
    rng = wl.rng_for(1)
    x = rng.standard_normal((7, 300), dtype=np.float32)
    q, s = wl.quantize_rows(x)
    assert q.shape == (7, 300) and s.shape == (7, 3)
    dec = oracle.decode_table(0)[q.astype(np.int64)]
    for kb in range(3):
        blk = x[:, kb * 128:(kb + 1) * 128]
        np.testing.assert_array_equal(s[:, kb], np.abs(blk).max(axis=1) / np.float32(448.0))
        # each group's largest magnitude lands on +-448 (or just below by rounding)
        assert np.all(np.abs(dec[:, kb * 128:(kb + 1) * 128]).max(axis=1) >= 416)
    # E4M3 keeps 3 mantissa bits: relative error of every element <= 2^-4 (or subnormal)
    rec = dec * np.repeat(s, 128, axis=1)[:, :300]
    err = np.abs(rec - x)
    tol = np.maximum(np.abs(x) * 2.0 ** -4, np.repeat(s, 128, axis=1)[:, :300] * 2.0 ** -10)
    assert np.all(err <= tol)


def test_block_quantization_recipe():
    rng = wl.rng_for(2)
    x = rng.standard_normal((200, 260), dtype=np.float32)
    q, s = wl.quantize_blocks(x)
    assert s.shape == (2, 3)
    for nb in range(2):
        for kb in range(3):
            blk = x[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            assert s[nb, kb] == np.float32(np.abs(blk).max() / np.float32(448.0))


def test_zero_group_gets_unit_scale():
    x = np.zeros((2, 256), np.float32)
    x[1, 130] = 3.0
    q, s = wl.quantize_rows(x)
    assert s[0, 0] == 1.0 and s[0, 1] == 1.0 and s[1, 0] == 1.0
    assert np.all(q[0] == 0)


def test_e5m2_quantization_uses_its_max():
    x = wl.rng_for(3).standard_normal((128, 128), dtype=np.float32)
    q, s = wl.quantize_blocks(x, wl.E5M2)
    assert s[0, 0] == np.float32(np.abs(x).max() / np.float32(57344.0))
    assert np.abs(oracle.decode_table(1)[q.astype(np.int64)]).max() == 57344.0


def test_generators_are_deterministic():
    a = wl.dense(64, 128, 256, seed=5)
    b = wl.dense(64, 128, 256, seed=5)
    c = wl.dense(64, 128, 256, seed=6)
    assert np.array_equal(a.A, b.A) and np.array_equal(a.sB, b.sB)
    assert not np.array_equal(a.A, c.A)


def test_loguniform_scales_range():
    p = wl.dense(128, 256, 1024, seed=4, scales="loguniform")
    for s in (p.sA, p.sB):
        assert s.min() >= 2.0 ** -8 and s.max() <= 2.0 ** 8
        assert np.log2(s).std() > 3.0


def test_contiguous_layout_alignment():
    p = wl.contiguous([1, 127, 128, 129, 0], n=64, k=128, seed=8)
    assert p.M == 128 + 128 + 128 + 256
    assert p.M % 128 == 0
    # each 128-row tile holds one group id and possibly -1 padding
    for t in range(p.M // 128):
        ids = set(p.m_indices[t * 128:(t + 1) * 128].tolist()) - {-1}
        assert len(ids) <= 1
    assert p.valid_rows == 1 + 127 + 128 + 129


def test_masked_counts_in_range():
    p = wl.masked(16, 256, n=64, k=128, seed=9)
    assert p.masked_m.dtype == np.int32
    assert np.all((p.masked_m >= 0) & (p.masked_m <= 256))


def test_scales_mn_major_layout():
    s = np.arange(15, dtype=np.float32).reshape(5, 3)
    t = wl.scales_mn_major(s)
    assert t.shape == (3, 8)
    assert np.array_equal(t[:, :5], s.T) and np.all(t[:, 5:] == 0)
    g = np.arange(2 * 5 * 3, dtype=np.float32).reshape(2, 5, 3)
    tg = wl.scales_mn_major(g)
    assert tg.shape == (2, 3, 8) and np.array_equal(tg[1, :, :5], g[1].T)


def test_workload_shapes():
    assert len(wl.dense_sweep_shapes()) == 15
    assert (4096, 24576, 1536) in wl.dense_sweep_shapes()
    assert wl.large_dense_shapes()[1][2] == 8576


def _imports(path):
    tree = ast.parse(open(path).read())
    out = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module:
            out.add(node.module.split(".")[0])
    return out


@pytest.mark.parametrize("sub", ["oracle", "workloads"])
def test_oracle_and_generators_do_not_import_the_cuda_library(sub):
    for f in os.listdir(os.path.join(ROOT, sub)):
        if f.endswith(".py"):
            imps = _imports(os.path.join(ROOT, sub, f))
            assert "moe_grouped_gemm_nt_gb300" not in imps, (sub, f)
    if sub == "workloads":
        for f in os.listdir(os.path.join(ROOT, sub)):
            if f.endswith(".py"):
                assert "oracle" not in _imports(os.path.join(ROOT, sub, f))


def test_cuda_library_does_not_use_the_oracle():
    pkg = os.path.join(ROOT, "moe_grouped_gemm_nt_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            p = os.path.join(dirpath, f)
            if f.endswith(".py"):
                imps = _imports(p)
                assert "oracle" not in imps and "workloads" not in imps, p
            if f.endswith((".cu", ".cuh", ".h", ".cpp")):
                assert "oracle" not in open(p).read().lower(), p


def test_sample_positions_cover_boundary_tiles():
    """The sampled check of the largest problems covers every element of the
    four corner tiles and of the last row block and last column block (the
    tiles where partial-tile and clipping logic lives), each position once, and
    at least one element of every other tile."""
    import sys
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from gpu_common import sample_positions

    rows, cols = 1000, 700   # ragged in both directions: last blocks of 104 rows, 188 columns
    r, c = sample_positions(rows, cols, seed=3, n_rows_full=2, boundary_tiles=True)
    lin = r * cols + c
    assert np.unique(lin).size == lin.size
    hit = np.zeros((rows, cols), bool)
    hit[r, c] = True
    assert hit[896:, :].all() and hit[:, 512:].all()      # last row block, last column block
    assert hit[:128, :256].all()                           # top-left corner tile
    for t0 in range(0, rows, 128):
        for c0 in range(0, cols, 256):
            assert hit[t0:t0 + 128, c0:c0 + 256].any()
