"""COO SpMV (row-sorted triplets, work split by nonzeros) against the fp64
oracle: one and many chunks, rows that span chunks or end exactly on a chunk
boundary, empty rows at the ends and in the middle, duplicates, alpha/beta,
determinism, and index/order errors reported without any fault."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import assert_within, dev

pytestmark = pytest.mark.gpu

CHUNK = 2048


def run_coo(M, K, row, col, val, x, y0, alpha, beta):
    y = dev(y0)
    spx.spx_spmv_coo(M, K, dev(row), dev(col), dev(val), dev(x), y, alpha, beta)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    return y.cpu().numpy()


def check(M, K, row, col, val, seed, alpha=1.0, beta=0.0):
    x = synth.uniform(seed, synth.T_X, K)
    y0 = synth.uniform(seed, synth.T_Y, M)
    got = run_coo(M, K, row, col, val, x, y0, alpha, beta)
    ref, bound = oracle.spmv_coo(M, K, row, col, val, x, alpha, beta, y0)
    assert_within(got, ref, bound, what=f"M={M} nnz={col.size}")
    return got


def from_lengths(seed, K, lengths):
    lengths = np.asarray(lengths, np.int32)
    row, col = synth.cols_uniform(seed, K, lengths)
    return row, col, synth.uniform(seed, synth.T_VAL, row.size)


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 1, 1), (37, 50, 0, 9), (500, 300, 0, 30), (4000, 4000, 1, 16),
                                           (20000, 9000, 0, 12)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-0.5, 2.0)])
def test_random(M, K, lmin, lmax, alpha, beta):
    d = synth.random_coo(M + K, M, K, lmin, lmax)
    check(M, K, d["row"], d["col"], d["val"], seed=M, alpha=alpha, beta=beta)


@pytest.mark.parametrize("lengths", [
    [CHUNK],                                  # one row, exactly one chunk
    [CHUNK, CHUNK, 1, 2 * CHUNK - 1, 5],      # rows ending on chunk boundaries
    [3, 7000, 2, 9000],                       # rows spanning three to five chunks
    [0, 0, 5000, 0, 0, 0, 1, 0, 2047, 0],     # empty rows around long ones
    [1] * 5000 + [0] * 40 + [3000],           # many short rows, a gap, a long tail row
])
def test_chunk_boundaries(lengths):
    row, col, val = from_lengths(21, 12000, lengths)
    check(len(lengths), 12000, row, col, val, seed=21, alpha=1.5, beta=-0.5)


def test_single_row_many_chunks():
    row, col, val = from_lengths(22, 40000, [30000])
    check(1, 40000, row, col, val, seed=22, alpha=1.0, beta=1.0)


def test_duplicates_summed():
    M, K = 64, 64
    row = np.repeat(np.arange(M, dtype=np.int32), 40)
    col = np.tile(np.array([3, 3, 5, 3] * 10, np.int32), M)
    val = synth.uniform(23, synth.T_VAL, row.size)
    check(M, K, row, col, val, seed=23)


def test_beta_zero_does_not_read_y():
    d = synth.random_coo(24, 3000, 2000, 0, 8)
    x = synth.uniform(24, synth.T_X, 2000)
    got = run_coo(3000, 2000, d["row"], d["col"], d["val"], x, np.full(3000, np.nan, np.float32), 1.0, 0.0)
    ref, bound = oracle.spmv_coo(3000, 2000, d["row"], d["col"], d["val"], x)
    assert_within(got, ref, bound)


@pytest.mark.parametrize("beta", [0.0, -3.0])
def test_no_entries(beta):
    y0 = synth.uniform(25, synth.T_Y, 777)
    z = np.zeros(0, np.int32)
    got = run_coo(777, 5, z, z, np.zeros(0, np.float32), np.ones(5, np.float32), y0, 1.0, beta)
    assert np.array_equal(got, np.float32(beta) * y0)


def test_deterministic_bitwise():
    row, col, val = from_lengths(26, 50000, synth.lengths_poisson(26, 30000, 12.0))
    x = synth.uniform(26, synth.T_X, 50000)
    y0 = synth.uniform(26, synth.T_Y, 30000)
    a = run_coo(30000, 50000, row, col, val, x, y0, 1.0, 0.5)
    b = run_coo(30000, 50000, row, col, val, x, y0, 1.0, 0.5)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_power_law_rows():
    """Power-law row lengths (Zipf 2.1, mean 16, up to 20000): short and very long rows together."""
    lengths, _ = synth.lengths_zipf(27, 60000, 2.1, 20000, 16.0)
    row, col, val = from_lengths(27, 60000, lengths)
    check(60000, 60000, row, col, val, seed=27, alpha=1.0, beta=0.5)


@pytest.mark.parametrize("bad", ["row_high", "row_negative", "col_high", "unsorted"])
def test_bad_indices_reported(bad):
    """Bad triplets are skipped by the kernel's own checks and reported; nothing
    outside x, y or the scratch buffer is touched (y's guard words stay intact)."""
    M, K = 5000, 3000
    d = synth.random_coo(28, M, K, 1, 8)
    row, col = d["row"].copy(), d["col"].copy()
    k = row.size // 2
    if bad == "row_high":
        row[k:k + 3] = M + 7
        row[k + 3:] = np.maximum(row[k + 3:], M + 7)
        want = -2
    elif bad == "row_negative":
        row[:3] = -4
        want = -2
    elif bad == "col_high":
        col[k] = K + 100
        want = -2
    else:
        row[k], row[k + 1] = row[k + 1] + 1, row[k]
        want = -3
    guard = torch.full((M + 64,), 123.0, device="cuda")
    y = guard[32:32 + M]
    spx.spx_spmv_coo(M, K, dev(row), dev(col), dev(d["val"]), dev(synth.uniform(28, synth.T_X, K)), y, 1.0, 0.0)
    assert spx.spx_last_device_error() == want
    g = guard.cpu().numpy()
    assert np.all(g[:32] == 123.0) and np.all(g[32 + M:] == 123.0)
    assert spx.spx_last_device_error() == 0  # the word is cleared by the read


@pytest.mark.slow
def test_power_law_full_size_every_row():
    """The benchmarked COO workload at full size: the 4,194,304-row power-law matrix (67.1M row-sorted
    triplets, 32,769 chunks, rows of up to ~10^5 entries spanning many chunks), y = Ax + 0.5y, in the
    launch configuration the benchmark times -- every output row against the oracle, and bitwise
    equal on a second run."""
    cfg = synth.power_law_rows()
    M, K = cfg["M"], cfg["K"]
    row, col, val = cfg["row"], cfg["col"], cfg["val"]
    assert np.all(np.diff(row) >= 0)
    drow, dcol, dval, dx = dev(row), dev(col), dev(val), dev(cfg["x"])
    scratch = torch.empty(max(1, spx.spx_spmv_coo_scratch_bytes(row.size) // 4), device="cuda")
    outs = []
    for _ in range(2):
        y = dev(cfg["y"])
        spx.spx_spmv_coo(M, K, drow, dcol, dval, dx, y, cfg["alpha"], cfg["beta"], scratch=scratch)
        torch.cuda.synchronize()
        assert spx.spx_last_device_error() == 0
        outs.append(y.cpu().numpy())
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    ref, bound = oracle.spmv_coo(M, K, row, col, val, cfg["x"], cfg["alpha"], cfg["beta"], cfg["y"])
    assert_within(outs[0], ref, bound, what="power-law COO full size")
    # the rows that cross chunk boundaries are among them; make sure there are many
    starts = np.arange(0, row.size, CHUNK)
    crossing = np.unique(row[starts[1:]][row[starts[1:]] == row[starts[1:] - 1]])
    assert crossing.size > 1000
