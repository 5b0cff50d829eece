"""Format builders on the GPU (stable radix sorts): COO -> CSR and
CSR -> CSR(A^T) with device arrays must equal the oracle's host builds bit for
bit -- shuffled input, duplicates kept in input order, empty rows and
columns, every value width, sizes that are not powers of two, and the full
4,194,304^2 power-law matrix; bad indices are rejected."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx

pytestmark = pytest.mark.gpu


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 0, 1), (7, 5, 0, 5), (1000, 777, 0, 40), (3000, 70000, 0, 9),
                                          (50, 50, 0, 0), (20000, 300, 1, 60), (5000, 1 << 24, 0, 12)])
@pytest.mark.parametrize("dtype", [np.float32, np.uint16, np.float64, np.uint8])
def test_build_csr_device_equals_oracle(M, K, lmin, lmax, dtype):
    d = synth.random_coo(101 + M, M, K, lmin, lmax)
    perm = synth.permutation(102 + M, d["row"].size)
    row, col = d["row"][perm], d["col"][perm]
    val = d["val"][perm] if dtype is np.float32 else (np.abs(d["val"][perm]) * 250).astype(dtype)
    want = oracle.build_csr(M, K, row, col, val)
    got = spx.spx_build_csr(M, K, cuda(row), cuda(col), cuda(val))
    torch.cuda.synchronize()
    for w, g in zip(want, got):
        assert np.array_equal(w, host(g))


def test_build_csr_device_duplicates_in_input_order():
    row = np.array([2, 0, 2, 2, 0, 1, 2], np.int32)
    col = np.array([5, 1, 5, 0, 1, 3, 5], np.int32)
    val = np.arange(7, dtype=np.float32)
    want = oracle.build_csr(3, 6, row, col, val)
    got = spx.spx_build_csr(3, 6, cuda(row), cuda(col), cuda(val))
    for w, g in zip(want, got):
        assert np.array_equal(w, host(g))
    assert host(got[2]).tolist() == [1.0, 4.0, 5.0, 3.0, 0.0, 2.0, 6.0]


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 0, 1), (7, 5, 0, 5), (1000, 777, 0, 40), (300, 90000, 0, 300),
                                          (60000, 500, 0, 5), (50, 50, 0, 0)])
@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_transpose_device_equals_oracle(M, K, lmin, lmax, dtype):
    d = synth.random_coo(103 + K, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    v = val if dtype is np.float32 else synth.to_bf16_bits(val)
    want = oracle.transpose(M, K, rp, col, v)
    got = spx.spx_transpose_csr(M, K, cuda(rp), cuda(col), cuda(v))
    for w, g in zip(want, got):
        assert np.array_equal(w, host(g))


def test_device_builders_reject_bad_input():
    row = cuda(np.array([0, 3], np.int32))
    col = cuda(np.array([0, 1], np.int32))
    one = cuda(np.ones(2, np.float32))
    cases = [(lambda: spx.spx_build_csr(3, 2, row, col, one), -2),                       # row 3 >= M
             (lambda: spx.spx_build_csr(4, 1, row, col, one), -2),                       # col 1 >= K
             (lambda: spx.spx_transpose_csr(2, 2, cuda(np.array([0, 2, 1], np.int32)), col, one), -1),
             (lambda: spx.spx_transpose_csr(3, 2, cuda(np.array([0, 2, 0, 2], np.int32)), col, one), -3),
             (lambda: spx.spx_transpose_csr(2, 2, cuda(np.array([0, 1, 2], np.int32)),
                                            cuda(np.array([0, 2], np.int32)), one), -2)]
    for f, code in cases:
        with pytest.raises(spx.SpxError) as e:
            f()
        assert e.value.code == code


@pytest.mark.slow
def test_power_law_full_size_device_build():
    """67.1M entries, shuffled: the GPU build and transpose equal the host ones bit for bit."""
    c = synth.power_law_rows()
    M, K = c["M"], c["K"]
    perm = synth.permutation(104, c["row"].size)
    row, col, val = c["row"][perm], c["col"][perm], c["val"][perm]
    want = spx.spx_build_csr(M, K, row, col, val)  # host counting sort
    got = spx.spx_build_csr(M, K, cuda(row), cuda(col), cuda(val))
    for w, g in zip(want, got):
        assert np.array_equal(w, host(g))
    wt = spx.spx_transpose_csr(M, K, *want)
    gt = spx.spx_transpose_csr(M, K, *got)
    for w, g in zip(wt, gt):
        assert np.array_equal(w, host(g))


def _shuffle_within_rows(seed, rp, col, val):
    """Same matrix, columns no longer ascending inside each row."""
    key = synth.uniform(seed, 9, col.size, 0.0, 1.0)
    rows = np.repeat(np.arange(rp.size - 1), np.diff(rp))
    order = np.lexsort((key, rows))
    return col[order], val[order]


@pytest.mark.parametrize("M,K,lmin,lmax,br,bc", [(1, 1, 0, 1, 1, 1), (7, 5, 0, 5, 2, 3), (1000, 777, 0, 40, 16, 16),
                                                 (300, 90000, 0, 300, 64, 64), (4097, 5000, 1, 12, 128, 8),
                                                 (50, 50, 0, 0, 4, 4), (2000, 3000, 0, 30, 1, 64),
                                                 (2000, 3000, 0, 30, 33, 1)])
@pytest.mark.parametrize("dtype", [np.float32, np.uint16, np.float64])
def test_build_bsr_device_equals_oracle(M, K, lmin, lmax, br, bc, dtype):
    d = synth.random_coo(105 + M + br, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    v = val.astype(dtype) if dtype is not np.uint16 else synth.to_bf16_bits(val)
    want = oracle.build_bsr(M, K, rp, col, v, br, bc)
    got = spx.spx_build_bsr(M, K, cuda(rp), cuda(col), cuda(v), br, bc)
    assert got[3] == want[3]
    for w, g in zip(want[:3], got[:3]):
        assert np.array_equal(w, host(g))
    # columns out of order inside the rows: same blocks
    c2, v2 = _shuffle_within_rows(106 + M, rp, col, v)
    got2 = spx.spx_build_bsr(M, K, cuda(rp), cuda(c2), cuda(v2), br, bc)
    for w, g in zip(want[:3], got2[:3]):
        assert np.array_equal(w, host(g))


def test_build_bsr_device_block_sparse_workload():
    """The tensor-core workload's shape (16,384^2, 64 x 64 blocks, 26 per block-row), bf16 bits."""
    c = synth.block_sparse()
    M, K, bs = c["M"], c["K"], c["bs"]
    rp, col, val = oracle.build_csr(M, K, c["row"], c["col"], c["val_bf16"])
    want = oracle.build_bsr(M, K, rp, col, val, bs, bs)
    got = spx.spx_build_bsr(M, K, cuda(rp), cuda(col), cuda(val), bs, bs)
    assert got[3] == want[3] == 1.0
    for w, g in zip(want[:3], got[:3]):
        assert np.array_equal(w, host(g))


def test_build_bsr_device_rejects_bad_input():
    one = cuda(np.ones(3, np.float32))
    rp = cuda(np.array([0, 2, 3], np.int32))
    cases = [(cuda(np.array([0, 0, 1], np.int32)), rp, -4),                       # (0, 0) twice
             (cuda(np.array([1, 0, 1], np.int32)), cuda(np.array([0, 3, 3], np.int32)), -4),  # not adjacent
             (cuda(np.array([0, 4, 1], np.int32)), rp, -2),                       # col 4 >= K
             (cuda(np.array([0, 1, 1], np.int32)), cuda(np.array([0, 3, 2], np.int32)), -3),  # row_ptr decreasing
             (cuda(np.array([0, 1, 1], np.int32)), cuda(np.array([1, 2, 3], np.int32)), -1)]  # row_ptr[0] != 0
    for c, r, code in cases:
        with pytest.raises(spx.SpxError) as e:
            spx.spx_build_bsr(2, 4, r, c, one, 2, 2)
        assert e.value.code == code


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 0, 1), (7, 5, 0, 5), (1000, 777, 0, 40), (300, 90000, 0, 300),
                                          (4097, 200, 1, 120), (50, 50, 0, 0), (64, 64, 64, 64), (130, 70, 0, 70)])
@pytest.mark.parametrize("dtype", [np.float32, np.uint16, np.float64, np.uint8])
def test_build_wcsr_device_equals_oracle(M, K, lmin, lmax, dtype):
    d = synth.random_coo(107 + M + K, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    v = synth.to_bf16_bits(val) if dtype is np.uint16 else (
        (np.abs(val) * 250).astype(dtype) if dtype is np.uint8 else val.astype(dtype))
    want = oracle.build_wcsr(M, K, rp, col, v)
    got = spx.spx_build_wcsr(M, K, cuda(rp), cuda(col), cuda(v))
    assert got[3] == want[3]
    for w, g in zip(want[:3], got[:3]):
        assert np.array_equal(w, host(g))
    c2, v2 = _shuffle_within_rows(108 + M, rp, col, v)
    got2 = spx.spx_build_wcsr(M, K, cuda(rp), cuda(c2), cuda(v2))
    for w, g in zip(want[:3], got2[:3]):
        assert np.array_equal(w, host(g))


def test_build_wcsr_device_window_pool_workload():
    """The WCSR workload's shape (16,384 rows, 64-row windows over a 512-column pool each)."""
    c = synth.window_pool()
    M, K = c["M"], c["K"]
    rp, col, val = oracle.build_csr(M, K, c["row"], c["col"], c["val_bf16"])
    want = oracle.build_wcsr(M, K, rp, col, val)
    got = spx.spx_build_wcsr(M, K, cuda(rp), cuda(col), cuda(val))
    assert got[3] == want[3]
    for w, g in zip(want[:3], got[:3]):
        assert np.array_equal(w, host(g))


def test_build_wcsr_device_rejects_bad_input():
    one = cuda(np.ones(3, np.float32))
    rp = cuda(np.array([0, 2, 3], np.int32))
    cases = [(cuda(np.array([1, 1, 0], np.int32)), rp, -4),                       # (0, 1) twice
             (cuda(np.array([1, 0, 1], np.int32)), cuda(np.array([0, 3, 3], np.int32)), -4),  # not adjacent
             (cuda(np.array([1, 4, 0], np.int32)), rp, -2),                       # col 4 >= K
             (cuda(np.array([1, 2, 0], np.int32)), cuda(np.array([0, 3, 2], np.int32)), -3),  # row_ptr decreasing
             (cuda(np.array([1, 2, 0], np.int32)), cuda(np.array([1, 2, 3], np.int32)), -1)]  # row_ptr[0] != 0
    for c, r, code in cases:
        with pytest.raises(spx.SpxError) as e:
            spx.spx_build_wcsr(2, 4, r, c, one)
        assert e.value.code == code


@pytest.mark.parametrize("M,lmin,lmax", [(1, 0, 0), (1, 5, 5), (7, 0, 5), (1000, 0, 40), (4097, 1, 3000),
                                         (300000, 0, 12), (50, 0, 0)])
def test_row_stats_device_equals_host(M, lmin, lmax):
    lengths = synth.lengths_uniform(109 + M, M, lmin, lmax)
    rp = np.zeros(M + 1, np.int32)
    rp[1:] = np.cumsum(lengths)
    want = spx.spx_row_stats(M, rp)
    got = spx.spx_row_stats(M, cuda(rp))
    assert got == want
    assert got == oracle.row_stats(M, rp)


def test_row_stats_device_power_law():
    """4,194,304 rows, lengths from 1 to ~10^5: every field equals the host's, and the percentiles the sorted lengths'."""
    M = 4_194_304
    lengths, _ = synth.lengths_zipf(2, M, 2.1, 200_000, 16.0)  # the power-law workload's row lengths
    rp = np.zeros(M + 1, np.int32)
    rp[1:] = np.cumsum(lengths)
    got = spx.spx_row_stats(M, cuda(rp))
    assert got == spx.spx_row_stats(M, rp)
    assert got == oracle.row_stats(M, rp)
    srt = np.sort(lengths)
    assert [got["p50"], got["p95"], got["p99"]] == [int(srt[(q * M + 99) // 100 - 1]) for q in (50, 95, 99)]
    assert got["max"] == int(srt[-1]) and got["min"] == int(srt[0])


@pytest.mark.parametrize("M,K", [(0, 0), (0, 7), (5, 0), (130, 0)])
def test_device_builders_empty_matrices(M, K):
    """No rows or no columns (so no entries): every GPU builder returns the host builders' empty forms."""
    rp = np.zeros(M + 1, np.int32)
    col = np.zeros(0, np.int32)
    val = np.zeros(0, np.float32)
    for want, got in ((oracle.build_bsr(M, K, rp, col, val, 4, 4),
                       spx.spx_build_bsr(M, K, cuda(rp), cuda(col), cuda(val), 4, 4)),
                      (oracle.build_wcsr(M, K, rp, col, val), spx.spx_build_wcsr(M, K, cuda(rp), cuda(col), cuda(val))),
                      (oracle.transpose(M, K, rp, col, val), spx.spx_transpose_csr(M, K, cuda(rp), cuda(col), cuda(val))),
                      (oracle.build_csr(M, K, col, col, val), spx.spx_build_csr(M, K, cuda(col), cuda(col), cuda(val)))):
        for w, g in zip(want[:3], got[:3]):
            assert np.array_equal(w, host(g))
    assert spx.spx_row_stats(M, cuda(rp)) == spx.spx_row_stats(M, rp)
    ph, pd = spx.spx_plan_csr(M, K, 0, rp), spx.spx_plan_csr(M, K, 0, cuda(rp))
    assert ph.info == pd.info
    Sh, Sd = spx.Sell(M, K, rp, col, val), spx.Sell(M, K, cuda(rp), cuda(col), cuda(val))
    assert Sh.info == Sd.info
    for a, b in zip(Sh.arrays(), Sd.arrays()):
        assert np.array_equal(a, b)
