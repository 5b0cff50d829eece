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
