"""SELL-C-sigma SpMV (slices of 32 rows, column-major, long rows cut into
pieces) against the fp64 oracle of the CSR product: random matrices under
several (sigma, piece), long and empty rows, alpha/beta, determinism, and the
4,194,304^2 power-law workload on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import assert_within, dev

pytestmark = pytest.mark.gpu


def run_sell(M, K, rp, col, val, x, y0, alpha, beta, opts=None):
    S = spx.Sell(M, K, rp, col, val, opts=opts)
    y = dev(y0)
    spx.spx_spmv_sell(S, dev(x), y, alpha, beta)
    torch.cuda.synchronize()
    return y.cpu().numpy(), S


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 1, 1), (37, 50, 0, 9), (1000, 700, 0, 40), (5000, 6000, 0, 700)])
@pytest.mark.parametrize("opts", [None, dict(sigma=32, piece=8), dict(sigma=1024, piece=64)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-2.0, 0.5)])
def test_random(M, K, lmin, lmax, opts, alpha, beta):
    d = synth.random_coo(M + 3, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    x = synth.uniform(M, synth.T_X, K)
    y0 = synth.uniform(M, synth.T_Y, M)
    got, _ = run_sell(M, K, rp, col, val, x, y0, alpha, beta, opts)
    ref, bound = oracle.spmv(M, rp, col, val, x, alpha, beta, y0)
    assert_within(got, ref, bound, what=f"M={M} opts={opts}")


def test_long_and_empty_rows_beta_zero_write_only():
    L = np.zeros(300, np.int32)
    L[5] = 20000
    L[6] = 257
    L[100:140] = 3
    L[299] = 4096
    row, col = synth.cols_uniform(51, 30000, L)
    rp, col, val = oracle.build_csr(300, 30000, row, col, synth.uniform(51, synth.T_VAL, row.size))
    x = synth.uniform(51, synth.T_X, 30000)
    got, S = run_sell(300, 30000, rp, col, val, x, np.full(300, np.nan, np.float32), 1.0, 0.0)
    assert S.info["long_rows"] == 3
    ref, bound = oracle.spmv(300, rp, col, val, x)
    assert_within(got, ref, bound)


def test_deterministic_bitwise():
    L, _ = synth.lengths_zipf(52, 100000, 2.1, 30000, 16.0)
    row, col = synth.cols_uniform(52, 100000, L)
    rp, col, val = oracle.build_csr(100000, 100000, row, col, synth.uniform(52, synth.T_VAL, row.size))
    x = synth.uniform(52, synth.T_X, 100000)
    y0 = synth.uniform(52, synth.T_Y, 100000)
    a, _ = run_sell(100000, 100000, rp, col, val, x, y0, 1.0, 0.5)
    b, _ = run_sell(100000, 100000, rp, col, val, x, y0, 1.0, 0.5)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    ref, bound = oracle.spmv(100000, rp, col, val, x, 1.0, 0.5, y0)
    assert_within(a, ref, bound)


@pytest.mark.slow
def test_power_law_full_size_sampled():
    """4,194,304^2, Zipf(2.1) rows with mean 16, alpha 1, beta 0.5, default
    SELL options: 20,000 sampled rows, every row cut into pieces among them."""
    c = synth.power_law_rows()
    M, K = c["M"], c["K"]
    rp, col, val = spx.spx_build_csr(M, K, c["row"], c["col"], c["val"])
    S = spx.Sell(M, K, rp, col, val)
    y = dev(c["y"])
    spx.spx_spmv_sell(S, dev(c["x"]), y, c["alpha"], c["beta"])
    torch.cuda.synchronize()
    lens = np.diff(rp)
    rows = np.unique(np.concatenate([np.flatnonzero(lens > 256),
                                     np.random.default_rng(5).integers(0, M, 20000)])).astype(np.int32)
    ref, bound = oracle.spmv(M, rp, col, val, c["x"], c["alpha"], c["beta"], c["y"], rows=rows)
    got = y[torch.from_numpy(rows).long().cuda()].cpu().numpy()
    assert_within(got, ref, bound, what="power-law SELL")


def _sell_arrays_equal(Sh, Sd):
    assert Sd.info == Sh.info
    for a, b in zip(Sh.arrays(), Sd.arrays()):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 0, 0), (1, 5, 5, 5), (37, 50, 0, 9), (1000, 700, 0, 40),
                                          (5000, 6000, 0, 700), (3000, 100, 0, 0)])
@pytest.mark.parametrize("opts", [None, dict(sigma=32, piece=8), dict(sigma=64, piece=1), dict(sigma=4096, piece=1000)])
def test_device_build_equals_host_build(M, K, lmin, lmax, opts):
    """SELL-C-sigma built on the GPU from device arrays: the same image as the host build,
    read back before and after the upload, and the same product bit for bit."""
    d = synth.random_coo(M + 5, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    Sh = spx.Sell(M, K, rp, col, val, opts=opts)
    Sd = spx.Sell(M, K, dev(rp), dev(col), dev(val), opts=opts, upload=False)
    _sell_arrays_equal(Sh, Sd)  # from the library's device copy
    Sd.image = torch.empty_like(Sh.image)
    Sd.scratch = torch.empty_like(Sh.scratch)
    spx._check(spx._lib().spx_sell_upload(Sd.handle, spx._ptr(Sd.image), Sd.image.numel() * 4, None), "upload")
    torch.cuda.synchronize()
    _sell_arrays_equal(Sh, Sd)  # from the uploaded image (the bytes between sections are unspecified)
    x = synth.uniform(M + 1, synth.T_X, K)
    y0 = synth.uniform(M + 1, synth.T_Y, M)
    yh, yd = dev(y0), dev(y0)
    spx.spx_spmv_sell(Sh, dev(x), yh, 1.5, -0.5)
    spx.spx_spmv_sell(Sd, dev(x), yd, 1.5, -0.5)
    assert torch.equal(yh, yd)


def test_device_build_power_law():
    """The 4,194,304^2 power-law workload built on the GPU equals the host build."""
    c = synth.power_law_rows()
    M, K = c["M"], c["K"]
    rp, col, val = spx.spx_build_csr(M, K, c["row"], c["col"], c["val"])
    Sh = spx.Sell(M, K, rp, col, val)
    Sd = spx.Sell(M, K, dev(rp), dev(col), dev(val))
    _sell_arrays_equal(Sh, Sd)


def test_device_build_rejects_bad_input():
    for rp, col, code in [([1, 2, 3], [0, 1, 1], -1),   # row_ptr[0] != 0
                          ([0, 3, 2], [0, 1], -3),      # decreasing
                          ([0, 2, 3], [0, 9, 1], -2)]:  # column outside [0, K)
        with pytest.raises(spx.SpxError) as e:
            spx.Sell(2, 4, dev(np.array(rp, np.int32)), dev(np.array(col, np.int32)),
                     dev(np.ones(len(col), np.float32)))
        assert e.value.code == code
