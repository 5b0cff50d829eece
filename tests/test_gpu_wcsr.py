"""WCSR SpMM on the tensor cores (bf16 in, fp32 accumulate; B rows gathered
into the swizzled tile by cp.async) against the fp64 oracle: exact
small-integer products, several chunks per window, empty windows, a partial
last window, padded leading dimensions, alpha/beta, determinism, and the
16384^2 window-pool workload at N = 1024 on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import BF16_ABS, BF16_REL, assert_within

pytestmark = pytest.mark.gpu


def bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def run_wcsr(M, K, rp, col, vbits, Bbits, N, ldb=None, ldc=None, alpha=1.0, beta=0.0, C0=None):
    wp, wc, wv, fill = spx.spx_build_wcsr(M, K, rp, col, vbits)
    ldb = ldb or N
    ldc = ldc or N
    Bfull = np.zeros((K, ldb), np.uint16)
    Bfull[:, :N] = Bbits
    Bd = bits(Bfull)[:, :N]
    Cfull = np.full((M, ldc), -7.0, np.float32)
    if C0 is not None:
        Cfull[:, :N] = C0
    Cd = torch.from_numpy(Cfull).cuda()
    spx.spx_spmm_wcsr(M, K, torch.from_numpy(wp).cuda(), torch.from_numpy(wc).cuda(), bits(wv.reshape(-1)), Bd,
                      Cd[:, :N], alpha, beta)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    out = Cd.cpu().numpy()
    assert np.all(out[:, N:] == -7.0)
    return out[:, :N], wp, fill


def test_small_integers_exact():
    """Entries and B in {-3..3}: every partial sum is an exact fp32 integer."""
    M, K, N = 150, 700, 256
    d = synth.random_coo(71, M, K, 0, 120, values="int")
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    B = np.floor(synth.uniform(71, synth.T_B, K * N, -3, 4)).astype(np.float32).reshape(K, N)
    got, wp, _ = run_wcsr(M, K, rp, col, synth.to_bf16_bits(val), synth.to_bf16_bits(B).reshape(K, N), N)
    assert np.diff(wp).max() >= 3  # several chunks in a window
    A = np.zeros((M, K))
    np.add.at(A, (d["row"], d["col"]), d["val"].astype(np.float64))
    assert np.array_equal(got, A @ B.astype(np.float64))


@pytest.mark.parametrize("M,K,lmin,lmax,N,ldb,ldc", [
    (64, 64, 1, 64, 128, None, None),
    (100, 3000, 0, 300, 384, 392, 400),       # partial last window, padded leading dimensions
    (300, 500, 0, 0, 128, None, None),        # no entries at all
    (1000, 20000, 0, 40, 128, None, None),    # many windows, wide unions
])
def test_random(M, K, lmin, lmax, N, ldb, ldc):
    d = synth.random_coo(72 + M, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    vb = synth.to_bf16_bits(val)
    Bb = synth.to_bf16_bits(synth.normal_f32(72, synth.T_B, K * N, 1.0)).reshape(K, N)
    got, _, _ = run_wcsr(M, K, rp, col, vb, Bb, N, ldb, ldc)
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(vb), synth.bf16_bits_to_f32(Bb).reshape(K, N))
    assert_within(got, ref, bound, 1e-5, 1e-6, what=f"M={M} K={K}")


def test_empty_windows_and_alpha_beta():
    L = np.zeros(320, np.int32)
    L[64:128] = 5          # window 1 only; windows 0, 2, 3, 4 empty
    L[300] = 77
    row, col = synth.cols_uniform(73, 2000, L)
    rp, col, val = oracle.build_csr(320, 2000, row, col, synth.uniform(73, synth.T_VAL, row.size))
    vb = synth.to_bf16_bits(val)
    Bb = synth.to_bf16_bits(synth.uniform(73, synth.T_B, 2000 * 256)).reshape(2000, 256)
    C0 = synth.uniform(73, synth.T_Y, 320 * 256).reshape(320, 256)
    for alpha, beta in [(1.0, 0.0), (-0.5, 2.0)]:
        got, wp, _ = run_wcsr(320, 2000, rp, col, vb, Bb, 256, alpha=alpha, beta=beta, C0=C0)
        assert (np.diff(wp) == 0).sum() == 3
        ref, bound = oracle.spmm(320, rp, col, synth.bf16_bits_to_f32(vb), synth.bf16_bits_to_f32(Bb).reshape(2000, 256),
                                 alpha, beta, C0)
        assert_within(got, ref, bound, 1e-5, 1e-6, what=f"alpha={alpha} beta={beta}")


def test_deterministic_bitwise():
    d = synth.random_coo(74, 640, 5000, 0, 100)
    rp, col, val = oracle.build_csr(640, 5000, d["row"], d["col"], d["val"])
    vb = synth.to_bf16_bits(val)
    Bb = synth.to_bf16_bits(synth.uniform(74, synth.T_B, 5000 * 512)).reshape(5000, 512)
    a, _, _ = run_wcsr(640, 5000, rp, col, vb, Bb, 512)
    b, _, _ = run_wcsr(640, 5000, rp, col, vb, Bb, 512)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.slow
def test_window_pool_full_size_sampled():
    """16384^2, 64-row windows with 512-column pools, l ~ U{32..96}, N = 1024:
    two sampled rows of every window against the oracle."""
    c = synth.window_pool()
    M, K, N = c["M"], c["K"], c["N"]
    rp, col, val = spx.spx_build_csr(M, K, c["row"], c["col"], c["val_bf16"])
    wp, wc, wv, fill = spx.spx_build_wcsr(M, K, rp, col, val)
    assert 0.1 < fill < 0.15
    Cd = torch.empty(M, N, device="cuda")
    spx.spx_spmm_wcsr(M, K, torch.from_numpy(wp).cuda(), torch.from_numpy(wc).cuda(), bits(wv.reshape(-1)),
                      bits(c["B_bf16"]), Cd)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    rows = np.sort(np.concatenate([np.arange(0, M, 64), np.arange(37, M, 64)])).astype(np.int32)
    got = Cd[torch.from_numpy(rows).long().cuda()].cpu().numpy()
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(val), synth.bf16_bits_to_f32(c["B_bf16"]).reshape(K, N),
                             rows=rows)
    assert_within(got, ref, bound, BF16_REL, BF16_ABS, what="window-pool")
    assert_within(got, ref, bound, 1e-5, 1e-6, what="window-pool fp32-level")


def _skewed_wcsr(M, N, seed=7):
    c = synth.window_pool_skewed(seed, M=M, N=N)
    rp, col, val = oracle.build_csr(M, c["K"], c["row"], c["col"], c["val_bf16"])
    wp, wc, wv, _ = oracle.build_wcsr(M, c["K"], rp, col, val)
    return c, rp, col, val, wp, wc, wv


@pytest.mark.parametrize("max_chunks", [0, 1, 4, 7])
@pytest.mark.parametrize("N,alpha,beta", [(128, 1.0, 0.0), (256, -0.5, 1.5)])
def test_planned_task_split(max_chunks, N, alpha, beta):
    """Wide windows split into pieces (partial tiles + fixed-order fix-up) against the fp64
    oracle; reproducible; equal within the bf16 bound to the unsplit call."""
    M = 2048
    c, rp, col, val, wp, wc, wv = _skewed_wcsr(M, N)
    K = c["K"]
    P = spx.WcsrPlan(M, wc.size // 64, torch.from_numpy(wp).cuda(), max_chunks=max_chunks)
    assert P.info["split_windows"] > 0
    C0 = synth.uniform(N, synth.T_Y, M * N).reshape(M, N)
    dwp, dwc, dwv, dB = torch.from_numpy(wp).cuda(), torch.from_numpy(wc).cuda(), bits(wv.reshape(-1)), bits(c["B_bf16"])
    Cd = torch.from_numpy(C0.copy()).cuda()
    spx.spx_spmm_wcsr_planned(P, M, K, dwp, dwc, dwv, dB, Cd, alpha, beta)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(val), synth.bf16_bits_to_f32(c["B_bf16"]), alpha, beta,
                             C0)
    assert_within(Cd.cpu().numpy(), ref, bound, rel=BF16_REL, ab=BF16_ABS, what=f"planned wcsr max={max_chunks}")
    C2 = torch.from_numpy(C0.copy()).cuda()
    spx.spx_spmm_wcsr_planned(P, M, K, dwp, dwc, dwv, dB, C2, alpha, beta)
    assert torch.equal(Cd, C2)
    C3 = torch.from_numpy(C0.copy()).cuda()
    spx.spx_spmm_wcsr(M, K, dwp, dwc, dwv, dB, C3, alpha, beta)
    assert_within(C3.cpu().numpy(), ref, bound, rel=BF16_REL, ab=BF16_ABS, what="unsplit wcsr")


def test_planned_errors():
    M, N = 256, 128
    c, rp, col, val, wp, wc, wv = _skewed_wcsr(M, N)
    K, nch = c["K"], wc.size // 64
    dwp, dwc, dwv, dB = torch.from_numpy(wp).cuda(), torch.from_numpy(wc).cuda(), bits(wv.reshape(-1)), bits(c["B_bf16"])
    C = torch.empty(M, N, device="cuda")
    P = spx.WcsrPlan(M, nch, wp, max_chunks=2)
    cases = [(lambda: spx.spx_spmm_wcsr_planned(spx.WcsrPlan(M, nch, wp, max_chunks=2, upload=False), M, K, dwp, dwc,
                                                dwv, dB, C), -10),
             (lambda: spx.spx_spmm_wcsr_planned(P, M, K, dwp, dwc, dwv, dB, C, scratch=torch.zeros(4, device="cuda")), -1),
             (lambda: spx.spx_spmm_wcsr_planned(P, M - 64, K, dwp, dwc, dwv, dB, C[:M - 64]), -1)]
    for f, code in cases:
        with pytest.raises(spx.SpxError) as e:
            f()
        assert e.value.code == code


@pytest.mark.slow
def test_planned_skewed_full_size_sampled():
    """The 16,384^2 skewed window-pool matrix at N = 1024 with the default split, two rows of every window."""
    M, N = 16384, 1024
    c, rp, col, val, wp, wc, wv = _skewed_wcsr(M, N)
    K = c["K"]
    P = spx.WcsrPlan(M, wc.size // 64, wp)
    Cd = torch.empty(M, N, device="cuda")
    spx.spx_spmm_wcsr_planned(P, M, K, torch.from_numpy(wp).cuda(), torch.from_numpy(wc).cuda(), bits(wv.reshape(-1)),
                              bits(c["B_bf16"]), Cd)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    rows = np.sort(np.concatenate([np.arange(0, M, 64), np.arange(37, M, 64)])).astype(np.int32)
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(val), synth.bf16_bits_to_f32(c["B_bf16"]), rows=rows)
    got = Cd[torch.from_numpy(rows).long().cuda()].cpu().numpy()
    assert_within(got, ref, bound, rel=BF16_REL, ab=BF16_ABS, what="planned skewed full size")


def test_planned_without_splits_equals_plain():
    """A plan that splits no window runs the same tiles: equal to spx_spmm_wcsr bit for bit."""
    M, N = 1024, 128
    c = synth.window_pool(6, M=M, N=N)
    rp, col, val = oracle.build_csr(M, c["K"], c["row"], c["col"], c["val_bf16"])
    wp, wc, wv, _ = oracle.build_wcsr(M, c["K"], rp, col, val)
    P = spx.WcsrPlan(M, wc.size // 64, wp, max_chunks=64)
    assert P.info["split_windows"] == 0
    args = (torch.from_numpy(wp).cuda(), torch.from_numpy(wc).cuda(), bits(wv.reshape(-1)), bits(c["B_bf16"]))
    C1, C2 = torch.empty(M, N, device="cuda"), torch.empty(M, N, device="cuda")
    spx.spx_spmm_wcsr(M, c["K"], *args, C1, 1.5, 0.0)
    spx.spx_spmm_wcsr_planned(P, M, c["K"], *args, C2, 1.5, 0.0)
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("M,K,N", [(150, 700, 8), (1, 50, 40), (64 * 3 + 5, 300, 136), (200, 2000, 200),
                                   (129, 4000, 392)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-0.5, 1.5)])
@pytest.mark.parametrize("split", [False, True])
def test_ragged_columns(M, K, N, alpha, beta, split):
    """N any multiple of 8: the last 128-column tile gathers zeros past column N and stores nothing there;
    a partial last window; split: the planned call with windows cut into single chunks."""
    d = synth.random_coo(120 + N, M, K, 1, 150)
    vb = synth.to_bf16_bits(d["val"])
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], vb)
    wp, wc, wv, _ = oracle.build_wcsr(M, K, rp, col, val)
    Bb = synth.to_bf16_bits(synth.uniform(121, synth.T_B, K * N)).reshape(K, N)
    ldb, ldc = N + 8, N + 5
    Bfull = np.zeros((K, ldb), np.uint16)
    Bfull[:, :N] = Bb
    C0 = synth.uniform(122, synth.T_Y, M * ldc).reshape(M, ldc)
    Cd = torch.from_numpy(C0.copy()).cuda()
    dwp, dwc, dwv, dB = torch.from_numpy(wp).cuda(), torch.from_numpy(wc).cuda(), bits(wv.reshape(-1)), bits(Bfull)[:, :N]
    if split:
        P = spx.WcsrPlan(M, wc.size // 64, dwp, max_chunks=1)
        spx.spx_spmm_wcsr_planned(P, M, K, dwp, dwc, dwv, dB, Cd[:, :N], alpha, beta)
    else:
        spx.spx_spmm_wcsr(M, K, dwp, dwc, dwv, dB, Cd[:, :N], alpha, beta)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    got = Cd.cpu().numpy()
    assert np.array_equal(got[:, N:], C0[:, N:])  # columns past N untouched
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(val), synth.bf16_bits_to_f32(Bb), alpha, beta,
                             C0[:, :N])
    assert_within(got[:, :N], ref, bound, rel=BF16_REL, ab=BF16_ABS, what=f"M={M} K={K} N={N} split={split}")
