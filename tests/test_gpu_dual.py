"""The two-direction pair u = A v - alpha_k u, v = A^T u - beta_k v over
CSR(A) and CSR(A^T) (CSC(A) stored as CSR(A^T)): parity per call (the second
product fed the GPU's u, so errors do not compound) and a short end-to-end
run of several iterations from the same start on both sides, checked element by
element against an error bound carried through the iterations."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import assert_within, csr_to_device, dev

pytestmark = pytest.mark.gpu


def setup_pair(cfg, device_transpose=False):
    m, n = cfg["M"], cfg["K"]
    rp, col, val = spx.spx_build_csr(m, n, cfg["row"], cfg["col"], cfg["val"])
    A = csr_to_device(m, n, rp, col, val)
    if device_transpose:
        trp, tc, tv = spx.spx_transpose_csr(m, n, A.row_ptr, A.col, A.val)
        At = spx.Csr(n, m, trp, tc, tv)
        t_host = (trp.cpu().numpy(), tc.cpu().numpy(), tv.cpu().numpy())
    else:
        t_host = spx.spx_transpose_csr(m, n, rp, col, val)
        At = csr_to_device(n, m, *t_host)
    pA = spx.spx_plan_csr(m, n, A.nnz, A.row_ptr)
    pAt = spx.spx_plan_csr(n, m, A.nnz, At.row_ptr)
    return (rp, col, val), t_host, A, At, pA, pAt


def test_pair_small_dense_reference():
    """Same small matrix from CSR and from CSC: both directions equal the dense
    products (the dual-path test of the LSMR operator page, §8)."""
    cfg = synth.banded_pair(11, m=3000, n=1500, half=100, iters=3)
    (rp, col, val), (trp, tc, tv), A, At, pA, pAt = setup_pair(cfg, device_transpose=True)
    dense = np.zeros((3000, 1500))
    dense[np.repeat(np.arange(3000), np.diff(rp)), col] = val
    u, v = dev(cfg["u0"]), dev(cfg["v0"])
    spx.spx_spmv_csr_dual(pA, pAt, A, At, v, u, 1.0, 0.0, 1.0, 0.0)
    torch.cuda.synchronize()
    u1 = dense @ cfg["v0"].astype(np.float64)
    assert_within(u.cpu().numpy(), u1, np.abs(dense) @ np.abs(cfg["v0"].astype(np.float64)))
    uu = u.cpu().numpy().astype(np.float64)
    assert_within(v.cpu().numpy(), dense.T @ uu, np.abs(dense.T) @ np.abs(uu))
    # the device transpose equals the host one bit for bit
    ht = oracle.transpose(3000, 1500, rp, col, val)
    for a, b in zip(ht, (trp, tc, tv)):
        assert np.array_equal(a, b)


@pytest.mark.slow
def test_pair_full_size_per_call():
    """2,000,000 x 1,000,000 banded operator, nnz ~ 20M: one iteration, each
    product checked on 20k sampled rows."""
    cfg = synth.banded_pair()
    m, n = cfg["M"], cfg["K"]
    (rp, col, val), (trp, tc, tv), A, At, pA, pAt = setup_pair(cfg)
    a, b = float(cfg["alphas"][0]), float(cfg["betas"][0])
    u, v = dev(cfg["u0"]), dev(cfg["v0"])
    rng = np.random.default_rng(1)
    ru = np.unique(rng.integers(0, m, 20000)).astype(np.int32)
    rv = np.unique(rng.integers(0, n, 20000)).astype(np.int32)
    spx.spx_spmv_csr_dual(pA, pAt, A, At, v, u, 1.0, -a, 1.0, -b)
    torch.cuda.synchronize()
    u1 = u.cpu().numpy()
    ref, bound = oracle.spmv(m, rp, col, val, cfg["v0"], 1.0, -a, cfg["u0"], rows=ru)
    assert_within(u1[ru], ref, bound, what="u = Av - alpha u")
    ref, bound = oracle.spmv(n, trp, tc, tv, u1, 1.0, -b, cfg["v0"], rows=rv)
    assert_within(v.cpu().numpy()[rv], ref, bound, what="v = A^T u - beta v")


def _gamma(k, u=2.0 ** -24):
    return k * u / (1 - k * u)


def test_pair_three_iterations_end_to_end():
    """Three iterations from the same start on both sides, checked element by element against
    an error bound carried through the iterations.  Both sides are compared with the exact
    iteration: the GPU's error in u_k is at most |A| E_v + a E_u (its inputs' errors) plus
    gamma_(l+3) (|A||v| + a|u|) (its own fp32 rounding, l = the longest row); the reference
    rounds its inputs to fp32 before each fp64 product, which adds |A| 2^-24 |v|; v_k likewise
    with A^T.  |got - ref| must stay within the sum of the two."""
    cfg = synth.banded_pair(12, m=40000, n=20000, half=512, iters=3)
    m, n = cfg["M"], cfg["K"]
    (rp, col, val), (trp, tc, tv), A, At, pA, pAt = setup_pair(cfg)
    u, v = dev(cfg["u0"]), dev(cfg["v0"])
    ur, vr = cfg["u0"].astype(np.float64), cfg["v0"].astype(np.float64)
    aval, atval = np.abs(val), np.abs(tv)
    g_u = _gamma(int(np.diff(rp).max()) + 3)
    g_v = _gamma(int(np.diff(trp).max()) + 3)
    eps = 2.0 ** -24
    E_u, E_v = np.zeros(m), np.zeros(n)  # GPU error bounds
    R_u, R_v = np.zeros(m), np.zeros(n)  # reference error bounds

    def abs_prod(M_, rp_, col_, aval_, w):
        # |A| w for w >= 0 (fp64 sums of fp32 inputs; w rounded up to fp32 so the product bounds |A| w)
        w32 = np.nextafter(w.astype(np.float32), np.float32(np.inf)).astype(np.float32)
        return oracle.spmv(M_, rp_, col_, aval_, w32, 1.0, 0.0)[0]

    for k in range(3):
        a, b = float(cfg["alphas"][k]), float(cfg["betas"][k])
        spx.spx_spmv_csr_dual(pA, pAt, A, At, v, u, 1.0, -a, 1.0, -b)
        # u_k = A v_(k-1) - a u_(k-1): the reference's product in fp64 of its fp32-rounded v
        rA, _ = oracle.spmv(m, rp, col, val, vr.astype(np.float32), 1.0, 0.0)
        mag_v = abs_prod(m, rp, col, aval, np.abs(vr) + E_v + R_v)  # bounds |A||v| for either side's v
        E_u_new = abs_prod(m, rp, col, aval, E_v) + a * E_u + g_u * (mag_v + a * (np.abs(ur) + E_u + R_u))
        R_u = abs_prod(m, rp, col, aval, R_v) + a * R_u + eps * mag_v
        ur = rA + (-a) * ur
        E_u = E_u_new
        # v_k = A^T u_k - b v_(k-1)
        rAt, _ = oracle.spmv(n, trp, tc, tv, ur.astype(np.float32), 1.0, 0.0)
        mag_u = abs_prod(n, trp, tc, atval, np.abs(ur) + E_u + R_u)
        E_v_new = abs_prod(n, trp, tc, atval, E_u) + b * E_v + g_v * (mag_u + b * (np.abs(vr) + E_v + R_v))
        R_v = abs_prod(n, trp, tc, atval, R_u) + b * R_v + eps * mag_u
        vr = rAt + (-b) * vr
        E_v = E_v_new
    torch.cuda.synchronize()
    for name, got, ref, E, R in (("u", u.cpu().numpy(), ur, E_u, R_u), ("v", v.cpu().numpy(), vr, E_v, R_v)):
        err = np.abs(got.astype(np.float64) - ref)
        bad = ~(err <= (E + R) * (1 + 1e-6))
        assert not bad.any(), (name, int(bad.sum()), float((err / np.maximum(E + R, 1e-300)).max()))
        # the bound is not vacuous: the largest error uses a visible share of it somewhere
        assert float((err / np.maximum(E + R, 1e-300)).max()) > 1e-4
