"""The two-direction pair u = A v - alpha_k u, v = A^T u - beta_k v over
CSR(A) and CSR(A^T) (CSC(A) stored as CSR(A^T)): parity per call (the second
product fed the GPU's u, so errors do not compound) and a short end-to-end
run of several iterations from the same start on both sides."""
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


def test_pair_three_iterations_end_to_end():
    cfg = synth.banded_pair(12, m=40000, n=20000, half=512, iters=3)
    m, n = cfg["M"], cfg["K"]
    (rp, col, val), (trp, tc, tv), A, At, pA, pAt = setup_pair(cfg)
    u, v = dev(cfg["u0"]), dev(cfg["v0"])
    ur, vr = cfg["u0"].astype(np.float64), cfg["v0"].astype(np.float64)
    for k in range(3):
        a, b = float(cfg["alphas"][k]), float(cfg["betas"][k])
        spx.spx_spmv_csr_dual(pA, pAt, A, At, v, u, 1.0, -a, 1.0, -b)
        # reference iteration in fp64 from the same start
        rA, _ = oracle.spmv(m, rp, col, val, vr.astype(np.float32), 1.0, 0.0)
        ur = rA + (-a) * ur
        rAt, _ = oracle.spmv(n, trp, tc, tv, ur.astype(np.float32), 1.0, 0.0)
        vr = rAt + (-b) * vr
    torch.cuda.synchronize()
    # errors compound over iterations; a loose relative check on the whole vectors
    for got, ref in ((u.cpu().numpy(), ur), (v.cpu().numpy(), vr)):
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel < 1e-5, rel
