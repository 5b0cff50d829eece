"""Shared helpers for the GPU parity tests (device upload, tolerance checks)."""
import numpy as np
import torch

from csr_bsr_spmv_gb300 import spx

# fp32 results: |y - ref| <= 1e-5 * sum_j |a_ij x_j| (+ |beta y_i|) + 1e-6 per output
FP32_REL, FP32_ABS = 1e-5, 1e-6
# bf16-input BSR with fp32 accumulation: |c - ref| <= 2e-2 * sum_k |a_ik b_kj| + 1e-3
BF16_REL, BF16_ABS = 2e-2, 1e-3


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def csr_to_device(M, K, rp, col, val) -> spx.Csr:
    return spx.Csr(M, K, dev(rp), dev(col), dev(val))


def assert_within(got, ref, bound, rel=FP32_REL, ab=FP32_ABS, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    tol = rel * bound + ab
    bad = ~(err <= tol)  # NaN counts as bad
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {i.tolist()}: "
                             f"got {got.ravel()[i].tolist()} ref {ref.ravel()[i].tolist()} "
                             f"tol {tol.ravel()[i].tolist()}")
    return float((err / np.maximum(tol, 1e-300)).max()) if err.size else 0.0
