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


def first_rows_expected(rp, tasks, block_nnz):
    """The plan's per-thread first-row entries of its groups, derived here with a
    sorted search of each group's row offsets: thread t of a group sums the
    products [t*Q, t*Q + Q) (T threads: block_nnz / 8 for 512..4096, else 256;
    Q = ceil(block_nnz / T)); its entry is 2*r + s with r the group's row holding
    product t*Q (the last row starting at or before it) and s = 1 when that row
    starts before t*Q; 0 past the group's products."""
    T = block_nnz // 8 if block_nnz in (512, 1024, 2048, 4096) else 256
    Q = -(-block_nnz // T)
    rp = np.asarray(rp, np.int64)
    groups = tasks[(tasks[:, 0] & 255) == 0]
    out = np.zeros((groups.shape[0], T), np.uint16)
    a = np.arange(T, dtype=np.int64) * Q
    for g, (_, r0, r1, _) in enumerate(groups):
        s = rp[r0:r1 + 1] - rp[r0]
        ok = a < s[-1]
        r = np.searchsorted(s, a, side="right") - 1
        r = np.clip(r, 0, max(len(s) - 2, 0))
        out[g] = np.where(ok, 2 * r + (s[r] < a), 0)
    return out
