"""The allocation-free SpMV entry point (spx_spmv_csr_noalloc).

For callers that cannot allocate device memory and so cannot hand over the
scratch buffer spx_spmv_csr needs: split-row partial sums go to the library's
fixed device array instead.  Checked through the C ABI against the existing
entry point -- bit for bit, since both run the same kernels in the same order
-- on two calls in a row (the array keeps the first call's contents when the
second starts), and against the oracle.  The limit is checked at its edge: a
plan of exactly SPX_NOALLOC_MAX_SLOTS partial sums runs, one more is refused
with nothing launched.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import assert_within, csr_to_device, dev

pytestmark = pytest.mark.gpu

MAX_SLOTS = 65536  # SPX_NOALLOC_MAX_SLOTS in include/spx.h


def _matrix(seed, M):
    L, _ = synth.lengths_zipf(seed, M, 2.1, 40000, 14.0)
    L[:3] = (30000, 9000, 20000)  # split rows (segments -> partial sums) and a CTA row
    row, col = synth.cols_uniform(seed, 50000, L)
    val = synth.uniform(seed, synth.T_VAL, row.size)
    rp, col, val = oracle.build_csr(M, 50000, row, col, val)
    return csr_to_device(M, 50000, rp, col, val), (rp, col, val)


def _noalloc(plan, A, x, y, alpha, beta):
    return spx._lib().spx_spmv_csr_noalloc(plan.handle, A.M, A.K, A.nnz, spx._ptr(A.row_ptr), spx._ptr(A.col),
                                           spx._ptr(A.val), ctypes.c_float(alpha), spx._ptr(x),
                                           ctypes.c_float(beta), spx._ptr(y), spx._stream())


def test_noalloc_matches_scratch_entry_on_two_calls():
    A1, host1 = _matrix(31, 6000)
    A2, host2 = _matrix(32, 4000)
    p1 = spx.spx_plan_csr(A1.M, A1.K, A1.nnz, A1.row_ptr)
    p2 = spx.spx_plan_csr(A2.M, A2.K, A2.nnz, A2.row_ptr, opts=dict(seg_nnz=1024, cta_max=2048))
    assert p1.info["slots"] > 0 and p2.info["slots"] > p1.info["slots"]
    assert p2.info["slots"] <= MAX_SLOTS
    calls = [(p1, A1, host1, 1.0, 0.5, 41), (p2, A2, host2, -2.0, 0.25, 42)]
    for plan, A, (rp, col, val), alpha, beta, seed in calls:  # two calls in a row on the shared array
        xh = synth.uniform(seed, synth.T_X, A.K)
        y0 = synth.uniform(seed, synth.T_Y, A.M)
        x, y_ref, y_new = dev(xh), dev(y0), dev(y0)
        spx.spx_spmv_csr(plan, A, x, y_ref, alpha, beta)
        rc = _noalloc(plan, A, x, y_new, alpha, beta)
        assert rc == 0, spx.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        got, want = y_new.cpu().numpy(), y_ref.cpu().numpy()
        # the same kernels, the same summation order: the scratch entry's result, bit for bit
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        # and right in absolute terms
        ref, bound = oracle.spmv(A.M, rp, col, val, xh, alpha, beta, y0)
        assert_within(got, ref, bound, what="noalloc vs oracle")


def _one_long_row(nslots):
    """One row of nslots ones cut into one-entry segments: exactly nslots partial sums."""
    rp = np.array([0, nslots], np.int32)
    col = np.arange(nslots, dtype=np.int32)
    A = csr_to_device(1, nslots, rp, col, np.ones(nslots, np.float32))
    plan = spx.spx_plan_csr(1, nslots, nslots, A.row_ptr,
                            opts=dict(block_nnz=8, block_rows=8, pack_max=8, cta_max=8, seg_nnz=1))
    assert plan.info["slots"] == nslots
    return A, plan


def test_noalloc_accepts_exactly_the_limit():
    A, plan = _one_long_row(MAX_SLOTS)
    x = torch.ones(MAX_SLOTS, device="cuda")
    y_ref, y_new = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
    spx.spx_spmv_csr(plan, A, x, y_ref, 1.0, 0.0)
    assert _noalloc(plan, A, x, y_new, 1.0, 0.0) == 0
    torch.cuda.synchronize()
    assert y_new.item() == float(MAX_SLOTS) == y_ref.item()  # integers below 2^24: exact in fp32


@pytest.mark.parametrize("nslots", [MAX_SLOTS + 1, 70000])
def test_noalloc_rejects_plans_beyond_the_fixed_buffer(nslots):
    A, plan = _one_long_row(nslots)
    y = torch.zeros(1, device="cuda")
    before = spx.launch_count()
    rc = _noalloc(plan, A, torch.ones(nslots, device="cuda"), y, 1.0, 0.0)
    assert spx.STATUS[rc] == "SPX_ERR_SCRATCH_LIMIT"
    assert spx.launch_count() == before
