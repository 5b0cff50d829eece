"""The allocation-free SpMV entry point (spx_spmv_csr_noalloc).

For callers that cannot allocate device memory and so cannot hand over the
scratch buffer spx_spmv_csr needs: split-row partial sums go to the library's
fixed device array instead.  Checked through the C ABI against the existing
entry point, on two calls in a row (the array keeps the first call's contents
when the second starts).  This file is collected last on purpose.
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


def _matrix(seed, M):
    L, _ = synth.lengths_zipf(seed, M, 2.1, 40000, 14.0)
    L[:3] = (30000, 9000, 20000)  # split rows (segments -> partial sums) and a CTA row
    row, col = synth.cols_uniform(seed, 50000, L)
    val = synth.uniform(seed, synth.T_VAL, row.size)
    rp, col, val = oracle.build_csr(M, 50000, row, col, val)
    return csr_to_device(M, 50000, rp, col, val), (rp, col, val)


def test_noalloc_matches_scratch_entry_on_two_calls():
    lib = spx._lib()
    A1, _ = _matrix(31, 6000)
    A2, host2 = _matrix(32, 4000)
    p1 = spx.spx_plan_csr(A1.M, A1.K, A1.nnz, A1.row_ptr)
    p2 = spx.spx_plan_csr(A2.M, A2.K, A2.nnz, A2.row_ptr, opts=dict(seg_nnz=1024, cta_max=2048))
    assert p1.info["slots"] > 0 and p2.info["slots"] > p1.info["slots"]
    assert p2.info["slots"] <= 65536
    calls = [(p1, A1, 1.0, 0.5, 41), (p2, A2, -2.0, 0.25, 42)]
    for plan, A, alpha, beta, seed in calls:  # two calls in a row on the shared array
        x = dev(synth.uniform(seed, synth.T_X, A.K))
        y0 = synth.uniform(seed, synth.T_Y, A.M)
        y_ref, y_new = dev(y0), dev(y0)
        spx.spx_spmv_csr(plan, A, x, y_ref, alpha, beta)
        rc = lib.spx_spmv_csr_noalloc(plan.handle, A.M, A.K, A.nnz, spx._ptr(A.row_ptr), spx._ptr(A.col),
                                      spx._ptr(A.val), ctypes.c_float(alpha), spx._ptr(x), ctypes.c_float(beta),
                                      spx._ptr(y_new), spx._stream())
        assert rc == 0, spx.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        got, want = y_new.cpu().numpy(), y_ref.cpu().numpy()
        # same tolerance as the oracle checks, with the scratch entry's result as the reference
        scale = np.abs(want).astype(np.float64) + np.abs(beta * y0)
        assert_within(got, want.astype(np.float64), scale, what="noalloc vs scratch entry")
    # and the second call is right in absolute terms too
    rp, col, val = host2
    ref, bound = oracle.spmv(A2.M, rp, col, val, synth.uniform(42, synth.T_X, A2.K), -2.0, 0.25,
                             synth.uniform(42, synth.T_Y, A2.M))
    assert_within(got, ref, bound, what="noalloc vs oracle")


def test_noalloc_rejects_plans_beyond_the_fixed_buffer():
    lib = spx._lib()
    rp = np.array([0, 70000], np.int32)
    col = np.arange(70000, dtype=np.int32)
    A = csr_to_device(1, 70000, rp, col, np.ones(70000, np.float32))
    plan = spx.spx_plan_csr(1, 70000, 70000, A.row_ptr,
                            opts=dict(block_nnz=8, block_rows=8, pack_max=8, cta_max=8, seg_nnz=1))
    assert plan.info["slots"] == 70000 > 65536
    y = torch.zeros(1, device="cuda")
    before = spx.launch_count()
    rc = lib.spx_spmv_csr_noalloc(plan.handle, 1, 70000, 70000, spx._ptr(A.row_ptr), spx._ptr(A.col),
                                  spx._ptr(A.val), ctypes.c_float(1.0), spx._ptr(torch.ones(70000, device="cuda")),
                                  ctypes.c_float(0.0), spx._ptr(y), spx._stream())
    assert spx.STATUS[rc] == "SPX_ERR_SCRATCH_LIMIT"
    assert spx.launch_count() == before
