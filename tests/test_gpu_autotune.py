"""spx_plan_autotune: times the candidate plan options on the device, returns
the fastest, caches the answer per matrix profile; the chosen plan computes
the same product (parity against the oracle)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import assert_within, csr_to_device, dev

pytestmark = pytest.mark.gpu


def matrix(seed=41, M=200_000):
    L, _ = synth.lengths_zipf(seed, M, 2.1, 20000, 16.0)
    row, col = synth.cols_uniform(seed, M, L)
    val = synth.uniform(seed, synth.T_VAL, row.size)
    rp, col, val = oracle.build_csr(M, M, row, col, val)
    return M, rp, col, val


def test_builtin_candidates_cached_and_correct():
    spx.spx_plan_autotune_forget()
    M, rp, col, val = matrix()
    A = csr_to_device(M, M, rp, col, val)
    x = synth.uniform(41, synth.T_X, M)
    xd = dev(x)
    best, times, cached = spx.spx_plan_autotune(A, rp, xd, reps=3)
    assert not cached and len(times) == 4 and all(t > 0 for t in times)
    d = spx.spx_plan_opts_default()
    cands = [dict(d), dict(d, lanes_div=4), dict(d, block_nnz=1024, lanes_div=0), dict(d, lanes_div=0)]
    assert best == cands[int(np.argmin(times))]
    again, times2, cached2 = spx.spx_plan_autotune(A, rp, xd, reps=3)
    assert cached2 and again == best and all(t == -1 for t in times2)
    plan = spx.spx_plan_csr(M, M, A.nnz, rp, opts=best, device=xd.device)
    y0 = synth.uniform(41, synth.T_Y, M)
    y = dev(y0)
    spx.spx_spmv_csr(plan, A, xd, y, 1.0, 0.5)
    torch.cuda.synchronize()
    ref, bound = oracle.spmv(M, rp, col, val, x, 1.0, 0.5, y0)
    assert_within(y.cpu().numpy(), ref, bound)


def test_explicit_candidates_and_forget():
    spx.spx_plan_autotune_forget()
    M, rp, col, val = matrix(42, 50_000)
    A = csr_to_device(M, M, rp, col, val)
    xd = dev(synth.uniform(42, synth.T_X, M))
    cands = [dict(block_nnz=2048, lanes_div=1), dict(block_nnz=4096, lanes_div=0)]
    best, times, cached = spx.spx_plan_autotune(A, rp, xd, candidates=cands, reps=2)
    assert not cached and len(times) == 2
    assert best["block_nnz"] == cands[int(np.argmin(times))]["block_nnz"]
    # a different candidate list is a different question: not answered from the cache
    _, _, cached_b = spx.spx_plan_autotune(A, rp, xd, reps=2)
    assert not cached_b
    _, _, cached_c = spx.spx_plan_autotune(A, rp, xd, candidates=cands, reps=2)
    assert cached_c
    spx.spx_plan_autotune_forget()
    _, _, cached_d = spx.spx_plan_autotune(A, rp, xd, candidates=cands, reps=2)
    assert not cached_d
