"""Several host threads calling the library at once, each on its own stream
with its own outputs and scratch, sharing the matrices, the SpMV plan, the
SELL form and the BSR / WCSR task splits (read-only once uploaded): every
result equals the single-threaded result bit for bit, and the calls raise
nothing.  The ctypes calls release the interpreter lock, so the host-side
work of the calls (argument checks, tensor-map encoding, the per-kernel
set-up caches) really runs concurrently."""
import threading

import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import csr_to_device, dev

pytestmark = pytest.mark.gpu


def _skewed(seed, M, K, lmax):
    L, _ = synth.lengths_zipf(seed, M, 2.1, lmax, 12.0)
    row, col = synth.cols_uniform(seed, K, L)
    return oracle.build_csr(M, K, row, col, synth.uniform(seed, synth.T_VAL, row.size))


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _problems():
    """kind -> (run(out, scratch, stream), start value of out, scratch floats)."""
    P = {}
    M, K = 6000, 30000
    rp, col, val = _skewed(71, M, K, 9000)
    A = csr_to_device(M, K, rp, col, val)
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, {"pack_max": 64, "cta_max": 1000, "seg_nnz": 500})
    assert plan.info["split_rows"] > 0
    x, y0 = dev(synth.uniform(71, synth.T_X, K)), dev(synth.uniform(71, synth.T_Y, M))
    P["spmv"] = (lambda o, sc, s: spx.spx_spmv_csr(plan, A, x, o, 1.0, 0.5, stream=s, scratch=sc), y0,
                 plan.scratch.numel())
    S = spx.Sell(M, K, A.row_ptr, A.col, A.val)
    P["sell"] = (lambda o, sc, s: spx.spx_spmv_sell(S, x, o, 1.0, 0.5, stream=s, scratch=sc), y0, S.scratch.numel())
    rows = dev(np.repeat(np.arange(M, dtype=np.int32), np.diff(rp)))
    P["coo"] = (lambda o, sc, s: spx.spx_spmv_coo(M, K, rows, A.col, A.val, x, o, 1.0, 0.5, stream=s, scratch=sc), y0,
                max(1, spx.spx_spmv_coo_scratch_bytes(A.nnz) // 4))
    N = 64
    B, C0 = dev(synth.uniform(72, synth.T_B, K * N).reshape(K, N)), dev(synth.uniform(72, synth.T_Y, M * N).reshape(M, N))
    need = int(spx._lib().spx_spmm_csr_planned_scratch_bytes(plan.handle, N))
    P["spmm"] = (lambda o, sc, s: spx.spx_spmm_csr_planned(plan, A, B, o, -0.5, 1.5, stream=s, scratch=sc), C0,
                 max(1, (need + 3) // 4))

    Mb, Nb = 2048, 256
    c = synth.block_sparse_skewed(9, M=Mb, N=Nb)
    r2, c2, v2 = oracle.build_csr(Mb, c["K"], c["row"], c["col"], c["val_bf16"])
    brp, bcol, bval, _ = oracle.build_bsr(Mb, c["K"], r2, c2, v2, 64, 64)
    dbrp, dbcol, dbval, dBb = dev(brp), dev(bcol), _bits(bval.reshape(-1)), _bits(c["B_bf16"])
    BP = spx.BsrPlan(Mb, bcol.size, dbrp, max_chunks=8)
    assert BP.info["split_windows"] > 0
    Kb = c["K"]
    Cb0 = dev(synth.uniform(73, synth.T_Y, Mb * Nb).reshape(Mb, Nb))
    need = int(spx._lib().spx_spmm_bsr_planned_scratch_bytes(BP.handle, Nb))
    P["bsr"] = (lambda o, sc, s: spx.spx_spmm_bsr_planned(BP, Mb, Kb, 64, 64, dbrp, dbcol, dbval, dBb, o, 2.0, -1.0,
                                                         stream=s, scratch=sc), Cb0, max(4, (need + 15) // 16 * 4))

    w = synth.window_pool_skewed(7, M=Mb, N=Nb)
    r3, c3, v3 = oracle.build_csr(Mb, w["K"], w["row"], w["col"], w["val_bf16"])
    wp, wc, wv, _ = oracle.build_wcsr(Mb, w["K"], r3, c3, v3)
    dwp, dwc, dwv, dBw = dev(wp), dev(wc), _bits(wv.reshape(-1)), _bits(w["B_bf16"])
    WP = spx.WcsrPlan(Mb, wc.size // 64, dwp, max_chunks=4)
    assert WP.info["split_windows"] > 0
    Kw = w["K"]
    need = int(spx._lib().spx_spmm_wcsr_planned_scratch_bytes(WP.handle, Nb))
    P["wcsr"] = (lambda o, sc, s: spx.spx_spmm_wcsr_planned(WP, Mb, Kw, dwp, dwc, dwv, dBw, o, 2.0, -1.0, stream=s,
                                                          scratch=sc), Cb0, max(4, (need + 15) // 16 * 4))
    P["_keep"] = (plan, S, BP, WP)  # the shared objects live as long as the problems
    return P


def test_threads_share_plans_and_matrices():
    P = _problems()
    kinds = [k for k in P if not k.startswith("_")]
    ref = {}
    for k in kinds:
        run, out0, nsc = P[k]
        out, sc = out0.clone(), torch.empty(nsc, device="cuda")
        run(out, sc, None)
        torch.cuda.synchronize()
        ref[k] = out
    assert spx.spx_last_device_error() == 0
    nthreads, reps = 4, 3
    errors = []
    start = threading.Barrier(nthreads)

    def worker(t):
        try:
            s = torch.cuda.Stream()
            order = kinds[t % len(kinds):] + kinds[:t % len(kinds)]
            with torch.cuda.stream(s):
                bufs = {k: (torch.empty_like(P[k][1]), torch.empty(P[k][2], device="cuda")) for k in order}
                start.wait()
                for rep in range(reps):
                    for k in order:
                        out, sc = bufs[k]
                        out.copy_(P[k][1])
                        P[k][0](out, sc, s)
                    s.synchronize()
                    for k in order:
                        if not torch.equal(bufs[k][0].view(torch.int32), ref[k].view(torch.int32)):
                            errors.append((t, rep, k))
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(nthreads)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads)
    torch.cuda.synchronize()
    assert not errors, errors[:8]
    assert spx.spx_last_device_error() == 0
