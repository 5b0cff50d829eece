"""Every stream-ordered product call enqueues kernels only: no allocation, no
host synchronisation, no copy through the host.  So each one can be captured
in a CUDA graph, and a replay from the same starting state gives the direct
call's output bit for bit.  The first direct call also sets up the library's
per-kernel state (shared-memory limits), so the capture sees steady-state
calls only."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import csr_to_device, dev

pytestmark = pytest.mark.gpu


def _graph_matches_direct(run, outs, reset):
    """run(stream) enqueues the call; outs are the tensors it writes; reset() restores the start state."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        reset()
        run(s)
        s.synchronize()
        direct = [o.clone() for o in outs]
        reset()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            run(s)
        reset()
        g.replay()
        s.synchronize()
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    for a, b in zip(direct, outs):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def _skewed(seed, M, K, lmax):
    L, _ = synth.lengths_zipf(seed, M, 2.1, lmax, 12.0)
    row, col = synth.cols_uniform(seed, K, L)
    return oracle.build_csr(M, K, row, col, synth.uniform(seed, synth.T_VAL, row.size))


def _restore(pairs):
    def reset():
        for dst, src in pairs:
            dst.copy_(src)
    return reset


def test_dual_pair():
    cfg = synth.banded_pair(13, m=3000, n=1500, half=100, iters=1)
    m, n = cfg["M"], cfg["K"]
    rp, col, val = oracle.build_csr(m, n, cfg["row"], cfg["col"], cfg["val"])
    A = csr_to_device(m, n, rp, col, val)
    At = csr_to_device(n, m, *oracle.transpose(m, n, rp, col, val))
    pA, pAt = spx.spx_plan_csr(m, n, A.nnz, A.row_ptr), spx.spx_plan_csr(n, m, At.nnz, At.row_ptr)
    u0, v0 = dev(cfg["u0"]), dev(cfg["v0"])
    u, v = u0.clone(), v0.clone()
    _graph_matches_direct(lambda s: spx.spx_spmv_csr_dual(pA, pAt, A, At, v, u, 1.0, -0.7, 1.0, -1.3, stream=s),
                          [u, v], _restore([(u, u0), (v, v0)]))


@pytest.mark.parametrize("fmt", ["sell", "coo"])
def test_sell_and_coo(fmt):
    M, K = 6000, 30000
    rp, col, val = _skewed(65, M, K, 9000)
    x = dev(synth.uniform(65, synth.T_X, K))
    y0 = dev(synth.uniform(65, synth.T_Y, M))
    y = y0.clone()
    if fmt == "sell":
        S = spx.Sell(M, K, dev(rp), dev(col), dev(val))
        run = lambda s: spx.spx_spmv_sell(S, x, y, 1.0, 0.5, stream=s)  # noqa: E731
    else:
        rows, dc, dv = dev(np.repeat(np.arange(M, dtype=np.int32), np.diff(rp))), dev(col), dev(val)
        scratch = torch.empty(max(1, spx.spx_spmv_coo_scratch_bytes(col.size) // 4), device="cuda")
        run = lambda s: spx.spx_spmv_coo(M, K, rows, dc, dv, x, y, 1.0, 0.5, stream=s, scratch=scratch)  # noqa: E731
    _graph_matches_direct(run, [y], _restore([(y, y0)]))


@pytest.mark.parametrize("kind", ["f32", "bf16", "f16"])
def test_planned_spmm(kind):
    M, K, N = 3000, 20000, 64
    rp, col, val = _skewed(66, M, K, 9000)
    Bf = synth.uniform(66, synth.T_B, K * N).reshape(K, N)
    if kind == "f32":
        A, B, fn = csr_to_device(M, K, rp, col, val), dev(Bf), spx.spx_spmm_csr_planned
    elif kind == "bf16":
        A = spx.Csr(M, K, dev(rp), dev(col), dev(synth.to_bf16_bits(val).view(np.int16)))
        B, fn = dev(synth.to_bf16_bits(Bf).reshape(K, N).view(np.int16)), spx.spx_spmm_csr_bf16_planned
    else:
        A = spx.Csr(M, K, dev(rp), dev(col), dev(val.astype(np.float16).view(np.int16)))
        B, fn = dev(Bf.astype(np.float16).view(np.int16)), spx.spx_spmm_csr_f16_planned
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, {"pack_max": 64, "cta_max": 1000, "seg_nnz": 500})
    assert plan.info["cta_rows"] > 0 and plan.info["split_rows"] > 0
    need = int(spx._lib().spx_spmm_csr_planned_scratch_bytes(plan.handle, N))
    scratch = torch.empty(max(1, (need + 3) // 4), device="cuda")
    C0 = dev(synth.uniform(67, synth.T_Y, M * N).reshape(M, N))
    C = C0.clone()
    _graph_matches_direct(lambda s: fn(plan, A, B, C, -0.5, 1.5, stream=s, scratch=scratch), [C],
                          _restore([(C, C0)]))


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.parametrize("how", ["plain", "planned"])
def test_bsr(how):
    M, N = 2048, 256
    c = synth.block_sparse_skewed(9, M=M, N=N)
    K = c["K"]
    rp, col, val = oracle.build_csr(M, K, c["row"], c["col"], c["val_bf16"])
    brp, bcol, bval, _ = oracle.build_bsr(M, K, rp, col, val, 64, 64)
    dbrp, dbcol, dbval, dB = dev(brp), dev(bcol), _bits(bval.reshape(-1)), _bits(c["B_bf16"])
    C0 = dev(synth.uniform(68, synth.T_Y, M * N).reshape(M, N))
    C = C0.clone()
    if how == "plain":
        run = lambda s: spx.spx_spmm_bsr(M, K, 64, 64, dbrp, dbcol, dbval, dB, C, stream=s,  # noqa: E731
                                         alpha=2.0, beta=-1.0)
    else:
        P = spx.BsrPlan(M, bcol.size, dbrp, max_chunks=8)
        assert P.info["split_windows"] > 0
        need = int(spx._lib().spx_spmm_bsr_planned_scratch_bytes(P.handle, N))
        scratch = torch.empty(max(4, (need + 15) // 16 * 4), device="cuda")
        run = lambda s: spx.spx_spmm_bsr_planned(P, M, K, 64, 64, dbrp, dbcol, dbval, dB, C, 2.0, -1.0,  # noqa: E731
                                                 stream=s, scratch=scratch)
    _graph_matches_direct(run, [C], _restore([(C, C0)]))


@pytest.mark.parametrize("how", ["plain", "planned"])
def test_wcsr(how):
    M, N = 2048, 256
    c = synth.window_pool_skewed(7, M=M, N=N)
    K = c["K"]
    rp, col, val = oracle.build_csr(M, K, c["row"], c["col"], c["val_bf16"])
    wp, wc, wv, _ = oracle.build_wcsr(M, K, rp, col, val)
    dwp, dwc, dwv, dB = dev(wp), dev(wc), _bits(wv.reshape(-1)), _bits(c["B_bf16"])
    C0 = dev(synth.uniform(69, synth.T_Y, M * N).reshape(M, N))
    C = C0.clone()
    if how == "plain":
        run = lambda s: spx.spx_spmm_wcsr(M, K, dwp, dwc, dwv, dB, C, 2.0, -1.0, stream=s)  # noqa: E731
    else:
        P = spx.WcsrPlan(M, wc.size // 64, dwp, max_chunks=4)
        assert P.info["split_windows"] > 0
        need = int(spx._lib().spx_spmm_wcsr_planned_scratch_bytes(P.handle, N))
        scratch = torch.empty(max(4, (need + 15) // 16 * 4), device="cuda")
        run = lambda s: spx.spx_spmm_wcsr_planned(P, M, K, dwp, dwc, dwv, dB, C, 2.0, -1.0,  # noqa: E731
                                                  stream=s, scratch=scratch)
    _graph_matches_direct(run, [C], _restore([(C, C0)]))
