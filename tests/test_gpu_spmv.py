"""CSR SpMV parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small matrices exercise every task kind (thread/lane groups, CTA rows, split
rows and the fix-up), empty rows and ragged tails; the full-size workloads are
checked on sampled rows plus every CTA/split row, in the same launch
configuration the benchmark times."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import FP32_ABS, FP32_REL, assert_within, csr_to_device, dev

pytestmark = pytest.mark.gpu

SMALL_OPTS = [
    None,
    dict(block_nnz=16, block_rows=3, pack_max=8, cta_max=100, seg_nnz=40, lanes_div=2),
    dict(block_nnz=1024, block_rows=128, pack_max=64, cta_max=300, seg_nnz=256, lanes_div=1),
    dict(block_nnz=4096, block_rows=1024, pack_max=4096, cta_max=4096, seg_nnz=1000, lanes_div=8),
    dict(block_nnz=2000, block_rows=77, pack_max=33, cta_max=2000, seg_nnz=777, lanes_div=3),
    dict(block_nnz=2048, block_rows=256, pack_max=512, cta_max=8192, seg_nnz=4096, lanes_div=4),
    dict(block_nnz=1024, block_rows=1024, pack_max=1024, cta_max=1024, seg_nnz=512, lanes_div=0),
    dict(block_nnz=4096, block_rows=300, pack_max=2000, cta_max=9000, seg_nnz=3000, lanes_div=0),
    dict(block_nnz=1000, block_rows=50, pack_max=999, cta_max=3000, seg_nnz=1000, lanes_div=0),
    dict(block_nnz=8, block_rows=3, pack_max=8, cta_max=100, seg_nnz=40, lanes_div=0),
    dict(block_nnz=512, block_rows=256, pack_max=512, cta_max=8192, seg_nnz=4096, lanes_div=0),
    dict(block_nnz=512, block_rows=64, pack_max=200, cta_max=1000, seg_nnz=600, lanes_div=16),
]


def run_spmv(M, K, rp, col, val, x, y0, alpha, beta, opts=None):
    A = csr_to_device(M, K, rp, col, val)
    plan = spx.spx_plan_csr(M, K, int(rp[-1]), A.row_ptr, opts=opts)
    xd, yd = dev(x), dev(y0)
    spx.spx_spmv_csr(plan, A, xd, yd, alpha, beta)
    torch.cuda.synchronize()
    return yd.cpu().numpy(), plan


def check(M, K, rp, col, val, x, y0, alpha, beta, opts=None, what=""):
    got, plan = run_spmv(M, K, rp, col, val, x, y0, alpha, beta, opts)
    ref, bound = oracle.spmv(M, rp, col, val, x, alpha, beta, y0)
    assert_within(got, ref, bound, what=what)
    return got, plan


@pytest.mark.parametrize("opts", SMALL_OPTS)
@pytest.mark.parametrize("seed", [1, 2])
def test_power_law_small(opts, seed):
    M = 3000
    L, _ = synth.lengths_zipf(seed, M, 2.1, 20000, 10.0)
    L[::13] = 0
    row, col = synth.cols_uniform(seed, M * 8, L)
    val = synth.uniform(seed, synth.T_VAL, row.size)
    rp, col, val = oracle.build_csr(M, M * 8, row, col, val)
    x = synth.uniform(seed, synth.T_X, M * 8)
    y0 = synth.uniform(seed, synth.T_Y, M)
    _, plan = check(M, M * 8, rp, col, val, x, y0, 1.0, 0.5, opts, what=f"opts={opts}")
    assert plan.info["tasks"] > 0


@pytest.mark.parametrize("B", [512, 1000, 4096])
def test_segmented_groups_with_runs_of_empty_rows(B):
    """Groups of up to 1024 rows, most of them empty (so a thread's first row, taken from the
    plan, lies hundreds of rows into its group), some rows starting exactly at a thread's first
    product: the oracle's result, and the same bits from a plan built on the host and one built
    on the GPU."""
    rng = np.random.default_rng(B)
    M, K = 40_000, 30_000
    L = np.where(rng.random(M) < 0.05, rng.integers(1, 40, M), 0).astype(np.int32)
    L[:900] = 0
    L[1000:1064] = 8  # runs of rows that each start on an eight-product boundary
    row, col = synth.cols_uniform(B, K, L)
    val = synth.uniform(B, synth.T_VAL, row.size)
    rp, col, val = oracle.build_csr(M, K, row, col, val)
    x = synth.uniform(B, synth.T_X, K)
    y0 = synth.uniform(B, synth.T_Y, M)
    opts = dict(block_nnz=B, block_rows=1024, pack_max=64, cta_max=4096, seg_nnz=1024, lanes_div=0)
    got, plan = check(M, K, rp, col, val, x, y0, 1.0, 0.5, opts, what=f"B={B}")
    assert plan.info["segmented_groups"] > 0 and plan.first_rows().max() > 1000
    A = csr_to_device(M, K, rp, col, val)
    ph = spx.spx_plan_csr(M, K, A.nnz, rp, opts=opts)  # host row_ptr: planned on the host
    yd = dev(y0)
    spx.spx_spmv_csr(ph, A, dev(x), yd, 1.0, 0.5)
    assert np.array_equal(yd.cpu().numpy().view(np.uint32), got.view(np.uint32))


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-2.5, 0.0), (1.0, 0.5), (0.0, 3.0), (0.75, -1.25)])
def test_alpha_beta(alpha, beta):
    d = synth.random_coo(4, 777, 555, 0, 70)
    rp, col, val = oracle.build_csr(777, 555, d["row"], d["col"], d["val"])
    x = synth.uniform(4, synth.T_X, 555)
    y0 = synth.uniform(4, synth.T_Y, 777)
    check(777, 555, rp, col, val, x, y0, alpha, beta)


def test_beta_zero_does_not_read_y():
    d = synth.random_coo(5, 513, 300, 0, 40)
    rp, col, val = oracle.build_csr(513, 300, d["row"], d["col"], d["val"])
    x = synth.uniform(5, synth.T_X, 300)
    y0 = np.full(513, np.nan, np.float32)
    got, _ = run_spmv(513, 300, rp, col, val, x, y0, 1.0, 0.0)
    ref, bound = oracle.spmv(513, rp, col, val, x)
    assert_within(got, ref, bound)


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 0, 0), (1, 1, 1, 1), (5, 3, 0, 0), (257, 1, 0, 1),
                                           (1, 100000, 100000, 100000), (33, 70000, 0, 70000)])
def test_edge_shapes(M, K, lmin, lmax):
    d = synth.random_coo(6, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    x = synth.uniform(6, synth.T_X, K)
    y0 = synth.uniform(6, synth.T_Y, M)
    check(M, K, rp, col, val, x, y0, 1.0, 0.5, what=f"{M}x{K}")


@pytest.mark.parametrize("l", [0, 1, 4096, 4097, 8192, 8193, 65536, 200_000])
def test_row_of_ones_closed_form(l):
    """A row of l ones times x = 1 gives exactly l in fp32 (integers <= 2^24):
    pins the segment split and the fix-up sum."""
    rp = np.array([0, l], np.int32)
    col = np.arange(l, dtype=np.int32)
    K = max(l, 1)
    got, _ = run_spmv(1, K, rp, col, np.ones(l, np.float32), np.ones(K, np.float32), np.zeros(1, np.float32), 1.0,
                      0.0)
    assert got[0] == l


def test_deterministic_bitwise():
    cfg = synth.power_law_rows(7, M=200_000, mean=16.0)
    rp, col, val = oracle.build_csr(cfg["M"], cfg["K"], cfg["row"], cfg["col"], cfg["val"])
    A = csr_to_device(cfg["M"], cfg["K"], rp, col, val)
    plan = spx.spx_plan_csr(A.M, A.K, A.nnz, A.row_ptr)
    assert plan.info["long_rows"] > 0
    xd = dev(cfg["x"])
    outs = []
    for _ in range(3):
        yd = dev(cfg["y"])
        spx.spx_spmv_csr(plan, A, xd, yd, 1.0, 0.5)
        outs.append(yd.cpu().numpy())
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])


def test_uniform_short_rows_full():
    """4096 x 4096, lengths U{1..16}: every output row against the oracle."""
    cfg = synth.uniform_short_rows()
    rp, col, val = oracle.build_csr(cfg["M"], cfg["K"], cfg["row"], cfg["col"], cfg["val"])
    check(cfg["M"], cfg["K"], rp, col, val, cfg["x"], cfg["y"], cfg["alpha"], cfg["beta"])


@pytest.mark.slow
def test_power_law_full_size_sampled():
    """4,194,304^2 Zipf(2.1) rows (nnz ~ 67M), y = Ax + 0.5y, default plan as
    the benchmark runs it; 20k sampled rows plus every CTA and split row."""
    cfg = synth.power_law_rows()
    M, K = cfg["M"], cfg["K"]
    rp, col, val = spx.spx_build_csr(M, K, cfg["row"], cfg["col"], cfg["val"])
    A = csr_to_device(M, K, rp, col, val)
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr)
    yd = dev(cfg["y"])
    spx.spx_spmv_csr(plan, A, dev(cfg["x"]), yd, 1.0, 0.5)
    got = yd.cpu().numpy()
    tasks, longrows = plan.tasks()
    heavy = np.concatenate([tasks[(tasks[:, 0] & 255) == 1, 1], longrows[:, 0]])
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.integers(0, M, 20000), heavy, [0, M - 1]])).astype(np.int32)
    ref, bound = oracle.spmv(M, rp, col, val, cfg["x"], 1.0, 0.5, cfg["y"], rows=rows)
    assert_within(got[rows], ref, bound, what="power-law full size")
    assert plan.info["split_rows"] > 0 and plan.info["cta_rows"] > 0
    tolerance_self_check(got[rows], M, rp, col, val, cfg["x"], 1.0, 0.5, cfg["y"], rows=rows)


# ------------------------------------------------------------ the tolerance self-check

def _gamma(n):
    """gamma_n = n u / (1 - n u), u = 2^-24: the rounding-error factor of a sum of fp32 products
    with at most n roundings along any path from an input to the result."""
    u = 2.0 ** -24
    return n * u / (1.0 - n * u)


def tolerance_self_check(got, M, rp, col, val, x, alpha, beta, y0, rows=None):
    """[SpMM-ops] §5: check the low-precision result against a reference and report the error.
    (1) Against the fp32 index-order oracle, the stated tolerance widened by that oracle's own
    rounding bound gamma_(l+4) * bound.  (2) Against the fp64 oracle, the rounding bound itself:
    any fp32 summation order of l products (a tree, segments and a fix-up, fused multiply-adds)
    plus the alpha/beta epilogue has at most l + 4 roundings on every path, so a correct kernel
    can never leave it -- a test tolerance or bound formula that is too loose or too tight shows."""
    ref, bound = oracle.spmv(M, rp, col, val, x, alpha, beta, y0, rows=rows)
    r32 = oracle.spmv_f32(M, rp, col, val, x, alpha, beta, y0, rows=rows).astype(np.float64)
    L = np.diff(rp).astype(np.float64)
    if rows is not None:
        L = L[rows]
    g = _gamma(L + 4)
    got = np.asarray(got, np.float64)
    e32 = np.abs(got - r32)
    assert np.all(e32 <= (FP32_REL + g) * bound + FP32_ABS), "GPU vs fp32 index-order oracle"
    e64 = np.abs(got - ref)
    assert np.all(e64 <= g * bound), "GPU vs fp64 oracle outside the fp32 rounding bound"
    return float(np.max(e64 / np.maximum(g * bound, 1e-300), initial=0.0))


@pytest.mark.parametrize("opts", [None, SMALL_OPTS[1], SMALL_OPTS[6], SMALL_OPTS[11]])
def test_tolerance_self_check_power_law_small(opts):
    M = 3000
    L, _ = synth.lengths_zipf(3, M, 2.1, 100000, 12.0)
    L[:2] = (100000, 0)
    row, col = synth.cols_uniform(3, 200000, L)
    val = synth.uniform(3, synth.T_VAL, row.size)
    rp, col, val = oracle.build_csr(M, 200000, row, col, val)
    x = synth.uniform(3, synth.T_X, 200000)
    y0 = synth.uniform(3, synth.T_Y, M)
    got, _ = run_spmv(M, 200000, rp, col, val, x, y0, -1.5, 0.5, opts)
    tolerance_self_check(got, M, rp, col, val, x, -1.5, 0.5, y0)


def test_tolerance_self_check_uniform_short_rows():
    cfg = synth.uniform_short_rows()
    rp, col, val = oracle.build_csr(cfg["M"], cfg["K"], cfg["row"], cfg["col"], cfg["val"])
    got, _ = run_spmv(cfg["M"], cfg["K"], rp, col, val, cfg["x"], cfg["y"], cfg["alpha"], cfg["beta"])
    tolerance_self_check(got, cfg["M"], rp, col, val, cfg["x"], cfg["alpha"], cfg["beta"], cfg["y"])


def test_gather_probe_reads_every_nonzero():
    """The floor probe does the gather work: its partial sums add up to sum_p val_p * x[col_p]."""
    d = synth.random_coo(55, 30000, 70000, 0, 40)
    rp, col, val = oracle.build_csr(30000, 70000, d["row"], d["col"], d["val"])
    A = csr_to_device(30000, 70000, rp, col, val)
    x = synth.uniform(55, synth.T_X, 70000)
    parts = spx.spx_gather_probe(A, dev(x))
    torch.cuda.synchronize()
    prods = val.astype(np.float64) * x[col].astype(np.float64)
    assert abs(parts.double().sum().item() - prods.sum()) <= 1e-5 * np.abs(prods).sum() + 1e-6


@pytest.mark.parametrize("nbatch,beta,shared_x", [(1, 0.0, False), (2, 0.5, False), (5, -1.25, False),
                                                  (4, 0.0, True), (3, 2.0, True)])
def test_hostio_pipeline_equals_device_calls(nbatch, beta, shared_x):
    """The host-buffer pipeline gives, batch by batch, the device call's result bit for bit."""
    L, _ = synth.lengths_zipf(56, 40000, 2.1, 20000, 14.0)
    row, col = synth.cols_uniform(56, 50000, L)
    rp, col, val = oracle.build_csr(40000, 50000, row, col, synth.uniform(56, synth.T_VAL, row.size))
    A = csr_to_device(40000, 50000, rp, col, val)
    plan = spx.spx_plan_csr(40000, 50000, A.nnz, rp)
    xs = np.stack([synth.uniform(57 + b, synth.T_X, 50000) for b in range(1 if shared_x else nbatch)])
    ys = np.stack([synth.uniform(57 + b, synth.T_Y, 40000) for b in range(nbatch)])
    xh = torch.from_numpy(xs).pin_memory()
    yh = torch.from_numpy(ys.copy()).pin_memory()
    spx.spx_spmv_csr_hostio(plan, A, xh, yh, 1.5, beta)
    for b in range(nbatch):
        x = xs[0 if shared_x else b]
        yd = dev(ys[b])
        spx.spx_spmv_csr(plan, A, dev(x), yd, 1.5, beta)
        torch.cuda.synchronize()
        assert np.array_equal(yh[b].numpy().view(np.uint32), yd.cpu().numpy().view(np.uint32))
        ref, bound = oracle.spmv(40000, rp, col, val, x, 1.5, beta, ys[b])
        assert_within(yh[b].numpy(), ref, bound)


def test_spmv_calls_capture_in_a_cuda_graph():
    """The SpMV call enqueues kernels only (no allocation, no host synchronisation): it can be
    captured in a CUDA graph, and replays give the direct call's result bit for bit."""
    d = synth.random_coo(58, 5000, 4000, 0, 30)
    rp, col, val = oracle.build_csr(5000, 4000, d["row"], d["col"], d["val"])
    A = csr_to_device(5000, 4000, rp, col, val)
    plan = spx.spx_plan_csr(5000, 4000, A.nnz, rp)
    x = dev(synth.uniform(58, synth.T_X, 4000))
    y_direct = dev(np.zeros(5000, np.float32))
    spx.spx_spmv_csr(plan, A, x, y_direct, 2.0, 0.0)
    y = dev(np.zeros(5000, np.float32))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        spx.spx_spmv_csr(plan, A, x, y, 2.0, 0.0, stream=s)
        torch.cuda.synchronize()
        y.zero_()
        with torch.cuda.graph(g, stream=s):
            for _ in range(4):
                spx.spx_spmv_csr(plan, A, x, y, 2.0, 0.0, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_direct.cpu().numpy().view(np.uint32))
