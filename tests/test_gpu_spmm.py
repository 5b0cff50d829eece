"""CSR SpMM parity against the fp64 oracle: every variant (chosen by N),
alpha/beta, leading dimensions, ragged tails, and the clustered 1M x 1M
workload at N = 32 and N = 128 on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import assert_within, csr_to_device, dev

pytestmark = pytest.mark.gpu


def run(M, K, d, N, alpha=1.0, beta=0.0, ldb=None, ldc=None, seed=0, want_variant=None):
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    A = csr_to_device(M, K, rp, col, val)
    ldb = ldb or N
    ldc = ldc or N
    Bfull = synth.uniform(seed, synth.T_B, K * ldb).reshape(K, ldb)
    Cfull = synth.uniform(seed, synth.T_Y, M * ldc).reshape(M, ldc)
    Bd = dev(Bfull)[:, :N]
    Cd = dev(Cfull)
    Cv = Cd[:, :N]
    if want_variant:
        assert spx.spx_spmm_csr_variant(Bd, Cv) == want_variant
    spx.spx_spmm_csr(A, Bd, Cv, alpha, beta)
    torch.cuda.synchronize()
    got = Cd.cpu().numpy()
    ref, bound = oracle.spmm(M, rp, col, val, Bfull[:, :N], alpha, beta, Cfull[:, :N])
    assert_within(got[:, :N], ref, bound, what=f"N={N}")
    assert np.array_equal(got[:, N:], Cfull[:, N:])  # columns beyond N untouched


@pytest.mark.parametrize("N,variant", [(1, "small-N"), (2, "small-N"), (3, "small-N"), (8, "small-N"),
                                       (12, "float4"), (16, "float4"), (32, "float4"),
                                       (64, "float4"), (100, "float4"), (128, "float4"),
                                       (132, "float4-wide"), (256, "float4-wide"), (520, "float4-wide"),
                                       (9, "scalar"), (33, "scalar"), (130, "scalar")])
def test_variants(N, variant):
    d = synth.random_coo(N, 1111, 777, 0, 50)
    run(1111, 777, d, N, alpha=1.0, beta=0.0, want_variant=variant, seed=N)


@pytest.mark.parametrize("N,tile", [(32, 8), (32, 16), (64, 32), (128, 16), (100, 64), (256, 128), (48, 8)])
def test_column_tiles(N, tile):
    d = synth.random_coo(N + tile, 900, 600, 0, 40)
    M, K = 900, 600
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    A = csr_to_device(M, K, rp, col, val)
    B = synth.uniform(5, synth.T_B, K * N).reshape(K, N)
    Cd = torch.full((M, N), float("nan"), device="cuda")
    spx.spx_spmm_csr(A, dev(B), Cd, col_tile=tile)
    torch.cuda.synchronize()
    ref, bound = oracle.spmm(M, rp, col, val, B)
    assert_within(Cd.cpu().numpy(), ref, bound, what=f"N={N} tile={tile}")


@pytest.mark.parametrize("alpha,beta", [(2.0, 0.0), (1.0, -0.5), (0.0, 1.5)])
@pytest.mark.parametrize("N", [4, 32, 256])
def test_alpha_beta(alpha, beta, N):
    d = synth.random_coo(3, 500, 400, 0, 30)
    run(500, 400, d, N, alpha, beta, seed=3)


@pytest.mark.parametrize("N,ldb,ldc", [(32, 36, 40), (128, 132, 128), (20, 21, 20)])
def test_leading_dimensions(N, ldb, ldc):
    d = synth.random_coo(4, 300, 200, 0, 25)
    run(300, 200, d, N, 1.0, 0.5, ldb=ldb, ldc=ldc, seed=4)


def test_long_and_empty_rows():
    L = np.zeros(70, np.int32)
    L[3] = 5000
    L[10:20] = 1
    L[40] = 900
    row, col = synth.cols_uniform(8, 6000, L)
    d = dict(row=row, col=col, val=synth.uniform(8, synth.T_VAL, row.size))
    for N in (2, 32, 160):
        run(70, 6000, d, N, 1.0, 0.25, seed=8)


@pytest.mark.slow
@pytest.mark.parametrize("N", [32, 128])
def test_clustered_full_size_sampled(N):
    """1,048,576^2, Poisson(32) rows in 4x4 clusters, B dense K x N: 4096
    sampled rows (whole 4-row clusters) against the oracle."""
    cfg = synth.clustered_spmm(N=N)
    M, K = cfg["M"], cfg["K"]
    rp, col, val = spx.spx_build_csr(M, K, cfg["row"], cfg["col"], cfg["val"])
    A = csr_to_device(M, K, rp, col, val)
    Bd = dev(cfg["B"])
    Cd = torch.full((M, N), float("nan"), device="cuda")
    spx.spx_spmm_csr(A, Bd, Cd)
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    g = rng.integers(0, M // 4, 1024)
    rows = np.unique((g[:, None] * 4 + np.arange(4)).ravel()).astype(np.int32)
    got = Cd[torch.from_numpy(rows).long().cuda()].cpu().numpy()
    ref, bound = oracle.spmm(M, rp, col, val, cfg["B"], rows=rows)
    assert_within(got, ref, bound, what=f"clustered N={N}")


@pytest.mark.parametrize("N,alpha,beta", [(8, 1.0, 0.0), (32, 1.0, 0.0), (64, -2.0, 0.5), (128, 1.0, 0.0),
                                          (256, 0.5, -1.0), (20, 1.0, 0.0)])
def test_bf16_values(N, alpha, beta):
    """bf16 A values and B: exact widening and exact products, so the fp32
    tolerance against the fp64 oracle (fed the same values widened) holds."""
    M, K = 700, 500
    d = synth.random_coo(N + 1, M, K, 0, 45)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    vb = synth.to_bf16_bits(val)
    Bb = synth.to_bf16_bits(synth.uniform(N, synth.T_B, K * N)).reshape(K, N)
    C0 = synth.uniform(N, synth.T_Y, M * N).reshape(M, N)
    A = spx.Csr(M, K, dev(rp), dev(col), dev(vb.view(np.int16)))
    Cd = dev(C0)
    spx.spx_spmm_csr_bf16(A, dev(Bb.view(np.int16)), Cd, alpha, beta)
    torch.cuda.synchronize()
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(vb), synth.bf16_bits_to_f32(Bb).reshape(K, N),
                             alpha, beta, C0)
    assert_within(Cd.cpu().numpy(), ref, bound, what=f"bf16 N={N}")


@pytest.mark.slow
def test_bf16_clustered_full_size_sampled():
    cfg = synth.clustered_spmm(N=32)
    M, K = cfg["M"], cfg["K"]
    rp, col, val = spx.spx_build_csr(M, K, cfg["row"], cfg["col"], cfg["val"])
    vb = synth.to_bf16_bits(val)
    Bb = synth.to_bf16_bits(cfg["B"]).reshape(K, 32)
    A = spx.Csr(M, K, dev(rp), dev(col), dev(vb.view(np.int16)))
    Cd = torch.empty(M, 32, device="cuda")
    spx.spx_spmm_csr_bf16(A, dev(Bb.view(np.int16)), Cd)
    torch.cuda.synchronize()
    rows = np.unique((np.random.default_rng(3).integers(0, M // 4, 512)[:, None] * 4 + np.arange(4)).ravel())
    rows = rows.astype(np.int32)
    got = Cd[torch.from_numpy(rows).long().cuda()].cpu().numpy()
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(vb), synth.bf16_bits_to_f32(Bb).reshape(K, 32),
                             rows=rows)
    assert_within(got, ref, bound, what="bf16 clustered")


def test_bf16_long_and_empty_rows():
    """A CTA whose rows hold more nonzeros than its shared-memory stage reads
    A from global memory; its neighbours are staged.  Both paths, bf16."""
    L = np.zeros(70, np.int32)
    L[3] = 5000
    L[10:20] = 1
    L[40] = 900
    row, col = synth.cols_uniform(9, 6000, L)
    rp, col, val = oracle.build_csr(70, 6000, row, col, synth.uniform(9, synth.T_VAL, row.size))
    vb = synth.to_bf16_bits(val)
    for N in (32, 160):
        Bb = synth.to_bf16_bits(synth.uniform(N, synth.T_B, 6000 * N)).reshape(6000, N)
        C0 = synth.uniform(N, synth.T_Y, 70 * N).reshape(70, N)
        Cd = dev(C0)
        spx.spx_spmm_csr_bf16(spx.Csr(70, 6000, dev(rp), dev(col), dev(vb.view(np.int16))), dev(Bb.view(np.int16)),
                              Cd, 1.0, 0.25)
        torch.cuda.synchronize()
        ref, bound = oracle.spmm(70, rp, col, synth.bf16_bits_to_f32(vb), synth.bf16_bits_to_f32(Bb).reshape(6000, N),
                                 1.0, 0.25, C0)
        assert_within(Cd.cpu().numpy(), ref, bound, what=f"bf16 long rows N={N}")


@pytest.mark.parametrize("N", [4, 32, 128, 256])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.5, -1.5)])
def test_f16_values(N, alpha, beta):
    """fp16 A values and B (subnormals and the largest finite values included):
    exact widening and exact products, so the fp32 sums meet the fp32 bound."""
    M, K = 700, 900
    d = synth.random_coo(N + 11, M, K, 0, 60)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    vh = val.astype(np.float16)
    Bh = synth.uniform(N + 12, synth.T_B, K * N).astype(np.float16).reshape(K, N)
    Bh[0, :2] = [np.float16(6.0e-8), np.float16(-6.5e4)]  # a subnormal and a near-maximal value
    vh[:3] = [np.float16(3.0e-5), np.float16(1.0e3), np.float16(-2.0e-7)]
    A = spx.Csr(M, K, dev(rp), dev(col), dev(vh.view(np.int16)))
    C0 = synth.uniform(N + 13, synth.T_Y, M * N).reshape(M, N)
    Cd = dev(C0)
    spx.spx_spmm_csr_f16(A, dev(Bh.view(np.int16)), Cd, alpha, beta)
    ref, bound = oracle.spmm(M, rp, col, vh.astype(np.float64), Bh.astype(np.float64), alpha, beta, C0)
    assert_within(Cd.cpu().numpy(), ref, bound, what=f"f16 N={N}")


def test_f16_rejects_unsupported_shapes():
    rp = dev(np.array([0, 1], np.int32))
    A = spx.Csr(1, 1, rp, dev(np.array([0], np.int32)), dev(np.zeros(1, np.int16)))
    with pytest.raises(spx.SpxError) as e:
        spx.spx_spmm_csr_f16(A, dev(np.zeros((1, 6), np.int16)), dev(np.zeros((1, 6), np.float32)))
    assert e.value.code == -7  # N not a multiple of 4


def _skewed(seed, M, K, lmax):
    """Power-law rows up to lmax (< K) entries (a few long ones), distinct uniform columns."""
    assert lmax < K
    L, _ = synth.lengths_zipf(seed, M, 2.1, lmax, 12.0)
    row, col = synth.cols_uniform(seed, K, L)
    val = synth.uniform(seed, synth.T_VAL, row.size)
    return oracle.build_csr(M, K, row, col, val)


PLAN_OPTS = [None, {"pack_max": 64, "cta_max": 1000, "seg_nnz": 500},
             {"block_nnz": 1024, "pack_max": 8, "cta_max": 8, "seg_nnz": 3, "lanes_div": 0}]


@pytest.mark.parametrize("opts", PLAN_OPTS)
@pytest.mark.parametrize("N,alpha,beta", [(4, 1.0, 0.0), (32, 1.0, 0.0), (32, -0.5, 2.0), (128, 1.0, 0.0),
                                          (256, 0.75, -1.0), (20, 1.0, 0.5)])
def test_planned_skewed_rows(opts, N, alpha, beta):
    """Planned SpMM on power-law rows (CTA rows and split rows under several plans) against the fp64 oracle."""
    M, K = 3000, 20000
    rp, col, val = _skewed(31, M, K, 9000)
    A = csr_to_device(M, K, rp, col, val)
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, opts)
    assert plan.info["cta_rows"] + plan.info["split_rows"] > 0
    Bm = synth.uniform(N + 2, synth.T_B, K * N).reshape(K, N)
    C0 = synth.uniform(N + 3, synth.T_Y, M * N).reshape(M, N)
    Cd = dev(C0)
    spx.spx_spmm_csr_planned(plan, A, dev(Bm), Cd, alpha, beta)
    ref, bound = oracle.spmm(M, rp, col, val, Bm, alpha, beta, C0)
    assert_within(Cd.cpu().numpy(), ref, bound, what=f"planned N={N} opts={opts}")
    C2 = dev(C0)
    spx.spx_spmm_csr_planned(plan, A, dev(Bm), C2, alpha, beta)
    assert torch.equal(Cd, C2)  # fixed-order sums: reproducible


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_planned_16bit(fmt):
    M, K, N = 2000, 12000, 64
    rp, col, val = _skewed(32, M, K, 6000)
    if fmt == "bf16":
        vb, Bb = synth.to_bf16_bits(val), synth.to_bf16_bits(synth.uniform(5, synth.T_B, K * N)).reshape(K, N)
        vf, Bf, fn = synth.bf16_bits_to_f32(vb), synth.bf16_bits_to_f32(Bb).reshape(K, N), spx.spx_spmm_csr_bf16_planned
    else:
        vb, Bb = val.astype(np.float16), synth.uniform(5, synth.T_B, K * N).astype(np.float16).reshape(K, N)
        vf, Bf, fn = vb.astype(np.float32), Bb.astype(np.float32), spx.spx_spmm_csr_f16_planned
    A = spx.Csr(M, K, dev(rp), dev(col), dev(vb.view(np.int16)))
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, {"pack_max": 32, "cta_max": 500, "seg_nnz": 400})
    Cd = torch.empty(M, N, device="cuda")
    fn(plan, A, dev(Bb.view(np.int16)), Cd)
    ref, bound = oracle.spmm(M, rp, col, vf, Bf)
    assert_within(Cd.cpu().numpy(), ref, bound, what=f"planned {fmt}")


def test_planned_errors():
    M, K = 300, 300
    rp, col, val = _skewed(33, M, K, 250)
    A = csr_to_device(M, K, rp, col, val)
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, {"pack_max": 16, "cta_max": 32, "seg_nnz": 8})
    B, C = torch.zeros(K, 32, device="cuda"), torch.zeros(M, 32, device="cuda")
    other = spx.spx_plan_csr(M + 1, K, A.nnz, torch.cat([A.row_ptr, A.row_ptr[-1:]]))
    cases = [(lambda: spx.spx_spmm_csr_planned(other, A, B, C), -1),                               # another matrix
             (lambda: spx.spx_spmm_csr_planned(plan, A, B, C, scratch=torch.zeros(1, device="cuda")), -1),
             (lambda: spx.spx_spmm_csr_planned(plan, A, B[:, :6], C[:, :6]), -7),                  # N % 4
             (lambda: spx.spx_spmm_csr_planned(spx.Plan(M, K, A.nnz, A.row_ptr, upload=False), A, B, C), -10)]
    for f, code in cases:
        with pytest.raises(spx.SpxError) as e:
            f()
        assert e.value.code == code


@pytest.mark.slow
def test_planned_power_law_full_size_sampled():
    """The 4,194,304-row power-law matrix (rows up to 200,000) at N = 32, sampled rows incl. every long row."""
    c = synth.power_law_rows()
    M, K = c["M"], c["K"]
    rp, col, val = spx.spx_build_csr(M, K, c["row"], c["col"], c["val"])
    A = csr_to_device(M, K, rp, col, val)
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr)
    N = 32
    Bm = synth.uniform(7, synth.T_B, K * N).reshape(K, N)
    Cd = torch.empty(M, N, device="cuda")
    spx.spx_spmm_csr_planned(plan, A, dev(Bm), Cd)
    L = np.diff(rp)
    rows = np.unique(np.concatenate([np.nonzero(L > plan.opts["pack_max"])[0], np.arange(0, M, 4099)])).astype(np.int32)
    ref, bound = oracle.spmm(M, rp, col, val, Bm, rows=rows)
    assert_within(Cd[torch.from_numpy(rows).long().cuda()].cpu().numpy(), ref, bound, what="planned power-law")


def test_planned_without_long_rows_equals_plain():
    """A plan whose rows are all short changes nothing: the planned call equals spx_spmm_csr bit for bit."""
    M, K, N = 5000, 3000, 64
    d = synth.random_coo(34, M, K, 0, 40)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    A = csr_to_device(M, K, rp, col, val)
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr)
    assert plan.info["cta_rows"] == 0 and plan.info["split_rows"] == 0
    Bm = dev(synth.uniform(35, synth.T_B, K * N).reshape(K, N))
    C1, C2 = torch.empty(M, N, device="cuda"), torch.empty(M, N, device="cuda")
    spx.spx_spmm_csr(A, Bm, C1, 2.0, 0.0)
    spx.spx_spmm_csr_planned(plan, A, Bm, C2, 2.0, 0.0)
    assert torch.equal(C1, C2)


def test_planned_empty_matrix():
    for M, K in ((0, 5), (7, 0), (7, 5)):
        rp = np.zeros(M + 1, np.int32)
        A = csr_to_device(M, K, rp, np.zeros(0, np.int32), np.zeros(0, np.float32))
        plan = spx.spx_plan_csr(M, K, 0, A.row_ptr)
        C = torch.full((M, 8), 3.0, device="cuda")
        spx.spx_spmm_csr_planned(plan, A, torch.zeros(K, 8, device="cuda"), C, 1.0, 0.5)
        assert torch.equal(C, torch.full((M, 8), 1.5, device="cuda"))
