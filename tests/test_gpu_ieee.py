"""IEEE special values through every product.

Two properties that hold for any input and pin down where each output's sum
comes from:
- beta == 0 makes the output write-only: NaN already in y or C never
  propagates (the BLAS convention the library documents);
- a NaN planted in x, or in one column n of B, reaches exactly the outputs
  whose sums include it: the rows with a stored entry in that column of A (for
  BSR every row of a stored block, for WCSR every row of a window whose column
  list holds it), and for SpMM only output column n.  Padding (SELL slots,
  WCSR padding columns, empty rows) is never multiplied into a sum.

An index slip in a gather, a segmented reduction, a split row's partials or a
fix-up moves or spreads the NaN; every output that stays finite is checked
against the fp64 oracle run on the same data with the planted entries zeroed
(those outputs do not depend on them)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import BF16_ABS, BF16_REL, assert_within, csr_to_device, dev

pytestmark = pytest.mark.gpu

BF16_NAN, F16_NAN = 0x7FC0, 0x7E00


def _skewed(seed, M, K, lmax):
    L, _ = synth.lengths_zipf(seed, M, 2.1, lmax, 12.0)
    row, col = synth.cols_uniform(seed, K, L)
    return oracle.build_csr(M, K, row, col, synth.uniform(seed, synth.T_VAL, row.size))


def _rows_touching(M, rp, col, cols):
    """Rows holding a stored entry in any of `cols`."""
    rows = np.repeat(np.arange(M), np.diff(rp))
    mask = np.zeros(M, bool)
    mask[rows[np.isin(col, cols)]] = True
    return mask


def _planted_cols(rp, col, K, seed):
    """Three columns: one of the longest row's, one of a short row's, one random (possibly unused)."""
    lens = np.diff(rp)
    r_long = int(np.argmax(lens))
    short = np.flatnonzero((lens > 0) & (lens < 8))
    r_short = int(short[len(short) // 2])
    rnd = int(synth.permutation(seed, K)[0])
    return np.unique(np.array([col[rp[r_long] + lens[r_long] // 3], col[rp[r_short]], rnd], np.int32))


def _check_masked(got, mask, ref, bound, rel=None, ab=None, what=""):
    """NaN exactly where `mask` holds; elsewhere finite and within the oracle's bound."""
    nan = np.isnan(got)
    assert np.array_equal(nan, mask), (f"{what}: NaN at {np.flatnonzero(nan & ~mask)[:5].tolist()} not expected, "
                                       f"missing at {np.flatnonzero(mask & ~nan)[:5].tolist()}")
    kw = {} if rel is None else {"rel": rel, "ab": ab}
    assert_within(got[~mask], ref[~mask], bound[~mask], what=what, **kw)


PLAN_OPTS = [None, {"pack_max": 64, "cta_max": 1000, "seg_nnz": 500},
             {"block_nnz": 1024, "pack_max": 8, "cta_max": 8, "seg_nnz": 3, "lanes_div": 0}]


@pytest.mark.parametrize("opts", PLAN_OPTS)
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_spmv_csr_nan_in_x(opts, beta):
    """Planned CSR SpMV (groups in lanes and segmented modes, CTA rows, split rows + fix-up)."""
    M, K = 6000, 30000
    rp, col, val = _skewed(61, M, K, 9000)
    A = csr_to_device(M, K, rp, col, val)
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, opts)
    J = _planted_cols(rp, col, K, 61)
    x = synth.uniform(61, synth.T_X, K)
    x0 = x.copy()
    x[J] = np.nan
    y0 = np.full(M, np.nan, np.float32) if beta == 0.0 else synth.uniform(61, synth.T_Y, M)
    yd = dev(y0)
    spx.spx_spmv_csr(plan, A, dev(x), yd, 1.0, beta)
    x0[J] = 0.0
    ref, bound = oracle.spmv(M, rp, col, val, x0, 1.0, beta, y0)
    mask = _rows_touching(M, rp, col, J)
    assert mask.sum() >= 2
    _check_masked(yd.cpu().numpy(), mask, ref, bound, what=f"csr opts={opts} beta={beta}")


@pytest.mark.parametrize("fmt", ["coo", "sell"])
def test_spmv_coo_sell_nan_in_x(fmt):
    """COO (segmented reduction over row-sorted triplets) and SELL-C-sigma (padded slices, long-row pieces)."""
    M, K = 6000, 30000
    rp, col, val = _skewed(62, M, K, 9000)
    J = _planted_cols(rp, col, K, 62)
    x = synth.uniform(62, synth.T_X, K)
    x0 = x.copy()
    x[J] = np.nan
    yd = dev(np.full(M, np.nan, np.float32))
    if fmt == "coo":
        rows = np.repeat(np.arange(M, dtype=np.int32), np.diff(rp))
        spx.spx_spmv_coo(M, K, dev(rows), dev(col), dev(val), dev(x), yd, 1.0, 0.0)
    else:
        S = spx.Sell(M, K, dev(rp), dev(col), dev(val))
        spx.spx_spmv_sell(S, dev(x), yd, 1.0, 0.0)
    x0[J] = 0.0
    ref, bound = oracle.spmv(M, rp, col, val, x0)
    _check_masked(yd.cpu().numpy(), _rows_touching(M, rp, col, J), ref, bound, what=fmt)


def test_dual_nan_flows_through_u():
    """u <- A v + 0 u over a NaN-filled u with one NaN in v, then v <- A^T u + 0 v: u is NaN on
    the rows that hold the planted column, v on the columns those rows hold."""
    cfg = synth.banded_pair(12, m=3000, n=1500, half=100, iters=1)
    m, n = cfg["M"], cfg["K"]
    rp, col, val = oracle.build_csr(m, n, cfg["row"], cfg["col"], cfg["val"])
    trp, tc, tv = oracle.transpose(m, n, rp, col, val)
    A, At = csr_to_device(m, n, rp, col, val), csr_to_device(n, m, trp, tc, tv)
    pA, pAt = spx.spx_plan_csr(m, n, A.nnz, A.row_ptr), spx.spx_plan_csr(n, m, At.nnz, At.row_ptr)
    j = int(col[rp[m // 2]])
    v0 = cfg["v0"].copy()
    v0[j] = np.nan
    u, v = dev(np.full(m, np.nan, np.float32)), dev(v0)
    spx.spx_spmv_csr_dual(pA, pAt, A, At, v, u, 1.0, 0.0, 1.0, 0.0)
    ug, vg = u.cpu().numpy(), v.cpu().numpy()
    umask = _rows_touching(m, rp, col, [j])
    vmask = _rows_touching(n, trp, tc, np.flatnonzero(umask))
    v0[j] = 0.0
    ref, bound = oracle.spmv(m, rp, col, val, v0)
    _check_masked(ug, umask, ref, bound, what="u")
    uz = np.where(umask, 0.0, ug).astype(np.float32)
    ref, bound = oracle.spmv(n, trp, tc, tv, uz)
    _check_masked(vg, vmask, ref, bound, what="v")


def _spmm_mask(M, rp, col, N, planted):
    mask = np.zeros((M, N), bool)
    for j, c in planted:
        mask[_rows_touching(M, rp, col, [j]), c] = True
    return mask


def _planted_b(rp, col, K, N, seed):
    """(row of B, column of B) pairs: columns of a long and a short row, spread over the output columns."""
    J = _planted_cols(rp, col, K, seed)
    return [(int(j), int((7 * i + 3) % N)) for i, j in enumerate(J)] + [(int(J[0]), N - 1)]


@pytest.mark.parametrize("N,how", [(n, "plain") for n in (1, 8, 12, 32, 33, 128, 256)]
                         + [(n, "planned") for n in (4, 32, 128, 256)])
def test_spmm_f32_nan_in_b(N, how):
    """fp32 CSR SpMM, every variant (small-N, float4, float4-wide, scalar) and the planned long-row path
    (N a multiple of 4); C starts NaN and beta = 0."""
    M, K = 3000, 20000
    rp, col, val = _skewed(63, M, K, 9000)
    A = csr_to_device(M, K, rp, col, val)
    Bm = synth.uniform(N + 63, synth.T_B, K * N).reshape(K, N)
    planted = _planted_b(rp, col, K, N, 63)
    B0 = Bm.copy()
    for j, c in planted:
        Bm[j, c] = np.nan
        B0[j, c] = 0.0
    Cd = torch.full((M, N), float("nan"), device="cuda")
    if how == "plain":
        spx.spx_spmm_csr(A, dev(Bm), Cd, 1.0, 0.0)
    else:
        plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, {"pack_max": 64, "cta_max": 1000, "seg_nnz": 500})
        spx.spx_spmm_csr_planned(plan, A, dev(Bm), Cd, 1.0, 0.0)
    ref, bound = oracle.spmm(M, rp, col, val, B0)
    _check_masked(Cd.cpu().numpy(), _spmm_mask(M, rp, col, N, planted), ref, bound, what=f"{how} N={N}")


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("how", ["plain", "planned"])
@pytest.mark.parametrize("N", [32, 128])
def test_spmm_16bit_nan_in_b(fmt, how, N):
    M, K = 2000, 12000
    rp, col, val = _skewed(64, M, K, 6000)
    Bf = synth.uniform(N + 64, synth.T_B, K * N).reshape(K, N)
    if fmt == "bf16":
        vb, Bb = synth.to_bf16_bits(val), synth.to_bf16_bits(Bf).reshape(K, N)
        vf, B0 = synth.bf16_bits_to_f32(vb), synth.bf16_bits_to_f32(Bb).reshape(K, N)
        nan_bits = BF16_NAN
    else:
        vh, Bh = val.astype(np.float16), Bf.astype(np.float16)
        vb, Bb, vf, B0 = vh.view(np.uint16), Bh.view(np.uint16).copy(), vh.astype(np.float32), Bh.astype(np.float32)
        nan_bits = F16_NAN
    planted = _planted_b(rp, col, K, N, 64)
    for j, c in planted:
        Bb[j, c] = nan_bits
        B0[j, c] = 0.0
    A = spx.Csr(M, K, dev(rp), dev(col), dev(vb.view(np.int16)))
    Cd = torch.full((M, N), float("nan"), device="cuda")
    Bd = dev(Bb.view(np.int16))
    if how == "plain":
        (spx.spx_spmm_csr_bf16 if fmt == "bf16" else spx.spx_spmm_csr_f16)(A, Bd, Cd, 1.0, 0.0)
    else:
        plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, {"pack_max": 32, "cta_max": 500, "seg_nnz": 400})
        (spx.spx_spmm_csr_bf16_planned if fmt == "bf16" else spx.spx_spmm_csr_f16_planned)(plan, A, Bd, Cd, 1.0, 0.0)
    ref, bound = oracle.spmm(M, rp, col, vf, B0)
    _check_masked(Cd.cpu().numpy(), _spmm_mask(M, rp, col, N, planted), ref, bound, what=f"{fmt} {how} N={N}")


def _bits_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.parametrize("how", ["plain", "planned"])
def test_bsr_nan_in_b(how):
    """Tensor-core BSR SpMM (long block-rows split in the planned call): a NaN in B row j, column n
    reaches column n of every row of each block-row with a stored block in block column j / 64."""
    M, N = 2048, 256
    c = synth.block_sparse_skewed(9, M=M, N=N)
    K = c["K"]
    rp, col, val = oracle.build_csr(M, K, c["row"], c["col"], c["val_bf16"])
    brp, bcol, bval, _ = oracle.build_bsr(M, K, rp, col, val, 64, 64)
    Bb = c["B_bf16"].copy()
    long_I = int(np.argmax(np.diff(brp)))
    planted = [(int(bcol[brp[long_I] + 5]) * 64 + 17, 3), (int(bcol[brp[1]]) * 64 + 63, N - 1),
               (int(bcol[brp[long_I]]) * 64, 128)]
    mask = np.zeros((M, N), bool)
    for j, n in planted:
        Bb[j, n] = BF16_NAN
        for I in range(M // 64):
            if (j // 64) in bcol[brp[I]:brp[I + 1]]:
                mask[I * 64:(I + 1) * 64, n] = True
    B0 = Bb.copy()
    for j, n in planted:
        B0[j, n] = 0
    dbrp, dbcol, dbval = dev(brp), dev(bcol), _bits_dev(bval.reshape(-1))
    Cd = torch.full((M, N), float("nan"), device="cuda")
    if how == "plain":
        spx.spx_spmm_bsr(M, K, 64, 64, dbrp, dbcol, dbval, _bits_dev(Bb), Cd)
    else:
        P = spx.BsrPlan(M, bcol.size, dbrp, max_chunks=8)
        assert P.info["split_windows"] > 0
        spx.spx_spmm_bsr_planned(P, M, K, 64, 64, dbrp, dbcol, dbval, _bits_dev(Bb), Cd)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(val), synth.bf16_bits_to_f32(B0))
    _check_masked(Cd.cpu().numpy(), mask, ref, bound, rel=BF16_REL, ab=BF16_ABS, what=f"bsr {how}")


@pytest.mark.parametrize("how", ["plain", "planned"])
def test_wcsr_nan_in_b(how):
    """Tensor-core WCSR SpMM (wide windows split in the planned call): a NaN in B row j, column n
    reaches column n of every row of each window whose column list holds j, and never leaks
    through padding columns."""
    M, N = 2048, 256
    c = synth.window_pool_skewed(7, M=M, N=N)
    K = c["K"]
    rp, col, val = oracle.build_csr(M, K, c["row"], c["col"], c["val_bf16"])
    wp, wc, wv, _ = oracle.build_wcsr(M, K, rp, col, val)
    assert (wc < 0).any()  # some padding columns exist
    Bb = c["B_bf16"].copy()
    wide = int(np.argmax(np.diff(wp)))
    planted = [(int(wc[wp[wide] * 64 + 100]), 5), (int(wc[wp[3] * 64]), N - 1), (int(wc[wp[wide] * 64]), 200)]
    mask = np.zeros((M, N), bool)
    for j, n in planted:
        Bb[j, n] = BF16_NAN
        for w in range(wp.size - 1):
            if j in wc[wp[w] * 64:wp[w + 1] * 64]:
                mask[w * 64:min(M, (w + 1) * 64), n] = True
    B0 = Bb.copy()
    for j, n in planted:
        B0[j, n] = 0
    dwp, dwc, dwv = dev(wp), dev(wc), _bits_dev(wv.reshape(-1))
    Cd = torch.full((M, N), float("nan"), device="cuda")
    if how == "plain":
        spx.spx_spmm_wcsr(M, K, dwp, dwc, dwv, _bits_dev(Bb), Cd)
    else:
        P = spx.WcsrPlan(M, wc.size // 64, dwp, max_chunks=4)
        assert P.info["split_windows"] > 0
        spx.spx_spmm_wcsr_planned(P, M, K, dwp, dwc, dwv, _bits_dev(Bb), Cd)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(val), synth.bf16_bits_to_f32(B0))
    _check_masked(Cd.cpu().numpy(), mask, ref, bound, rel=BF16_REL, ab=BF16_ABS, what=f"wcsr {how}")
