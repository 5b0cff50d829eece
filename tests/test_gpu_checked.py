"""The bounds-checked build (libspx_check.so, the same sources compiled with
SPX_CHECK): every index a kernel reads from the caller's arrays is tested
before it is used, a failed test skips the access and is reported as
SPX_ERR_INDEX_RANGE by spx_last_device_error ([LSMR-dual] §8: the sanitizer run
of the operator pair finds no access errors; compute-sanitizer itself is not
available here, so this build stands in for it).

Valid inputs give the product build's results bit for bit.  Corrupted inputs
-- planted here, on the host side of the calls, and only ever handed to the
checked build -- are reported, leave the memory around the outputs untouched,
and leave the context usable."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import assert_within, csr_to_device, dev

pytestmark = pytest.mark.gpu

INDEX_RANGE = -2


def bits(t):
    return t.cpu().numpy().view(np.uint32)


def _csr(seed, M, K, mean=10.0, lmax=20000):
    L, _ = synth.lengths_zipf(seed, M, 2.1, lmax, mean)
    L[:3] = (9000, 700, 0)  # a split row, a CTA row, an empty row
    row, col = synth.cols_uniform(seed, K, L)
    return oracle.build_csr(M, K, row, col, synth.uniform(seed, synth.T_VAL, row.size))


def _guarded(n, fill):
    g = torch.full((n + 64,), 777.0, device="cuda")
    g[32:32 + n] = torch.from_numpy(np.ascontiguousarray(fill, np.float32)).cuda()
    return g, g[32:32 + n]


def _guards_intact(g, n):
    h = g.cpu().numpy()
    return np.all(h[:32] == 777.0) and np.all(h[32 + n:] == 777.0)


@pytest.mark.parametrize("opts", [None, dict(block_nnz=1024, lanes_div=0),
                                  dict(block_nnz=64, block_rows=3, pack_max=8, cta_max=20, seg_nnz=7, lanes_div=2)])
def test_valid_spmv_is_bitwise_the_product_build(opts):
    M, K = 4000, 30000
    rp, col, val = _csr(1, M, K)
    x = synth.uniform(1, synth.T_X, K)
    y0 = synth.uniform(1, synth.T_Y, M)
    A = csr_to_device(M, K, rp, col, val)
    y_prod = dev(y0)
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, opts=opts)
    spx.spx_spmv_csr(plan, A, dev(x), y_prod, 1.5, 0.5)
    with spx.checked_build():
        pc = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, opts=opts)
        y_chk = dev(y0)
        spx.spx_spmv_csr(pc, A, dev(x), y_chk, 1.5, 0.5)
        assert spx.spx_last_device_error() == 0
    torch.cuda.synchronize()
    assert np.array_equal(bits(y_chk), bits(y_prod))


@pytest.mark.parametrize("opts", [None, dict(block_nnz=1024, lanes_div=0)])
def test_spmv_bad_columns_reported_and_skipped(opts):
    """Columns past K and below 0 in a packed row, the CTA row and the split row: reported; each bad term counts
    as zero (the oracle with those values zeroed), and nothing around y changes."""
    M, K = 4000, 30000
    rp, col, val = _csr(2, M, K)
    bad = np.array([rp[0] + 5, rp[1] + 3, rp[10] if rp[11] > rp[10] else rp[20], rp[0] + 8000], np.int64)
    col_bad = col.copy()
    col_bad[bad[:2]] = K + 1000
    col_bad[bad[2:]] = -5
    x = synth.uniform(2, synth.T_X, K)
    y0 = synth.uniform(2, synth.T_Y, M)
    with spx.checked_build():
        A = csr_to_device(M, K, rp, col_bad, val)
        plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, opts=opts)
        assert plan.info["split_rows"] >= 1 and plan.info["cta_rows"] >= 1
        g, y = _guarded(M, y0)
        spx.spx_spmv_csr(plan, A, dev(x), y, 1.0, 0.5)
        assert spx.spx_last_device_error() == INDEX_RANGE
        assert spx.spx_last_device_error() == 0  # read and cleared
    assert _guards_intact(g, M)
    v0 = val.copy()
    v0[bad] = 0.0
    ref, bound = oracle.spmv(M, rp, col, v0, x, 1.0, 0.5, y0)
    assert_within(y.cpu().numpy(), ref, bound, what="checked SpMV with bad columns")


def test_spmv_inconsistent_row_offsets_reported():
    """A row offset beyond nnz inside a packed group: the group's rows are not reduced (no shared-memory read past
    its products), the error is reported, the other rows are right and nothing around y changes."""
    M, K = 3000, 20000
    rp, col, val = _csr(3, M, K)
    x = synth.uniform(3, synth.T_X, K)
    with spx.checked_build():
        A = csr_to_device(M, K, rp, col, val)
        plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr)
        tasks, _ = plan.tasks()
        groups = tasks[(tasks[:, 0] & 255) == 0]
        r0, r1 = int(groups[len(groups) // 2, 1]), int(groups[len(groups) // 2, 2])
        assert r1 - r0 >= 3
        rbad = rp.copy()
        rbad[r0 + 1] = int(rp[-1]) + 100
        A.row_ptr.copy_(torch.from_numpy(rbad).cuda())
        g, y = _guarded(M, np.zeros(M, np.float32))
        spx.spx_spmv_csr(plan, A, dev(x), y, 1.0, 0.0)
        assert spx.spx_last_device_error() == INDEX_RANGE
    assert _guards_intact(g, M)
    ref, bound = oracle.spmv(M, rp, col, val, x)
    keep = np.ones(M, bool)
    keep[r0:r1] = False
    assert_within(y.cpu().numpy()[keep], ref[keep], bound[keep], what="rows outside the bad group")


@pytest.mark.parametrize("how", ["row past the group", "carry bit flipped"])
def test_spmv_corrupt_first_rows_reported(how):
    """The plan's per-thread first rows (uploaded into caller memory with the task table) corrupted for
    one segmented group: the group is not reduced, the error is reported, the other rows are right and
    nothing around y changes."""
    M, K = 3000, 20000
    rp, col, val = _csr(6, M, K)
    x = synth.uniform(6, synth.T_X, K)
    with spx.checked_build():
        A = csr_to_device(M, K, rp, col, val)
        plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, opts=dict(block_nnz=1024, lanes_div=0))
        tasks, longrows = plan.tasks()
        gidx = np.flatnonzero((tasks[:, 0] & 255) == 0)
        g = len(gidx) // 2
        r0, r1 = int(tasks[gidx[g], 1]), int(tasks[gidx[g], 2])
        assert r1 - r0 >= 3 and rp[r1] - rp[r0] > 16
        first = plan.first_rows()
        e = int(first[g, 1]) if how == "carry bit flipped" else 2 * (r1 - r0 + 3)
        e ^= 1 if how == "carry bit flipped" else 0
        table = plan.table.view(torch.int16)  # the uploaded device table, as 2-byte words
        table[8 * (len(tasks) + len(longrows)) + g * first.shape[1] + 1] = e
        gy, y = _guarded(M, np.zeros(M, np.float32))
        spx.spx_spmv_csr(plan, A, dev(x), y, 1.0, 0.0)
        assert spx.spx_last_device_error() == INDEX_RANGE
    assert _guards_intact(gy, M)
    ref, bound = oracle.spmv(M, rp, col, val, x)
    keep = np.ones(M, bool)
    keep[r0:r1] = False
    assert_within(y.cpu().numpy()[keep], ref[keep], bound[keep], what="rows outside the corrupted group")
    assert not y.cpu().numpy()[r0:r1].any()  # the group was not reduced


def test_spmm_bad_columns_and_rows_reported():
    M, K, N = 3000, 5000, 32
    d = synth.random_coo(4, M, K, 1, 40)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    B = synth.uniform(4, synth.T_B, K * N).reshape(K, N)
    C_prod = torch.zeros(M, N, device="cuda")
    A = csr_to_device(M, K, rp, col, val)
    spx.spx_spmm_csr(A, dev(B), C_prod, 1.0, 0.0)
    with spx.checked_build():
        C_chk = torch.zeros(M, N, device="cuda")
        spx.spx_spmm_csr(A, dev(B), C_chk, 1.0, 0.0)
        assert spx.spx_last_device_error() == 0
        torch.cuda.synchronize()
        assert np.array_equal(bits(C_chk), bits(C_prod))
        col_bad = col.copy()
        col_bad[[3, 700, 5000]] = [K + 3, -1, 2 ** 30]
        rbad = rp.copy()
        rbad[1500] = int(rp[-1]) + 7
        Ab = csr_to_device(M, K, rbad, col_bad, val)
        gC = torch.full(((M + 2) * N,), 777.0, device="cuda")
        C = gC[N:N + M * N].view(M, N)
        spx.spx_spmm_csr(Ab, dev(B), C, 1.0, 0.0)
        assert spx.spx_last_device_error() == INDEX_RANGE
    h = gC.cpu().numpy()
    assert np.all(h[:N] == 777.0) and np.all(h[N + M * N:] == 777.0)


def test_sell_bad_image_column_reported():
    M, K = 3000, 20000
    rp, col, val = _csr(5, M, K, lmax=3000)
    x = synth.uniform(5, synth.T_X, K)
    with spx.checked_build():
        S = spx.Sell(M, K, rp, col, val)
        y = torch.zeros(M, device="cuda")
        spx.spx_spmv_sell(S, dev(x), y, 1.0, 0.0)
        assert spx.spx_last_device_error() == 0
        ref, bound = oracle.spmv(M, rp, col, val, x)
        assert_within(y.cpu().numpy(), ref, bound)
        sp, pr, lr, sc, sv = S.arrays()
        img = S.image.cpu().numpy()
        # the column section of the uploaded image: find it by its contents
        n = min(64, sc.size)
        starts = [i for i in range(img.size - n) if img[i] == sc[0] and np.array_equal(img[i:i + n], sc[:n])]
        assert starts
        j = starts[0] + int(np.flatnonzero(sc >= 0)[0])
        img[j] = K + 55
        S.image.copy_(torch.from_numpy(img).cuda())
        g, y = _guarded(M, np.zeros(M, np.float32))
        spx.spx_spmv_sell(S, dev(x), y, 1.0, 0.0)
        assert spx.spx_last_device_error() == INDEX_RANGE
    assert _guards_intact(g, M)


def test_bsr_bad_block_column_and_offsets_reported():
    MB, KB, N = 6, 10, 256
    counts = [3, 0, 5, 2, 4, 1]
    brp = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    bcol = np.concatenate([np.sort(synth.permutation(60 + I, KB)[:c]) for I, c in enumerate(counts)]).astype(np.int32)
    nb = bcol.size
    A = synth.normal_bf16(6, synth.T_VAL, nb * 4096, 0.02).reshape(nb, 64, 64)
    B = synth.normal_bf16(6, synth.T_B, KB * 64 * N, 1.0).reshape(KB * 64, N)

    def call(brp_, bcol_):
        C = torch.zeros(MB * 64, N, device="cuda")
        spx.spx_spmm_bsr(MB * 64, KB * 64, 64, 64, dev(brp_), dev(bcol_), dev(A.reshape(-1).view(np.int16)),
                         dev(B.view(np.int16)), C)
        return C

    C_prod = call(brp, bcol)
    with spx.checked_build():
        C_chk = call(brp, bcol)
        assert spx.spx_last_device_error() == 0
        torch.cuda.synchronize()
        assert np.array_equal(bits(C_chk), bits(C_prod))
        b2 = bcol.copy()
        b2[4] = KB + 3
        call(brp, b2)
        assert spx.spx_last_device_error() == INDEX_RANGE
        r2 = brp.copy()
        r2[3] = nb + 50
        call(r2, bcol)
        assert spx.spx_last_device_error() == INDEX_RANGE
        call(brp, bcol)
        assert spx.spx_last_device_error() == 0


def test_bsr_other_shape_bad_block_column_and_offsets_reported():
    """The CUDA-core kernel of block shapes other than 64 x 64 (here 16 x 8)."""
    br, bc, MB, KB, N = 16, 8, 7, 12, 100
    counts = [2, 0, 5, 12, 1, 3, 4]
    brp = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    bcol = np.concatenate([np.sort(synth.permutation(70 + I, KB)[:c]) for I, c in enumerate(counts)]).astype(np.int32)
    nb = bcol.size
    A = synth.normal_bf16(8, synth.T_VAL, nb * br * bc, 0.5).reshape(nb, br, bc)
    B = synth.normal_bf16(8, synth.T_B, KB * bc * N, 1.0).reshape(KB * bc, N)

    def call(brp_, bcol_):
        C = torch.zeros(MB * br, N, device="cuda")
        spx.spx_spmm_bsr(MB * br, KB * bc, br, bc, dev(brp_), dev(bcol_), dev(A.reshape(-1).view(np.int16)),
                         dev(B.view(np.int16)), C)
        return C

    C_prod = call(brp, bcol)
    with spx.checked_build():
        C_chk = call(brp, bcol)
        assert spx.spx_last_device_error() == 0
        torch.cuda.synchronize()
        assert np.array_equal(bits(C_chk), bits(C_prod))
        b2 = bcol.copy()
        b2[6] = -1
        call(brp, b2)
        assert spx.spx_last_device_error() == INDEX_RANGE
        r2 = brp.copy()
        r2[2] = nb + 9
        call(r2, bcol)
        assert spx.spx_last_device_error() == INDEX_RANGE
        call(brp, bcol)
        assert spx.spx_last_device_error() == 0


def test_wcsr_bad_window_column_reported():
    M, K, N = 256, 4096, 128
    d = synth.random_coo(7, M, K, 5, 60)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], synth.to_bf16_bits(d["val"]))
    wp, wc, wv, _ = oracle.build_wcsr(M, K, rp, col, val)
    B = synth.normal_bf16(7, synth.T_B, K * N, 1.0).reshape(K, N)
    with spx.checked_build():
        C = torch.zeros(M, N, device="cuda")
        spx.spx_spmm_wcsr(M, K, dev(wp), dev(wc), dev(wv.reshape(-1).view(np.int16)), dev(B.view(np.int16)), C)
        assert spx.spx_last_device_error() == 0
        wc2 = wc.copy()
        wc2[int(np.flatnonzero(wc >= 0)[3])] = K + 9
        spx.spx_spmm_wcsr(M, K, dev(wp), dev(wc2), dev(wv.reshape(-1).view(np.int16)), dev(B.view(np.int16)), C)
        assert spx.spx_last_device_error() == INDEX_RANGE


def test_product_calls_after_the_checked_ones_are_right():
    M, K = 2000, 9000
    rp, col, val = _csr(8, M, K)
    A = csr_to_device(M, K, rp, col, val)
    plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr)
    x = synth.uniform(8, synth.T_X, K)
    y = torch.zeros(M, device="cuda")
    spx.spx_spmv_csr(plan, A, dev(x), y, 1.0, 0.0)
    assert spx.spx_last_device_error() == 0
    ref, bound = oracle.spmv(M, rp, col, val, x)
    assert_within(y.cpu().numpy(), ref, bound)
