"""Host-side logic of the C ABI (no GPU): the library loads and exports every
symbol of include/spx.h; the host format builders, statistics and dispatch
plan match the oracle bit-exactly; arguments are rejected with the documented
status codes."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import first_rows_expected


@pytest.mark.parametrize("path", [spx.LIB_PATH, spx.LIB_CHECK_PATH])
def test_exports_every_header_symbol(path):
    """The product library and its bounds-checked twin both export every call the header declares."""
    names = spx.header_symbols()
    assert len(names) >= 22
    lib = ctypes.CDLL(path)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


@pytest.mark.parametrize("path", [spx.LIB_PATH, spx.LIB_CHECK_PATH])
def test_exports_only_the_c_abi(path):
    """Each library's dynamic symbol table defines the spx_* C calls and nothing else: C++ statics
    (and their initialisation guards) of one library must never bind to the other's when both are
    loaded in one process."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    names = [line.split()[-1] for line in out.splitlines() if line.strip()]
    others = [n for n in names if not n.startswith("spx_")]
    assert not others, others[:10]
    assert set(spx.header_symbols()) <= set(names)


def test_status_strings():
    lib = spx._lib()
    for code, name in spx.STATUS.items():
        assert lib.spx_status_string(code).decode().startswith(name)


MATS = [(1, 1, 0, 1), (40, 30, 0, 12), (300, 7, 0, 7), (7, 300, 50, 120), (1000, 1000, 0, 40), (64, 64, 64, 64),
        (3, 5, 0, 0)]


def _mat(seed, M, K, lmin, lmax):
    return synth.random_coo(seed, M, K, lmin, lmax)


@pytest.mark.parametrize("M,K,lmin,lmax", MATS)
def test_build_csr_matches_oracle(M, K, lmin, lmax):
    d = _mat(3, M, K, lmin, lmax)
    perm = synth.permutation(9, d["row"].size)
    args = (d["row"][perm], d["col"][perm], d["val"][perm])
    got = spx.spx_build_csr(M, K, *args)
    want = oracle.build_csr(M, K, *args)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


def test_build_csr_keeps_duplicates_in_input_order():
    row = np.array([1, 0, 1, 1, 0], np.int32)
    col = np.array([2, 0, 2, 0, 0], np.int32)
    val = np.arange(5, dtype=np.float32)
    got = spx.spx_build_csr(2, 3, row, col, val)
    want = oracle.build_csr(2, 3, row, col, val)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


@pytest.mark.parametrize("vdtype", [np.float32, np.uint16, np.float64])
def test_build_csr_value_widths(vdtype):
    d = _mat(4, 200, 90, 0, 20)
    perm = synth.permutation(2, d["row"].size)
    val = (np.arange(d["row"].size) * 7 % 65000).astype(vdtype)
    got = spx.spx_build_csr(200, 90, d["row"][perm], d["col"][perm], val[perm])
    want = oracle.build_csr(200, 90, d["row"][perm], d["col"][perm], val[perm])
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


@pytest.mark.parametrize("M,K,lmin,lmax", MATS)
def test_transpose_matches_oracle(M, K, lmin, lmax):
    d = _mat(5, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    got = spx.spx_transpose_csr(M, K, rp, col, val)
    want = oracle.transpose(M, K, rp, col, val)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


@pytest.mark.parametrize("M,K,lmin,lmax", MATS)
@pytest.mark.parametrize("br,bc", [(1, 1), (2, 2), (4, 3), (64, 64)])
def test_build_bsr_matches_oracle(M, K, lmin, lmax, br, bc):
    d = _mat(6, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    g = spx.spx_build_bsr(M, K, rp, col, val, br, bc)
    w = oracle.build_bsr(M, K, rp, col, val, br, bc)
    for a, b in zip(g[:3], w[:3]):
        assert np.array_equal(a, b)
    assert g[3] == w[3]


def test_build_bsr_duplicate_rejected():
    rp = np.array([0, 2], np.int32)
    with pytest.raises(spx.SpxError) as e:
        spx.spx_build_bsr(1, 4, rp, np.array([1, 1], np.int32), np.ones(2, np.float32), 2, 2)
    assert e.value.name == "SPX_ERR_DUPLICATE"


@pytest.mark.parametrize("seed", range(5))
def test_row_stats_bit_exact(seed):
    L, _ = synth.lengths_zipf(seed, 5000 + 17 * seed, 2.1, 4000, 9.0)
    L[:: 7 + seed] = 0
    rp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    assert spx.spx_row_stats(L.size, rp) == oracle.row_stats(L.size, rp)


PLAN_OPTS = [
    None,
    dict(block_nnz=16, block_rows=3, pack_max=8, cta_max=100, seg_nnz=40, lanes_div=2),
    dict(block_nnz=1024, block_rows=256, pack_max=1024, cta_max=1024, seg_nnz=1024, lanes_div=1),
    dict(block_nnz=4096, block_rows=512, pack_max=64, cta_max=20000, seg_nnz=3000, lanes_div=8),
    dict(block_nnz=1000, block_rows=100, pack_max=999, cta_max=5000, seg_nnz=700, lanes_div=0),
    dict(block_nnz=512, block_rows=1024, pack_max=512, cta_max=4096, seg_nnz=2048, lanes_div=0),
    dict(block_nnz=4096, block_rows=300, pack_max=200, cta_max=8192, seg_nnz=4096, lanes_div=0),
    dict(block_nnz=16, block_rows=1024, pack_max=16, cta_max=64, seg_nnz=64, lanes_div=0),
]


@pytest.mark.parametrize("opts", PLAN_OPTS)
@pytest.mark.parametrize("seed", range(3))
def test_plan_matches_oracle(opts, seed):
    L, _ = synth.lengths_zipf(seed, 20000, 2.1, 60000, 12.0)
    L[::31] = 0
    rp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    if opts is None:
        full = oracle.plan_opts_auto(L.size, rp)
    else:
        full = spx.spx_plan_opts_default()
        full.update(opts)
    p = spx.spx_plan_csr(L.size, 70000, int(rp[-1]), rp, opts=opts, upload=False)
    tasks, longrows = p.tasks()
    w = oracle.plan_spmv(L.size, rp, **full)
    assert np.array_equal(tasks, w["tasks"]) and np.array_equal(longrows, w["longrows"])
    for k, v in w["counts"].items():
        assert p.info[k] == v, k
    assert p.stats == oracle.row_stats(L.size, rp)
    groups = int((tasks[:, 0] & 255).tolist().count(0))
    first = 2 * groups * (full["block_nnz"] // 8 if full["block_nnz"] in (512, 1024, 2048, 4096) else 256)
    assert p.info["table_bytes"] == 16 * (tasks.shape[0] + longrows.shape[0]) + (first if full["lanes_div"] == 0 else 0)
    assert p.info["scratch_bytes"] == 4 * w["counts"]["slots"]
    if full["lanes_div"] == 0:
        assert np.array_equal(p.first_rows(), first_rows_expected(rp, tasks, full["block_nnz"]))
    else:
        assert p.first_rows().size == 0


@pytest.mark.parametrize("B", [512, 1000, 4096])
def test_plan_first_rows_with_runs_of_empty_rows(B):
    """Groups of up to 1024 rows, most of them empty: each thread's first row is the
    last row starting at or before its first product, never an empty row before it."""
    rng = np.random.default_rng(B)
    L = np.where(rng.random(50_000) < 0.05, rng.integers(1, 40, 50_000), 0).astype(np.int32)
    L[:700] = 0
    rp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    opts = dict(block_nnz=B, block_rows=1024, pack_max=64, cta_max=4096, seg_nnz=1024, lanes_div=0)
    p = spx.spx_plan_csr(L.size, 100, int(rp[-1]), rp, opts=opts, upload=False)
    tasks, _ = p.tasks()
    got = p.first_rows()
    assert got.shape[0] == p.info["segmented_groups"] > 0
    assert np.array_equal(got, first_rows_expected(rp, tasks, B))
    assert got.max() > 1000  # rows deep inside a group of mostly empty rows


def test_plan_default_options_documented():
    o = spx.spx_plan_opts_default()
    assert o == dict(block_nnz=2048, block_rows=256, pack_max=512, cta_max=8192, seg_nnz=4096, lanes_div=16)


@pytest.mark.parametrize("kind", ["skewed", "uniform", "empty", "constant"])
def test_plan_auto_options_match_oracle(kind):
    if kind == "skewed":
        L, _ = synth.lengths_zipf(3, 50000, 2.1, 100000, 16.0)
    elif kind == "uniform":
        L = synth.lengths_uniform(3, 50000, 1, 16)
    elif kind == "empty":
        L = np.zeros(100, np.int32)
    else:
        L = np.full(1000, 7, np.int32)
    rp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    want = oracle.plan_opts_auto(L.size, rp)
    lib = spx._lib()
    st = spx.RowStats()
    assert lib.spx_row_stats(L.size, spx._ptr(rp), 0, ctypes.byref(st)) == 0
    o = spx.PlanOpts()
    assert lib.spx_plan_opts_auto(ctypes.byref(st), ctypes.byref(o)) == 0
    assert {f: getattr(o, f) for f, _ in spx.PlanOpts._fields_} == want
    assert want["lanes_div"] == (0 if kind == "skewed" else 16)


def test_plan_rejects_bad_rows_and_options():
    lib = spx._lib()
    h = ctypes.c_void_p()
    bad = np.array([0, 3, 2, 4], np.int32)  # not monotone
    assert lib.spx_plan_csr(3, 5, 4, spx._ptr(bad), 0, None, ctypes.byref(h)) == -3
    rp = np.array([0, 1, 2], np.int32)
    assert lib.spx_plan_csr(2, 5, 3, spx._ptr(rp), 0, None, ctypes.byref(h)) == -1  # row_ptr[M] != nnz
    o = spx.PlanOpts(block_nnz=16, block_rows=4, pack_max=32, cta_max=64, seg_nnz=8, lanes_div=1)  # P > B
    assert lib.spx_plan_csr(2, 5, 2, spx._ptr(rp), 0, ctypes.byref(o), ctypes.byref(h)) == -1
    assert lib.spx_plan_csr(2, 5, 2 ** 31, spx._ptr(rp), 0, None, ctypes.byref(h)) == -2  # int32 overflow


def test_int32_overflow_rejected_not_truncated():
    lib = spx._lib()
    one = np.zeros(4, np.int32)
    assert lib.spx_build_csr(4, 4, 2 ** 31, spx._ptr(one), spx._ptr(one), spx._ptr(one), 4, spx._ptr(one),
                             spx._ptr(one), spx._ptr(one), 0, None) == -2
    assert lib.spx_transpose_csr(4, 4, 2 ** 32 + 1, spx._ptr(one), spx._ptr(one), spx._ptr(one), 4,
                                 spx._ptr(one), spx._ptr(one), spx._ptr(one), 0, None) == -2
    assert lib.spx_spmm_csr(4, 4, 2 ** 31, spx._ptr(one), spx._ptr(one), spx._ptr(one), 1, spx._ptr(one), 1,
                            1.0, 0.0, spx._ptr(one), 1, None) == -2


def test_index_range_rejected():
    with pytest.raises(spx.SpxError) as e:
        spx.spx_build_csr(2, 2, np.array([0, 2], np.int32), np.array([0, 0], np.int32), np.ones(2, np.float32))
    assert e.value.name == "SPX_ERR_INDEX_RANGE"
    rp = np.array([0, 1, 2], np.int32)
    with pytest.raises(spx.SpxError) as e:
        spx.spx_transpose_csr(2, 2, rp, np.array([0, 5], np.int32), np.ones(2, np.float32))
    assert e.value.name == "SPX_ERR_INDEX_RANGE"


def test_check_csr():
    rp = np.array([0, 2, 3], np.int32)
    assert spx.spx_check_csr(2, 4, rp, np.array([0, 3, 1], np.int32)) == 0
    assert spx.spx_check_csr(2, 4, rp, np.array([3, 0, 1], np.int32)) == -3
    assert spx.spx_check_csr(2, 4, rp, np.array([3, 0, 1], np.int32), strict=False) == 0
    assert spx.spx_check_csr(2, 4, rp, np.array([1, 1, 1], np.int32)) == -4
    assert spx.spx_check_csr(2, 4, rp, np.array([0, 4, 1], np.int32)) == -2
    assert spx.spx_check_csr(2, 4, np.array([0, 3, 2], np.int32), np.array([0, 1, 2], np.int32)) in (-1, -3)


def test_compute_calls_reject_bad_plans_without_launching():
    lib = spx._lib()
    before = spx.launch_count()
    assert lib.spx_spmv_csr(None, 1, 1, 0, None, None, None, 1.0, None, 0.0, None, None, 0, None) == -1
    rp = np.array([0, 1], np.int32)
    p = spx.spx_plan_csr(1, 1, 1, rp, upload=False)
    # a plan that was never uploaded
    assert lib.spx_spmv_csr(p.handle, 1, 1, 1, None, None, None, 1.0, None, 0.0, None, None, 0, None) == -10
    # sizes that do not match the plan
    assert lib.spx_spmv_csr(p.handle, 2, 1, 1, None, None, None, 1.0, None, 0.0, None, None, 0, None) == -1
    assert spx.launch_count() == before


def test_spmm_variant_rule():
    lib = spx._lib()
    a16 = ctypes.c_void_p(1 << 20)
    for N, want in [(1, 0), (8, 0), (12, 1), (32, 1), (128, 1), (132, 2), (1024, 2), (9, 3), (130, 3)]:
        assert lib.spx_spmm_csr_variant(N, a16, N, a16, N) == want, N
    assert lib.spx_spmm_csr_variant(32, ctypes.c_void_p((1 << 20) + 4), 32, a16, 32) == 3  # misaligned B
    assert lib.spx_spmm_csr_variant(32, a16, 34, a16, 32) == 3  # ldb not a multiple of 4


def test_coo_spmv_rejects_bad_arguments_without_launching():
    lib = spx._lib()
    before = spx.launch_count()
    a = ctypes.c_void_p(1 << 20)
    big = ctypes.c_void_p(1 << 30)
    # scratch: two floats per 2048 entries
    assert spx.spx_spmv_coo_scratch_bytes(0) == 0
    assert spx.spx_spmv_coo_scratch_bytes(1) == 8
    assert spx.spx_spmv_coo_scratch_bytes(2048) == 8
    assert spx.spx_spmv_coo_scratch_bytes(2049) == 16
    assert lib.spx_spmv_coo(-1, 4, 1, a, a, a, 1.0, a, 0.0, big, a, 8, None) == -1
    assert lib.spx_spmv_coo(4, 4, 1 << 31, a, a, a, 1.0, a, 0.0, big, a, 1 << 22, None) == -2
    assert lib.spx_spmv_coo(4, 4, 1, None, a, a, 1.0, a, 0.0, big, a, 8, None) == -1
    assert lib.spx_spmv_coo(4, 4, 3000, a, a, a, 1.0, a, 0.0, big, a, 8, None) == -1      # scratch too small
    assert lib.spx_spmv_coo(4, 4, 1, a, a, a, 1.0, a, 0.0, a, big, 8, None) == -1          # x and y overlap
    assert lib.spx_spmv_coo(4, 4, 1, ctypes.c_void_p((1 << 20) + 2), a, a, 1.0, a, 0.0, big, a, 8, None) == -8
    assert lib.spx_spmv_coo(0, 4, 1, a, a, a, 1.0, a, 0.0, big, a, 8, None) == -2          # entries but no rows
    assert lib.spx_spmv_coo(0, 4, 0, None, None, None, 1.0, None, 0.0, big, None, 0, None) == 0
    assert spx.launch_count() == before


def test_autotune_rejects_bad_arguments_without_launching():
    lib = spx._lib()
    before = spx.launch_count()
    rp = np.array([0, 1, 2], np.int32)
    a = ctypes.c_void_p(1 << 20)
    best = spx.PlanOpts()
    P = spx._ptr(rp)
    assert lib.spx_plan_autotune(2, 2, 2, None, a, a, a, a, a, None, 0, 3, None, ctypes.byref(best), None, None) == -1
    assert lib.spx_plan_autotune(2, 2, 2, P, a, a, a, a, a, None, 0, 0, None, ctypes.byref(best), None, None) == -1
    assert lib.spx_plan_autotune(2, 2, 2, P, a, a, a, a, a, None, 0, 3, None, None, None, None) == -1
    assert lib.spx_plan_autotune(2, 2, 3, P, a, a, a, a, a, None, 0, 3, None, ctypes.byref(best), None, None) == -1
    cand = (spx.PlanOpts * 1)()
    assert lib.spx_plan_autotune(2, 2, 2, P, a, a, a, a, a, cand, 0, 3, None, ctypes.byref(best), None, None) == -1
    assert lib.spx_plan_autotune(2, 2, 2, P, a, a, a, a, a, cand, 17, 3, None, ctypes.byref(best), None, None) == -1
    assert lib.spx_plan_autotune_forget() == 0
    assert spx.launch_count() == before


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 0, 1), (40, 30, 0, 9), (0, 3, 0, 1), (700, 900, 0, 300)])
@pytest.mark.parametrize("opts", [None, dict(sigma=32, piece=5), dict(sigma=96, piece=64), dict(sigma=1 << 20)])
def test_sell_matches_oracle(M, K, lmin, lmax, opts):
    d = synth.random_coo(33, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    S = spx.Sell(M, K, rp, col, val, opts=opts, upload=False)
    o = dict(sigma=1024, piece=64)
    o.update(opts or {})
    assert S.opts == o
    want = oracle.build_sell(M, rp, col, val, **o)
    got = S.arrays()
    for w, g in zip(want, got):
        assert np.array_equal(w, g)
    assert S.info["slices"] == want[0].size - 1 and S.info["padded"] == want[3].size
    assert S.info["scratch_bytes"] == 4 * int(want[2][:, 2].sum()) if want[2].size else S.info["scratch_bytes"] == 0


def test_sell_rejects_bad_input_and_unuploaded_use():
    lib = spx._lib()
    rp = np.array([0, 1, 2], np.int32)
    for o in (dict(sigma=48), dict(sigma=16), dict(piece=0)):
        with pytest.raises(spx.SpxError):
            spx.Sell(2, 2, rp, np.array([0, 1], np.int32), np.ones(2, np.float32), opts=o, upload=False)
    with pytest.raises(spx.SpxError):  # column out of range
        spx.Sell(2, 2, rp, np.array([0, 2], np.int32), np.ones(2, np.float32), upload=False)
    with pytest.raises(spx.SpxError):  # row_ptr decreasing
        spx.Sell(2, 2, np.array([0, 2, 1], np.int32), np.array([0, 1], np.int32), np.ones(2, np.float32),
                 upload=False)
    S = spx.Sell(2, 2, rp, np.array([0, 1], np.int32), np.ones(2, np.float32), upload=False)
    before = spx.launch_count()
    a = ctypes.c_void_p(1 << 20)
    assert lib.spx_spmv_sell(S.handle, 2, 2, 1.0, a, 0.0, ctypes.c_void_p(1 << 22), None, 0, None) == -10
    assert lib.spx_spmv_sell(S.handle, 3, 2, 1.0, a, 0.0, ctypes.c_void_p(1 << 22), None, 0, None) == -1
    assert spx.launch_count() == before


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 0, 1), (64, 300, 0, 90), (130, 200, 0, 40), (0, 5, 0, 1),
                                          (257, 4000, 0, 200)])
@pytest.mark.parametrize("vdtype", [np.float32, np.uint16])
def test_build_wcsr_matches_oracle(M, K, lmin, lmax, vdtype):
    d = synth.random_coo(62, M, K, lmin, lmax)
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    v = val if vdtype is np.float32 else synth.to_bf16_bits(val)
    want = oracle.build_wcsr(M, K, rp, col, v)
    got = spx.spx_build_wcsr(M, K, rp, col, v)
    for w, g in zip(want[:3], got[:3]):
        assert np.array_equal(w, g)
    assert want[3] == got[3]


def test_build_wcsr_errors():
    rp = np.array([0, 2, 3], np.int32)
    with pytest.raises(spx.SpxError):   # duplicate (row, col)
        spx.spx_build_wcsr(2, 4, rp, np.array([1, 1, 0], np.int32), np.ones(3, np.float32))
    with pytest.raises(spx.SpxError):   # column out of range
        spx.spx_build_wcsr(2, 4, rp, np.array([1, 4, 0], np.int32), np.ones(3, np.float32))
    with pytest.raises(spx.SpxError):   # row_ptr decreasing
        spx.spx_build_wcsr(2, 4, np.array([0, 3, 2], np.int32), np.array([1, 2, 0], np.int32), np.ones(3, np.float32))


def test_spmm_wcsr_rejects_unsupported_without_launching():
    lib = spx._lib()
    before = spx.launch_count()
    a = ctypes.c_void_p(1 << 20)
    assert lib.spx_spmm_wcsr(64, 64, 1, a, a, a, 100, a, 128, 1.0, 0.0, a, 128, None) == -7   # N % 8
    assert lib.spx_spmm_wcsr(64, 64, 1, a, a, a, 128, a, 132, 1.0, 0.0, a, 128, None) == -8   # ldb % 8
    assert lib.spx_spmm_wcsr(64, 64, 1, a, a, a, 128, a, 64, 1.0, 0.0, a, 128, None) == -1    # ldb < N
    assert lib.spx_spmm_wcsr(64, 64, -1, a, a, a, 128, a, 128, 1.0, 0.0, a, 128, None) == -1
    assert spx.launch_count() == before


def test_gather_probe_rejects_bad_arguments_without_launching():
    lib = spx._lib()
    before = spx.launch_count()
    a = ctypes.c_void_p(1 << 20)
    assert lib.spx_gather_probe(-1, a, a, a, 4, a, 8, None) == -1
    assert lib.spx_gather_probe(10, None, a, a, 4, a, 8, None) == -1
    assert lib.spx_gather_probe(10, a, a, a, 4, a, 0, None) == -1
    assert lib.spx_gather_probe(10, a, a, a, 4, None, 8, None) == -1
    assert spx.launch_count() == before


def test_hostio_rejects_bad_arguments_without_launching():
    lib = spx._lib()
    rp = np.array([0, 1, 2], np.int32)
    p = spx.spx_plan_csr(2, 3, 2, rp, upload=False)
    a = ctypes.c_void_p(1 << 20)
    w = ctypes.c_void_p(1 << 24)
    need = lib.spx_spmv_csr_hostio_work_bytes(2, 3)
    assert need == 2 * (256 + 256)
    before = spx.launch_count()
    assert lib.spx_spmv_csr_hostio(p.handle, 2, 3, 2, a, a, a, 1.0, a, 2, 0.0, a, 2, 1, w, need, None, 0, None) == -1
    assert lib.spx_spmv_csr_hostio(p.handle, 2, 3, 2, a, a, a, 1.0, a, 3, 0.0, a, 1, 1, w, need, None, 0, None) == -1
    assert lib.spx_spmv_csr_hostio(p.handle, 2, 3, 2, a, a, a, 1.0, a, 3, 0.0, a, 2, 1, w, need - 4, None, 0,
                                   None) == -1
    assert lib.spx_spmv_csr_hostio(p.handle, 2, 3, 2, a, a, a, 1.0, a, 3, 0.0, a, 2, 1,
                                   ctypes.c_void_p((1 << 24) + 16), need, None, 0, None) == -8
    assert lib.spx_spmv_csr_hostio(p.handle, 2, 3, 2, a, a, a, 1.0, a, 0, 0.0, a, 2, 1, w, need, None, 0,
                                   None) == -10  # x broadcast is fine; the plan was never uploaded
    assert lib.spx_spmv_csr_hostio(p.handle, 2, 3, 2, a, a, a, 1.0, a, 3, 0.0, a, 2, 0, w, need, None, 0, None) == 0
    assert spx.launch_count() == before


def test_binding_rejects_strided_views():
    """The binding hands raw addresses to the library, so a view whose elements
    are not dense (a strided slice, a transpose) is refused instead of misread."""
    row = np.array([0, 1, 1, 2, 0, 2], np.int32)
    col = np.array([0, 0, 1, 1, 2, 2], np.int32)
    val = np.ones(12, np.float32)
    with pytest.raises(ValueError):
        spx.spx_build_csr(3, 3, row, col, val[::2])
    with pytest.raises(ValueError):
        spx.spx_build_csr(3, 3, row, col, np.ones((2, 3), np.float32).T)
    rp, c, v = spx.spx_build_csr(3, 3, row, col, np.ascontiguousarray(val[::2]))  # a dense copy is fine
    assert rp.tolist() == [0, 2, 4, 6]


def test_wcsr_plan_task_split():
    """Windows with more than max_chunks chunks are cut into balanced pieces of consecutive
    chunks with consecutive partial slots; the others stay whole (slot -1).  Tasks are listed
    longest first, ties in window and piece order."""
    wp = np.array([0, 3, 3, 20, 21, 33], np.int32)  # chunks per window: 3, 0, 17, 1, 12
    P = spx.WcsrPlan(5 * 64 - 10, 33, wp, max_chunks=5, upload=False)
    tasks, splits = P.tasks()
    assert P.info["split_windows"] == 2 and P.info["slots"] == 4 + 3
    # window 2: 17 chunks -> 4 pieces of 5, 4, 4, 4; window 4: 12 chunks -> 3 pieces of 4
    assert tasks.tolist() == [[2, 3, 5, 0], [2, 8, 4, 1], [2, 12, 4, 2], [2, 16, 4, 3],
                              [4, 21, 4, 4], [4, 25, 4, 5], [4, 29, 4, 6],
                              [0, 0, 3, -1], [3, 20, 1, -1], [1, 3, 0, -1]]
    assert splits.tolist() == [[2, 0, 4, 0], [4, 4, 3, 0]]
    assert P.info["table_bytes"] == 4 * 4 * (10 + 2)
    whole = spx.WcsrPlan(5 * 64, 33, wp, max_chunks=0, upload=False)  # default 16: only window 2 splits
    assert whole.info["split_windows"] == 1 and whole.info["max_chunks"] == 16


def test_wcsr_plan_errors():
    for wp, nch, code in [([1, 2], 2, -1), ([0, 2], 3, -1), ([0, 3, 2], 2, -3)]:
        with pytest.raises(spx.SpxError) as e:
            spx.WcsrPlan(64 * (len(wp) - 1), nch, np.array(wp, np.int32), upload=False)
        assert e.value.code == code


def _fingerprint(rp):
    """The documented plan fingerprint, restated: sum of SplitMix64 outputs of 2^32*i + row_ptr[i]."""
    mask = (1 << 64) - 1
    f = 0
    for i, v in enumerate(np.asarray(rp, np.int64).tolist()):
        z = (((i << 32) | (v & 0xFFFFFFFF)) + 0x9E3779B97F4A7C15) & mask
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        f = (f + (z ^ (z >> 31))) & mask
    return f


def test_plan_fingerprint_and_validate():
    """The fingerprint of row_ptr = [0] is SplitMix64's first output from seed 0
    (0xE220A8397B1DCDAF, its published first value); larger row_ptrs follow the
    documented sum.  validate accepts the plan's own row_ptr and rejects a row_ptr
    with the same M, K, nnz but one nonzero moved to the next row, and other sizes."""
    p0 = spx.spx_plan_csr(0, 7, 0, np.zeros(1, np.int32), upload=False)
    assert p0.fingerprint == 0xE220A8397B1DCDAF
    L, _ = synth.lengths_zipf(81, 5000, 2.1, 3000, 12.0)
    rp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    nnz = int(rp[-1])
    p = spx.spx_plan_csr(5000, 70000, nnz, rp, upload=False)
    assert p.fingerprint == _fingerprint(rp)
    assert p.validate(rp) == 0
    moved = rp.copy()
    r = int(np.flatnonzero(L > 0)[7])
    moved[r + 1] -= 1  # the last entry of row r now belongs to row r + 1
    assert moved[r + 1] >= moved[r]
    assert p.validate(moved) == -1
    lib = spx._lib()
    assert lib.spx_plan_validate(p.handle, 5000, 70001, nnz, spx._ptr(rp), 0, None) == -1  # K differs
    assert lib.spx_plan_validate(p.handle, 5000, 70000, nnz, None, 0, None) == -1
    assert lib.spx_plan_validate(p.handle, 5000, 70000, nnz, spx._ptr(rp), 7, None) == -1  # bad location


def test_wait_probe_rejects_limits_out_of_range_without_launching():
    lib = spx._lib()
    before = spx.launch_count()
    assert lib.spx_wait_probe(-1, None) == -1
    assert lib.spx_wait_probe(3_000_000_000, None) == -1
    assert spx.launch_count() == before
