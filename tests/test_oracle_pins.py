"""Pins of the oracle against things other than itself.

The printed worked example (tests/golden/worked_example_5x5.json), values
derived from it by hand, dense brute force with small-integer values (where
fp64 sums are exact, so any dropped term, wrong index or transposed operand
shows), scipy's own sparse conversions, round trips and closed forms.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden", "worked_example_5x5.json")


@pytest.fixture(scope="module")
def ex():
    g = json.load(open(GOLD))
    v = g["values_used"]
    p = g["printed"]
    val = np.array([v[s] for s in p["coo_val"]], np.float32)
    return g, v, val


def _vals(names, v):
    return [v[s] if isinstance(s, str) else float(s) for s in names]


# ------------------------------------------------------------ worked example

def test_worked_example_coo_to_csr(ex):
    g, v, val = ex
    p = g["printed"]
    rp, col, vo = oracle.build_csr(5, 5, p["coo_row"], p["coo_col"], val)
    assert rp.tolist() == p["csr_row_ptr"]
    assert col.tolist() == p["csr_col"]
    assert vo.tolist() == _vals(p["csr_val"], v)


def test_worked_example_coo_any_order(ex):
    """COO may come in any order ([Formats] §2); the CSR is the same."""
    g, v, val = ex
    p = g["printed"]
    for seed in range(6):
        perm = synth.permutation(seed, 8)
        rp, col, vo = oracle.build_csr(5, 5, np.array(p["coo_row"])[perm], np.array(p["coo_col"])[perm], val[perm])
        assert rp.tolist() == p["csr_row_ptr"]
        assert col.tolist() == p["csr_col"]
        assert vo.tolist() == _vals(p["csr_val"], v)


def test_worked_example_transpose(ex):
    g, v, val = ex
    p, d = g["printed"], g["derived_by_hand"]
    trp, tc, tv = oracle.transpose(5, 5, p["csr_row_ptr"], p["csr_col"], val)
    assert trp.tolist() == d["csr_transpose_row_ptr"]
    assert tc.tolist() == d["csr_transpose_col"]
    assert tv.tolist() == _vals(d["csr_transpose_val"], v)


def test_worked_example_bsr(ex):
    g, v, val = ex
    p, d = g["printed"], g["derived_by_hand"]
    brp, bcol, bval, fill = oracle.build_bsr(5, 5, p["csr_row_ptr"], p["csr_col"], val, 2, 2)
    assert brp.tolist() == d["bsr_2x2_row_ptr"]
    assert bcol.tolist() == d["bsr_2x2_col"]
    want = [_vals(b, v) for b in d["bsr_2x2_val_rowmajor"]]
    assert bval.reshape(-1, 4).tolist() == want
    assert fill == 8 / 24


def test_worked_example_stats(ex):
    g, v, val = ex
    p, d = g["printed"], g["derived_by_hand"]
    st = oracle.row_stats(5, p["csr_row_ptr"])
    for k, want in d["stats"].items():
        assert st[k] == pytest.approx(want, rel=0, abs=1e-15), k
    assert st["mean"] == 1.6 and st["var"] == 16 / 25


def test_worked_example_spmv(ex):
    g, v, val = ex
    p, d = g["printed"], g["derived_by_hand"]
    ref, bound = oracle.spmv(5, p["csr_row_ptr"], p["csr_col"], val, np.ones(5, np.float32))
    assert ref.tolist() == d["y_for_x_all_ones"]
    assert bound.tolist() == d["y_for_x_all_ones"]  # all values positive
    # A e_j is column j of the matrix written out in the page's entry list
    dense = np.zeros((5, 5))
    for r, c, s in zip(p["coo_row"], p["coo_col"], p["coo_val"]):
        dense[r, c] = v[s]
    for j in range(5):
        e = np.zeros(5, np.float32)
        e[j] = 1
        ref, _ = oracle.spmv(5, p["csr_row_ptr"], p["csr_col"], val, e)
        assert ref.tolist() == dense[:, j].tolist()


def test_worked_example_coo_spmv(ex):
    """The page's triplet list, multiplied as triplets, gives the row sums."""
    g, v, val = ex
    p, d = g["printed"], g["derived_by_hand"]
    ref, _ = oracle.spmv_coo(5, 5, p["coo_row"], p["coo_col"], val, np.ones(5, np.float32))
    assert ref.tolist() == d["y_for_x_all_ones"]


def test_worked_example_sell(ex):
    """SELL-C-sigma of the printed matrix (sigma 32, pieces of 2), worked out by hand."""
    g, v, val = ex
    p, d = g["printed"], g["derived_by_hand"]["sell_sigma32_piece2"]
    sp, pr, lr, sc, sv = oracle.build_sell(5, p["csr_row_ptr"], p["csr_col"], val, sigma=32, piece=2)
    assert sp.tolist() == d["slice_ptr"]
    assert pr[:6].tolist() == d["prow_used"] and np.all(pr[6:] == np.iinfo(np.int32).min)
    assert lr.tolist() == d["longrows"]
    assert sc[:6].tolist() == d["scol_j0_used"] and sc[32:38].tolist() == d["scol_j1_used"]
    assert sv[:6].tolist() == _vals(d["sval_j0_used"], v) and sv[32:38].tolist() == _vals(d["sval_j1_used"], v)
    assert np.all(sc[6:32] == -1) and np.all(sc[38:] == -1) and not sv[6:32].any() and not sv[38:].any()


def sell_rows(M, sp, pr, lr, sc, sv):
    """Each row's (col, val) entries read back out of the SELL arrays: whole
    rows from their lane, long rows by concatenating their pieces in slot order."""
    piece_of = {}
    rows = {i: ([], []) for i in range(M)}
    for t, r in enumerate(pr):
        if r == np.iinfo(np.int32).min:
            continue
        s, lane = divmod(t, 32)
        L = (sp[s + 1] - sp[s]) // 32
        idx = sp[s] + 32 * np.arange(L) + lane
        keep = sc[idx] >= 0
        ent = (sc[idx][keep].tolist(), sv[idx][keep].tolist())
        if r >= 0:
            rows[r] = ent
        else:
            piece_of[-1 - r] = ent
    for row, first, n, _ in lr:
        cs, vs = [], []
        for k in range(n):
            cs += piece_of[first + k][0]
            vs += piece_of[first + k][1]
        rows[row] = (cs, vs)
    return rows


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 0, 1), (7, 5, 0, 5), (33, 64, 0, 9), (50, 50, 0, 0), (0, 4, 0, 2),
                                          (300, 500, 0, 120)])
@pytest.mark.parametrize("sigma,piece", [(32, 1), (32, 7), (64, 16), (256, 256)])
def test_sell_round_trip_and_order(M, K, lmin, lmax, sigma, piece):
    """Reading the rows back out of SELL gives the CSR exactly; windows are
    sorted longest first, equal lengths in listing order; slices are as wide
    as their longest pseudo-row; padding is (-1, 0)."""
    d = synth.random_coo(31, M, K, lmin, lmax, values="int")
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    sp, pr, lr, sc, sv = oracle.build_sell(M, rp, col, val, sigma=sigma, piece=piece)
    rows = sell_rows(M, sp, pr, lr, sc, sv)
    for i in range(M):
        assert rows[i][0] == col[rp[i]:rp[i + 1]].tolist()
        assert rows[i][1] == val[rp[i]:rp[i + 1]].tolist()
    # listing: (row, piece index, length) in row order
    listing = []
    for i in range(M):
        l = int(rp[i + 1] - rp[i])
        if l <= piece:
            listing.append((i, 0, l))
        else:
            listing += [(i, k, min(piece, l - k * piece)) for k in range(-(-l // piece))]
    got = []
    for t, r in enumerate(pr[:len(listing)]):
        s, lane = divmod(t, 32)
        L = (sp[s + 1] - sp[s]) // 32
        n = int((sc[sp[s] + 32 * np.arange(L) + lane] >= 0).sum())
        got.append(n)
    for w0 in range(0, len(listing), sigma):
        win = listing[w0:w0 + sigma]
        want = sorted(range(len(win)), key=lambda k: (-win[k][2], k))
        assert got[w0:w0 + len(win)] == [win[k][2] for k in want]
    for s in range(sp.size - 1):
        lens = got[32 * s:32 * s + 32]
        assert sp[s + 1] - sp[s] == 32 * (max(lens) if lens else 0)
    assert np.all(sv[sc < 0] == 0)
    assert lr.shape[0] == sum(1 for i in range(M) if rp[i + 1] - rp[i] > piece)


def test_worked_example_wcsr(ex):
    g, v, val = ex
    p, d = g["printed"], g["derived_by_hand"]["wcsr_window64"]
    wp, wc, wv, fill = oracle.build_wcsr(5, 5, p["csr_row_ptr"], p["csr_col"], val)
    assert wp.tolist() == d["win_ptr"]
    assert wc[:5].tolist() == d["win_col_used"] and np.all(wc[5:] == -1)
    want = np.zeros((64, 64))
    want[:5, :5] = [_vals(r, v) for r in d["chunk_top_left_5x5"]]
    assert np.array_equal(wv[0], want)
    assert fill == 8 / 4096


@pytest.mark.parametrize("M,K,lmin,lmax", [(1, 1, 0, 1), (7, 5, 0, 5), (64, 300, 0, 90), (130, 200, 0, 40),
                                          (200, 1000, 0, 70), (50, 50, 0, 0)])
def test_wcsr_against_dense(M, K, lmin, lmax):
    """Expanding WCSR back to dense gives the matrix; each window's columns are
    exactly the sorted set of columns its rows use, padded with -1 to whole
    chunks of 64; the fill ratio is nnz over stored slots."""
    d = synth.random_coo(61, M, K, lmin, lmax, values="int")
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    A = _dense(M, K, d["row"], d["col"], d["val"])
    wp, wc, wv, fill = oracle.build_wcsr(M, K, rp, col, val)
    W = -(-M // 64)
    assert wp.size == W + 1
    D = np.zeros((W * 64, K))
    for w in range(W):
        used = sorted(set(col[rp[w * 64]:rp[min(w * 64 + 64, M)]].tolist()))
        cols = wc[64 * wp[w]:64 * wp[w + 1]]
        assert wp[w + 1] - wp[w] == -(-len(used) // 64)
        assert cols[:len(used)].tolist() == used and np.all(cols[len(used):] == -1)
        for ch in range(wp[w], wp[w + 1]):
            for k in range(64):
                c = wc[64 * ch + k]
                if c < 0:
                    assert not wv[ch][:, k].any()
                else:
                    D[w * 64:(w + 1) * 64, c] += wv[ch][:, k]
    assert np.array_equal(D[:M], A) and not D[M:].any()
    assert fill == (rp[-1] / (wp[-1] * 4096) if wp[-1] else 0.0)


def test_wcsr_duplicate_rejected():
    with pytest.raises(Exception):
        oracle.build_wcsr(2, 4, [0, 2, 3], [1, 1, 0], np.ones(3, np.float32))


def test_coo_index_range_rejected():
    with pytest.raises(Exception):
        oracle.spmv_coo(2, 2, [0, 2], [0, 1], [1.0, 1.0], np.ones(2, np.float32))
    with pytest.raises(Exception):
        oracle.spmv_coo(2, 2, [0, 1], [0, 2], [1.0, 1.0], np.ones(2, np.float32))


# ------------------------------------------------------------ brute force

def _dense(M, K, row, col, val):
    A = np.zeros((M, K))
    np.add.at(A, (row, col), val.astype(np.float64))
    return A


CASES = [(1, 1, 0, 1), (7, 5, 0, 5), (33, 64, 0, 9), (64, 17, 3, 17), (50, 50, 0, 0), (0, 4, 0, 2), (9, 1, 0, 1)]


@pytest.mark.parametrize("M,K,lmin,lmax", CASES)
@pytest.mark.parametrize("seed", [11, 12])
def test_bruteforce_spmv_spmm(M, K, lmin, lmax, seed):
    d = synth.random_coo(seed, M, K, lmin, lmax, values="int")
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    A = _dense(M, K, d["row"], d["col"], d["val"])
    x = np.floor(synth.uniform(seed, synth.T_X, K, -3, 4)).astype(np.float32)
    y = np.floor(synth.uniform(seed, synth.T_Y, M, -3, 4)).astype(np.float32)
    ref, bound = oracle.spmv(M, rp, col, val, x, alpha=2.0, beta=-3.0, y=y)
    assert np.array_equal(ref, 2.0 * (A @ x.astype(np.float64)) - 3.0 * y)
    assert np.array_equal(bound, 2.0 * (np.abs(A) @ np.abs(x.astype(np.float64))) + 3.0 * np.abs(y))
    # beta == 0: y is not read (NaN must not leak)
    ref0, _ = oracle.spmv(M, rp, col, val, x, alpha=1.0, beta=0.0, y=np.full(M, np.nan, np.float32))
    assert np.array_equal(ref0, A @ x.astype(np.float64))
    for N in (1, 3, 8):
        B = np.floor(synth.uniform(seed, synth.T_B, K * N, -3, 4)).astype(np.float32).reshape(K, N)
        C = np.floor(synth.uniform(seed, synth.T_Y, M * N, -3, 4)).astype(np.float32).reshape(M, N)
        ref, _ = oracle.spmm(M, rp, col, val, B, alpha=-1.0, beta=0.5, C=C)
        assert np.array_equal(ref, -(A @ B.astype(np.float64)) + 0.5 * C)
    # COO product straight from the triplets, in the generator's order and shuffled
    for order in (np.arange(d["row"].size), synth.permutation(seed, d["row"].size)):
        refc, boundc = oracle.spmv_coo(M, K, d["row"][order], d["col"][order], d["val"][order], x, alpha=2.0,
                                       beta=-3.0, y=y)
        assert np.array_equal(refc, 2.0 * (A @ x.astype(np.float64)) - 3.0 * y)
        assert np.array_equal(boundc, 2.0 * (np.abs(A) @ np.abs(x.astype(np.float64))) + 3.0 * np.abs(y))
    # the dual direction: CSR(A^T) times u equals the transposed dense product
    trp, tc, tv = oracle.transpose(M, K, rp, col, val)
    u = np.floor(synth.uniform(seed, 7, M, -3, 4)).astype(np.float32)
    reft, _ = oracle.spmv(K, trp, tc, tv, u)
    assert np.array_equal(reft, A.T @ u.astype(np.float64))


@pytest.mark.parametrize("M,K,lmin,lmax", CASES)
@pytest.mark.parametrize("bs", [(1, 1), (2, 2), (3, 2), (4, 8)])
def test_bruteforce_bsr(M, K, lmin, lmax, bs):
    br, bc = bs
    d = synth.random_coo(5, M, K, lmin, lmax, values="int")
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
    A = _dense(M, K, d["row"], d["col"], d["val"])
    brp, bcol, bval, fill = oracle.build_bsr(M, K, rp, col, val, br, bc)
    # BSR expanded back to dense equals the CSR's dense form
    MB, KB = -(-M // br), -(-K // bc)
    D = np.zeros((MB * br, KB * bc))
    for I in range(MB):
        for b in range(brp[I], brp[I + 1]):
            D[I * br:(I + 1) * br, bcol[b] * bc:(bcol[b] + 1) * bc] = bval[b]
    assert np.array_equal(D[:M, :K], A)
    assert not D[M:, :].any() and not D[:, K:].any()
    # every stored block holds a nonzero; block columns ascend inside a block-row
    for I in range(MB):
        cs = bcol[brp[I]:brp[I + 1]]
        assert np.all(np.diff(cs) > 0)
    nnzb = brp[-1]
    assert fill == (rp[-1] / (nnzb * br * bc) if nnzb else 0.0)
    # BSR SpMM on bf16 bit patterns of small integers (exact in bf16 and fp64)
    N = 5
    Bf = np.floor(synth.uniform(3, synth.T_B, K * N, -3, 4)).astype(np.float32).reshape(K, N)
    ref, bound = oracle.bsr_spmm(M, K, br, bc, brp, bcol, synth.to_bf16_bits(bval).reshape(bval.shape),
                                 synth.to_bf16_bits(Bf).reshape(K, N))
    assert np.array_equal(ref, A @ Bf.astype(np.float64))
    assert np.array_equal(bound, np.abs(A) @ np.abs(Bf.astype(np.float64)))
    # C = alpha*A*B + beta*C with dyadic scalars and integer C: still exact
    C0 = np.floor(synth.uniform(4, synth.T_Y, M * N, -5, 6)).astype(np.float32).reshape(M, N)
    ref2, bound2 = oracle.bsr_spmm(M, K, br, bc, brp, bcol, synth.to_bf16_bits(bval).reshape(bval.shape),
                                   synth.to_bf16_bits(Bf).reshape(K, N), alpha=-1.5, beta=0.25, C=C0)
    assert np.array_equal(ref2, -1.5 * (A @ Bf.astype(np.float64)) + 0.25 * C0)
    assert np.array_equal(bound2, 1.5 * (np.abs(A) @ np.abs(Bf.astype(np.float64))) + 0.25 * np.abs(C0))


def test_bsr_stored_blocks_nonempty():
    d = synth.random_coo(8, 40, 40, 0, 6, values="ones")
    rp, col, val = oracle.build_csr(40, 40, d["row"], d["col"], d["val"])
    brp, bcol, bval, _ = oracle.build_bsr(40, 40, rp, col, val, 4, 4)
    assert all(b.any() for b in bval)
    # count of distinct (i//4, j//4) equals nnzb
    blocks = {(r // 4, c // 4) for r, c in zip(d["row"], d["col"])}
    assert len(blocks) == brp[-1]


def test_bsr_duplicate_rejected():
    rp = np.array([0, 2], np.int32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.build_bsr(1, 4, rp, np.array([1, 1], np.int32), np.ones(2, np.float32), 2, 2)
    assert e.value.code == oracle.ERR_DUP


def test_scipy_agrees_on_formats():
    sp = pytest.importorskip("scipy.sparse")
    for seed, (M, K) in enumerate([(30, 20), (64, 64), (5, 90)]):
        d = synth.random_coo(seed, M, K, 0, 12)
        perm = synth.permutation(seed, d["row"].size)
        rp, col, val = oracle.build_csr(M, K, d["row"][perm], d["col"][perm], d["val"][perm])
        S = sp.coo_matrix((d["val"], (d["row"], d["col"])), shape=(M, K)).tocsr()
        S.sort_indices()
        assert np.array_equal(rp, S.indptr) and np.array_equal(col, S.indices) and np.array_equal(val, S.data)
        T = S.T.tocsr()
        T.sort_indices()
        trp, tc, tv = oracle.transpose(M, K, rp, col, val)
        assert np.array_equal(trp, T.indptr) and np.array_equal(tc, T.indices) and np.array_equal(tv, T.data)
        Mp, Kp = -(-M // 4) * 4, -(-K // 2) * 2
        Sp = sp.csr_matrix((S.data, S.indices, np.concatenate([S.indptr, np.full(Mp - M, S.indptr[-1])])),
                           shape=(Mp, Kp))
        Bs = Sp.tobsr(blocksize=(4, 2))
        Bs.sort_indices()
        brp, bcol, bval, _ = oracle.build_bsr(M, K, rp, col, val, 4, 2)
        keep = np.array([np.any(b != 0) for b in Bs.data], bool)  # scipy may keep all-zero blocks
        assert np.array_equal(bcol, Bs.indices[keep]) and np.array_equal(bval, Bs.data[keep])


# ------------------------------------------------------------ invariants

def test_transpose_twice_is_identity():
    for seed, (M, K) in enumerate([(100, 37), (1, 300), (300, 1), (257, 513)]):
        d = synth.random_coo(seed, M, K, 0, 20)
        rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], d["val"])
        t = oracle.transpose(M, K, rp, col, val)
        back = oracle.transpose(K, M, *t)
        for a, b in zip((rp, col, val), back):
            assert np.array_equal(a, b)


def test_coo_shuffle_round_trip():
    d = synth.random_coo(21, 500, 700, 0, 30)
    rp, col, val = oracle.build_csr(500, 700, d["row"], d["col"], d["val"])
    perm = synth.permutation(4, rp[-1])
    row = np.repeat(np.arange(500, dtype=np.int32), np.diff(rp))
    again = oracle.build_csr(500, 700, row[perm], col[perm], val[perm])
    for a, b in zip((rp, col, val), again):
        assert np.array_equal(a, b)


def test_duplicates_kept_in_input_order():
    """Equal (row, col) pairs are kept, not summed, in input order (the pages
    are silent; this is the reading the library follows)."""
    row = np.array([1, 0, 1, 1], np.int32)
    col = np.array([2, 0, 2, 0], np.int32)
    val = np.array([10, 20, 30, 40], np.float32)
    rp, c, v = oracle.build_csr(2, 3, row, col, val)
    assert rp.tolist() == [0, 1, 4] and c.tolist() == [0, 0, 2, 2] and v.tolist() == [20, 40, 10, 30]


def test_index_range_rejected():
    with pytest.raises(oracle.OracleError) as e:
        oracle.build_csr(2, 2, np.array([0, 2], np.int32), np.array([0, 0], np.int32), np.ones(2, np.float32))
    assert e.value.code == oracle.ERR_INDEX
    with pytest.raises(oracle.OracleError):
        oracle.build_csr(2, 2, np.array([0, 1], np.int32), np.array([0, -1], np.int32), np.ones(2, np.float32))


# ------------------------------------------------------------ closed forms

@pytest.mark.parametrize("l", [0, 1, 31, 32, 33, 4097, 200_000])
def test_row_of_ones(l):
    K = max(l, 1)
    rp = np.array([0, l], np.int32)
    col = np.arange(l, dtype=np.int32)
    ref, _ = oracle.spmv(1, rp, col, np.ones(l, np.float32), np.ones(K, np.float32))
    assert ref[0] == l


def test_stats_against_numpy():
    for seed in range(4):
        L = synth.lengths_uniform(seed, 1000 + seed, 0, 50)
        rp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
        st = oracle.row_stats(L.size, rp)
        assert st["nnz"] == L.sum() and st["sumsq"] == (L.astype(np.int64) ** 2).sum()
        assert st["max"] == L.max() and st["min"] == L.min() and st["empty"] == (L == 0).sum()
        assert st["mean"] == pytest.approx(L.mean(), rel=1e-15)
        assert st["var"] == pytest.approx(L.var(), rel=1e-12)
        for q in (50, 95, 99):
            assert st[f"p{q}"] == np.percentile(L, q, method="inverted_cdf")
    L = np.full(77, 9, np.int32)
    st = oracle.row_stats(77, np.arange(0, 78 * 9, 9, dtype=np.int32))
    assert st["var"] == 0.0 and st["cv"] == 0.0 and st["p99"] == 9 and st["mean"] == 9.0


def test_stats_exact_rational():
    """var is the exact rational (M*S2 - S1^2)/M^2 rounded: compare with
    Python's exact fractions."""
    from fractions import Fraction

    L = synth.lengths_uniform(3, 12345, 0, 1000)
    rp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    st = oracle.row_stats(L.size, rp)
    M, S1, S2 = L.size, int(L.sum()), int((L.astype(np.int64) ** 2).sum())
    num = M * S2 - S1 * S1
    assert st["var"] == float(num) / (float(M) * float(M))
    assert abs(Fraction(st["var"]) - Fraction(num, M * M)) <= Fraction(num, M * M) * Fraction(1, 2 ** 51)


# ------------------------------------------------------------ the plan

OPTS_SMALL = dict(block_nnz=16, block_rows=3, pack_max=8, cta_max=100, seg_nnz=40, lanes_div=2)


def test_plan_hand_example():
    L = [3, 0, 5, 8, 2, 50, 4, 0, 250, 6, 6, 6]
    rp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    p = oracle.plan_spmv(len(L), rp, **OPTS_SMALL)
    want = [[1, 5, 0, 0]] + [[2, 8, s, s] for s in range(7)] + [
        [256, 0, 3, 0], [512, 3, 5, 0], [0, 6, 8, 0], [512, 9, 11, 0], [512, 11, 12, 0]]
    assert p["tasks"].tolist() == want
    assert p["longrows"].tolist() == [[8, 0, 7, 0]]
    assert p["counts"] == dict(tasks=13, long_rows=1, slots=7, packed_rows=10, cta_rows=1, split_rows=1,
                               thread_groups=1, lane_groups=4, segmented_groups=0)
    # D = 0: the same groups, every one with the segmented reduction (code 6)
    q = oracle.plan_spmv(len(L), rp, **dict(OPTS_SMALL, lanes_div=0))
    seg = [t if t[0] & 255 else [6 * 256, t[1], t[2], 0] for t in want]
    assert q["tasks"].tolist() == seg
    assert q["counts"]["segmented_groups"] == 5 and q["counts"]["thread_groups"] == 0


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("div", [0, 4])
def test_plan_invariants(seed, div):
    L, _ = synth.lengths_zipf(seed, 3000, 2.1, 3000, 6.0)
    L[::97] = 0
    rp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    o = dict(block_nnz=64, block_rows=16, pack_max=32, cta_max=200, seg_nnz=50, lanes_div=div)
    p = oracle.plan_spmv(L.size, rp, **o)
    covered = np.zeros(L.size, np.int64)
    seg_cover = {}
    for kind, a, b, c in p["tasks"].tolist():
        k = kind & 255
        if k == 0:
            rows = np.arange(a, b)
            assert 1 <= b - a <= o["block_rows"]
            assert np.all(L[rows] <= o["pack_max"]) and L[rows].sum() <= o["block_nnz"]
            if div == 0:
                assert kind >> 8 == 6
            else:
                w = 1 << (kind >> 8)
                per = -(-int(L[rows].sum()) // ((b - a) * o["lanes_div"]))
                assert w == min(32, max(1, 1 << int(np.ceil(np.log2(max(per, 1))))))
            covered[rows] += 1
        elif k == 1:
            assert o["pack_max"] < L[a] <= o["cta_max"]
            covered[a] += 1
        else:
            assert L[a] > o["cta_max"]
            seg_cover.setdefault(a, []).append((b, c))
    for row, first, ns, _ in p["longrows"].tolist():
        segs = seg_cover.pop(row)
        assert [s for s, _ in segs] == list(range(ns)) and [c for _, c in segs] == list(range(first, first + ns))
        assert (ns - 1) * o["seg_nnz"] < L[row] <= ns * o["seg_nnz"]
        covered[row] += 1
    assert not seg_cover
    assert np.all(covered == 1)
    c = p["counts"]
    assert c["packed_rows"] + c["cta_rows"] + c["split_rows"] == L.size
    # groups are maximal: the next packed row would break a limit
    groups = [t for t in p["tasks"].tolist() if t[0] & 255 == 0]
    for (k1, a1, b1, _), (k2, a2, b2, _) in zip(groups, groups[1:]):
        if b1 == a2:
            assert b1 - a1 == o["block_rows"] or L[a1:b1].sum() + L[a2] > o["block_nnz"]


# ------------------------------------------------------------ the automatic plan options

# The rule as this library defines it (the pages give the dispatch key -- mean,
# spread and tail of the row lengths -- but no thresholds, [SpMM-ops] §4): a
# coefficient of variation of 2 or more picks 1024-nonzero groups with the
# segmented reduction, anything below keeps the defaults.  Written out here
# field by field, not taken from either implementation.
RULE_SKEWED = dict(block_nnz=1024, block_rows=256, pack_max=512, cta_max=8192, seg_nnz=4096, lanes_div=0)
RULE_DEFAULT = dict(block_nnz=2048, block_rows=256, pack_max=512, cta_max=8192, seg_nnz=4096, lanes_div=16)


def _stats(cv, **kw):
    base = dict(rows=1000, nnz=16000, sumsq=400000, min=1, max=300, p50=10, p95=60, p99=200, empty=0,
                mean=16.0, var=(cv * 16.0) ** 2, cv=cv)
    base.update(kw)
    return base


@pytest.mark.parametrize("cv,skewed", [(0.0, False), (0.5, False), (1.0, False), (np.nextafter(2.0, 0.0), False),
                                       (2.0, True), (np.nextafter(2.0, 3.0), True), (2.5, True), (40.0, True)])
def test_plan_opts_auto_threshold(cv, skewed):
    """The cv >= 2 edge, one ulp either side of it, and every field of both outcomes."""
    assert oracle.plan_opts_from_stats(_stats(cv)) == (RULE_SKEWED if skewed else RULE_DEFAULT)


def test_plan_opts_auto_reads_only_cv():
    """Extreme values in every other field (an enormous tail, all-empty rows, a huge mean) do not move the choice."""
    for kw in (dict(max=200000, p99=100000, p95=50000), dict(empty=1000, min=0, nnz=0, mean=0.0),
               dict(mean=1e6, nnz=10 ** 12, sumsq=10 ** 15), dict(rows=1, p50=0)):
        assert oracle.plan_opts_from_stats(_stats(1.99, **kw)) == RULE_DEFAULT
        assert oracle.plan_opts_from_stats(_stats(2.01, **kw)) == RULE_SKEWED


def test_plan_opts_auto_on_the_worked_example(ex):
    """The worked example's lengths [2, 1, 3, 1, 1]: mean 1.6, variance 0.64, cv 0.5 -> the defaults."""
    g, _, _ = ex
    rp = np.array(g["printed"]["csr_row_ptr"], np.int32)
    st = oracle.row_stats(5, rp)
    assert st["cv"] == pytest.approx(0.5, rel=1e-15)
    assert oracle.plan_opts_from_stats(st) == RULE_DEFAULT
    assert oracle.plan_opts_auto(5, rp) == RULE_DEFAULT


def test_plan_opts_auto_on_closed_form_lengths():
    """Lengths with a cv known in closed form: constant rows (cv 0) and one row of n with M-1 empty rows
    (cv = sqrt(M - 1)): M = 4 gives sqrt(3) < 2, M = 5 gives exactly 2, M = 6 gives sqrt(5) > 2."""
    for M, want in ((4, RULE_DEFAULT), (5, RULE_SKEWED), (6, RULE_SKEWED)):
        rp = np.array([0] + [7] * M, np.int32)
        st = oracle.row_stats(M, rp)
        assert st["cv"] == pytest.approx(np.sqrt(M - 1), rel=1e-15)
        assert oracle.plan_opts_auto(M, rp) == want
    rp = np.arange(0, 9 * 100 + 1, 9, dtype=np.int32)
    assert oracle.row_stats(100, rp)["cv"] == 0.0 and oracle.plan_opts_auto(100, rp) == RULE_DEFAULT


# ------------------------------------------------------------ the fp32 sequential variant

U32 = 2.0 ** -24


def gamma(n):
    """gamma_n = n u / (1 - n u): the textbook bound on the relative error of n
    fp32 roundings in a recursively summed dot product (u = 2^-24)."""
    return n * U32 / (1.0 - n * U32)


def _f32_bound_check(M, rp, col, val, x, alpha, beta, y0):
    ref, bound = oracle.spmv(M, rp, col, val, x, alpha, beta, y0)
    r32 = oracle.spmv_f32(M, rp, col, val, x, alpha, beta, y0).astype(np.float64)
    L = np.diff(rp).astype(np.float64)
    # l products and l - 1 additions in the row, then alpha * s, beta * y and their sum: at most l + 2
    # roundings along any path; the fp64 reference's own error (2^-52 per step) is added for rigour
    tol = gamma(L + 2) * bound + (L + 2) * 2.0 ** -52 * bound
    err = np.abs(r32 - ref)
    assert np.all(err <= tol), np.max(err - tol)
    return err, ref, bound


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-1.5, 0.5)])
def test_fp32_sequential_within_textbook_bound(seed, alpha, beta):
    """Random rows of lengths 0 .. 200,000 with values and x in [-1, 1): the fp32 index-order sum stays within
    gamma_(l+2) times the oracle's bound of the fp64 result, row by row."""
    L, _ = synth.lengths_zipf(seed, 2000, 2.1, 200_000, 30.0)
    L[:2] = (200_000, 0)
    row, col = synth.cols_uniform(seed, 300_000, L)
    val = synth.uniform(seed, synth.T_VAL, row.size)
    rp, col, val = oracle.build_csr(L.size, 300_000, row, col, val)
    x = synth.uniform(seed, synth.T_X, 300_000)
    y0 = synth.uniform(seed, synth.T_Y, L.size)
    _f32_bound_check(L.size, rp, col, val, x, alpha, beta, y0)


def test_fp32_sequential_exact_on_small_integers():
    """Small-integer values and x: every fp32 partial sum is an integer below 2^24, so both variants agree exactly."""
    d = synth.random_coo(12, 300, 200, 0, 60)
    rp, col, _ = oracle.build_csr(300, 200, d["row"], d["col"], d["val"])
    rng = np.random.default_rng(12)
    val = rng.integers(-8, 9, col.size).astype(np.float32)
    x = rng.integers(-8, 9, 200).astype(np.float32)
    y0 = rng.integers(-8, 9, 300).astype(np.float32)
    ref, _ = oracle.spmv(300, rp, col, val, x, 2.0, -3.0, y0)
    assert np.array_equal(oracle.spmv_f32(300, rp, col, val, x, 2.0, -3.0, y0).astype(np.float64), ref)


def test_fp32_bound_needs_absolute_values():
    """Heavy cancellation: l - 1 products of 0.1 then one product of -(l - 1) * 0.1.  The fp32 running sum drifts
    by far more than gamma_l times |exact sum|, yet stays within gamma_l times sum |products| -- so a bound
    written with the signed sum (a dropped absolute value) would fail the check above."""
    for l in (1000, 50_000, 200_000):
        val = np.full(l, np.float32(0.1), np.float32)
        val[-1] = np.float32(-(l - 1) * 0.1)
        col = np.zeros(l, np.int32)
        rp = np.array([0, l], np.int32)
        x = np.ones(1, np.float32)
        err, ref, bound = _f32_bound_check(1, rp, col, val, x, 1.0, 0.0, None)
        assert err[0] > gamma(l + 2) * abs(ref[0])
        assert bound[0] > 10 * abs(ref[0])
