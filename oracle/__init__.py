"""The test oracle: plain CPU restatement of the sparse x dense products.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with ``csr_bsr_spmv_gb300`` and never imports it; the arithmetic lives in
``oracle.c`` (plain C, fp64 accumulation, single-threaded), built with the
host C compiler; a second build of the same source with OpenMP runs the
products' independent row loops on all host cores for the CPU baseline.  Each function's docstring in ``oracle.c`` cites the page
section it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_LIB_OMP = os.path.join(_HERE, "liboracle_omp.so")
_lock = threading.Lock()
_lib = None
_lib_omp = None

OK, ERR_ARG, ERR_INDEX, ERR_DUP = 0, -1, -2, -4

# plan option order mirrors or_plan_opts_t
PLAN_FIELDS = ("block_nnz", "block_rows", "pack_max", "cta_max", "seg_nnz", "lanes_div")
TASK_GROUP, TASK_CTA, TASK_SEG = 0, 1, 2


class PlanOpts(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int32) for f in PLAN_FIELDS]


class RowStats(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("nnz", ctypes.c_int64), ("sumsq", ctypes.c_int64),
                ("min", ctypes.c_int32), ("max", ctypes.c_int32), ("p50", ctypes.c_int32),
                ("p95", ctypes.c_int32), ("p99", ctypes.c_int32), ("empty", ctypes.c_int32),
                ("mean", ctypes.c_double), ("var", ctypes.c_double), ("cv", ctypes.c_double)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile liboracle.so: -O2, no fast-math, no FMA contraction.  With
    openmp=True the same source goes to liboracle_omp.so with -fopenmp: the
    all-core build that the CPU baseline times (row loops on all cores)."""
    out = _LIB_OMP if openmp else _LIB
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off"] + (["-fopenmp"] if openmp else []) + [_SRC, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


def _lib_(threads: int = 1):
    """The single-thread library, or with threads > 1 the all-core build set to that many threads."""
    global _lib, _lib_omp
    if threads > 1:
        with _lock:
            if _lib_omp is None:
                lib = ctypes.CDLL(build(openmp=True))
                _declare(lib)
                _lib_omp = lib
        _lib_omp.or_threads(int(threads))
        return _lib_omp
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            _declare(lib)
            _lib = lib
    return _lib


def omp_threads(threads: int) -> int:
    """Threads the all-core build actually runs with when asked for `threads`."""
    return int(_lib_(max(2, threads)).or_threads(int(threads)))


def _declare(lib):
    vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    sig = {
        "or_build_csr": [i32, i32, i64, vp, vp, vp, i32, vp, vp, vp],
        "or_transpose": [i32, i32, i64, vp, vp, vp, i32, vp, vp, vp],
        "or_build_bsr": [i32, i32, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp],
        "or_row_stats": [i32, vp, vp],
        "or_plan_spmv": [i32, vp, vp, vp, vp, vp],
        "or_plan_opts_auto": [vp, vp],
        "or_spmv": [i32, vp, vp, vp, vp, dbl, dbl, vp, vp, i64, vp, vp],
        "or_spmv_f32": [i32, vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp, vp, i64, vp],
        "or_threads": [i32],
        "or_spmv_coo": [i32, i32, i64, vp, vp, vp, vp, dbl, dbl, vp, vp, vp],
        "or_build_wcsr": [i32, i32, vp, vp, vp, i32, vp, vp, vp, ctypes.POINTER(ctypes.c_int64),
                          ctypes.POINTER(ctypes.c_double)],
        "or_build_sell": [i32, vp, vp, vp, i32, i32, ctypes.POINTER(ctypes.c_int64),
                          ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                          ctypes.POINTER(ctypes.c_int64), vp, vp, vp, vp, vp],
        "or_spmm": [i32, i32, vp, vp, vp, vp, i64, dbl, dbl, vp, i64, vp, i64, vp, vp],
        "or_bsr_spmm": [i32, i32, i32, i32, vp, vp, vp, i32, vp, i64, dbl, dbl, vp, i64, vp, i64, vp, vp],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__(f"oracle status {code}")
        self.code = code


def _check(rc):
    if rc != OK:
        raise OracleError(rc)


def build_csr(M, K, row, col, val):
    row, col = _c(row, np.int32), _c(col, np.int32)
    val = np.ascontiguousarray(val)
    nnz = row.size
    rp = np.empty(M + 1, np.int32)
    co = np.empty(nnz, np.int32)
    vo = np.empty(nnz, val.dtype)
    _check(_lib_().or_build_csr(M, K, nnz, _p(row), _p(col), _p(val), val.itemsize, _p(rp), _p(co), _p(vo)))
    return rp, co, vo


def transpose(M, K, rp, col, val):
    rp, col = _c(rp, np.int32), _c(col, np.int32)
    val = np.ascontiguousarray(val)
    nnz = int(rp[M])
    trp = np.empty(K + 1, np.int32)
    tc = np.empty(nnz, np.int32)
    tv = np.empty(nnz, val.dtype)
    _check(_lib_().or_transpose(M, K, nnz, _p(rp), _p(col), _p(val), val.itemsize, _p(trp), _p(tc), _p(tv)))
    return trp, tc, tv


def build_bsr(M, K, rp, col, val, br, bc):
    """Returns (bsr_row_ptr, bsr_col, bsr_val[nnzb, br, bc], fill)."""
    rp, col = _c(rp, np.int32), _c(col, np.int32)
    val = np.ascontiguousarray(val)
    MB = (M + br - 1) // br
    nnzb = ctypes.c_int64(0)
    fill = ctypes.c_double(0.0)
    brp = np.empty(MB + 1, np.int32)
    lib = _lib_()
    _check(lib.or_build_bsr(M, K, _p(rp), _p(col), _p(val), val.itemsize, br, bc, _p(brp), None, None,
                            ctypes.byref(nnzb), ctypes.byref(fill)))
    nb = nnzb.value
    bcol = np.empty(nb, np.int32)
    bval = np.empty(nb * br * bc, val.dtype)
    _check(lib.or_build_bsr(M, K, _p(rp), _p(col), _p(val), val.itemsize, br, bc, _p(brp), _p(bcol), _p(bval),
                            ctypes.byref(nnzb), ctypes.byref(fill)))
    return brp, bcol, bval.reshape(nb, br, bc), fill.value


def build_sell(M, rp, col, val, sigma=1024, piece=64):
    """SELL-C-sigma (C = 32) with rows longer than `piece` cut into pieces.
    Returns (slice_ptr, prow, longrows[nlong, 4], scol, sval)."""
    rp, col, val = _c(rp, np.int32), _c(col, np.int32), _c(val, np.float32)
    n = [ctypes.c_int64(0) for _ in range(4)]
    lib = _lib_()
    _check(lib.or_build_sell(M, _p(rp), _p(col), _p(val), sigma, piece, *[ctypes.byref(v) for v in n],
                             None, None, None, None, None))
    npseudo, ns, pad, nl = (v.value for v in n)
    sp = np.empty(ns + 1, np.int32)
    pr = np.empty(32 * ns, np.int32)
    lr = np.empty((nl, 4), np.int32)
    sc = np.empty(pad, np.int32)
    sv = np.empty(pad, np.float32)
    _check(lib.or_build_sell(M, _p(rp), _p(col), _p(val), sigma, piece, *[ctypes.byref(v) for v in n], _p(sp),
                             _p(pr), _p(lr), _p(sc), _p(sv)))
    return sp, pr, lr, sc, sv


def build_wcsr(M, K, rp, col, val):
    """Returns (win_ptr, win_col[nchunks*64], win_val[nchunks, 64, 64], fill)."""
    rp, col = _c(rp, np.int32), _c(col, np.int32)
    val = np.ascontiguousarray(val)
    W = (M + 63) // 64
    nch = ctypes.c_int64(0)
    fill = ctypes.c_double(0.0)
    wp = np.empty(W + 1, np.int32)
    lib = _lib_()
    _check(lib.or_build_wcsr(M, K, _p(rp), _p(col), _p(val), val.itemsize, _p(wp), None, None, ctypes.byref(nch),
                             ctypes.byref(fill)))
    nc = nch.value
    wc = np.empty(nc * 64, np.int32)
    wv = np.empty(nc * 4096, val.dtype)
    _check(lib.or_build_wcsr(M, K, _p(rp), _p(col), _p(val), val.itemsize, _p(wp), _p(wc), _p(wv),
                             ctypes.byref(nch), ctypes.byref(fill)))
    return wp, wc, wv.reshape(nc, 64, 64), fill.value


def row_stats(M, rp):
    rp = _c(rp, np.int32)
    st = RowStats()
    _check(_lib_().or_row_stats(M, _p(rp), ctypes.byref(st)))
    return st.as_dict()


def plan_opts_auto(M, rp):
    """Plan options the statistics rule picks for this matrix."""
    rp = _c(rp, np.int32)
    st = RowStats()
    _check(_lib_().or_row_stats(M, _p(rp), ctypes.byref(st)))
    o = PlanOpts()
    _check(_lib_().or_plan_opts_auto(ctypes.byref(st), ctypes.byref(o)))
    return {f: getattr(o, f) for f in PLAN_FIELDS}


def plan_opts_from_stats(stats):
    """Plan options the statistics rule picks for a row-statistics record (dict with the RowStats fields)."""
    st = RowStats(**{f: stats[f] for f, _ in RowStats._fields_})
    o = PlanOpts()
    _check(_lib_().or_plan_opts_auto(ctypes.byref(st), ctypes.byref(o)))
    return {f: getattr(o, f) for f in PLAN_FIELDS}


def plan_spmv(M, rp, **opts):
    """Returns dict(tasks[ntasks,4], longrows[nlong,4], counts)."""
    rp = _c(rp, np.int32)
    o = PlanOpts(**{f: int(opts[f]) for f in PLAN_FIELDS})
    counts = np.zeros(9, np.int64)
    lib = _lib_()
    _check(lib.or_plan_spmv(M, _p(rp), ctypes.byref(o), None, None, _p(counts)))
    tasks = np.empty((int(counts[0]), 4), np.int32)
    longrows = np.empty((int(counts[1]), 4), np.int32)
    _check(lib.or_plan_spmv(M, _p(rp), ctypes.byref(o), _p(tasks), _p(longrows), _p(counts)))
    names = ("tasks", "long_rows", "slots", "packed_rows", "cta_rows", "split_rows", "thread_groups",
             "lane_groups", "segmented_groups")
    return dict(tasks=tasks, longrows=longrows, counts=dict(zip(names, (int(c) for c in counts))))


def spmv(M, rp, col, val, x, alpha=1.0, beta=0.0, y=None, rows=None, threads=1):
    """(ref, bound) in fp64, for all rows or the given sample of rows
    (threads > 1: the all-core build, same result)."""
    rp, col, val, x = _c(rp, np.int32), _c(col, np.int32), _c(val, np.float32), _c(x, np.float32)
    yv = _c(y, np.float32) if (y is not None and beta != 0.0) else None
    rr = None if rows is None else _c(rows, np.int32)
    n = M if rr is None else rr.size
    ref = np.empty(n, np.float64)
    bnd = np.empty(n, np.float64)
    _check(_lib_(threads).or_spmv(M, _p(rp), _p(col), _p(val), _p(x), float(alpha), float(beta), _p(yv), _p(rr),
                                  0 if rr is None else rr.size, _p(ref), _p(bnd)))
    return ref, bnd


def spmv_f32(M, rp, col, val, x, alpha=1.0, beta=0.0, y=None, rows=None):
    """The fp32 index-order SpMV (products and running sums rounded to fp32), for all rows or a sample."""
    rp, col, val, x = _c(rp, np.int32), _c(col, np.int32), _c(val, np.float32), _c(x, np.float32)
    yv = _c(y, np.float32) if (y is not None and beta != 0.0) else None
    rr = None if rows is None else _c(rows, np.int32)
    n = M if rr is None else rr.size
    out = np.empty(max(n, 1), np.float32)
    _check(_lib_().or_spmv_f32(M, _p(rp), _p(col), _p(val), _p(x), float(alpha), float(beta), _p(yv), _p(rr),
                               0 if rr is None else rr.size, _p(out)))
    return out[:n]


def spmv_coo(M, K, row, col, val, x, alpha=1.0, beta=0.0, y=None):
    """(ref, bound) in fp64 of the COO product over all M rows (triplets in any order)."""
    row, col, val, x = _c(row, np.int32), _c(col, np.int32), _c(val, np.float32), _c(x, np.float32)
    yv = _c(y, np.float32) if (y is not None and beta != 0.0) else None
    ref = np.empty(max(M, 1), np.float64)
    bnd = np.empty(max(M, 1), np.float64)
    _check(_lib_().or_spmv_coo(M, K, col.size, _p(row), _p(col), _p(val), _p(x), float(alpha), float(beta), _p(yv),
                               _p(ref), _p(bnd)))
    return ref[:M], bnd[:M]


def spmm(M, rp, col, val, B, alpha=1.0, beta=0.0, C=None, rows=None, threads=1):
    rp, col, val = _c(rp, np.int32), _c(col, np.int32), _c(val, np.float32)
    B = _c(B, np.float32)
    N = B.shape[1]
    Cv = _c(C, np.float32) if (C is not None and beta != 0.0) else None
    rr = None if rows is None else _c(rows, np.int32)
    n = M if rr is None else rr.size
    ref = np.empty((n, N), np.float64)
    bnd = np.empty((n, N), np.float64)
    _check(_lib_(threads).or_spmm(M, N, _p(rp), _p(col), _p(val), _p(B), N, float(alpha), float(beta), _p(Cv),
                           N if Cv is not None else 0, _p(rr), 0 if rr is None else rr.size, _p(ref), _p(bnd)))
    return ref, bnd


def bsr_spmm(M, K, br, bc, brp, bcol, bval_bf16, B_bf16, rows=None, alpha=1.0, beta=0.0, C=None, threads=1):
    brp, bcol = _c(brp, np.int32), _c(bcol, np.int32)
    bval = _c(bval_bf16, np.uint16)
    B = _c(B_bf16, np.uint16)
    N = B.shape[1]
    rr = None if rows is None else _c(rows, np.int32)
    n = M if rr is None else rr.size
    ref = np.empty((n, N), np.float64)
    bnd = np.empty((n, N), np.float64)
    Cv = _c(C, np.float32) if (C is not None and beta != 0.0) else None
    _check(_lib_(threads).or_bsr_spmm(M, K, br, bc, _p(brp), _p(bcol), _p(bval), N, _p(B), N, float(alpha), float(beta),
                               _p(Cv), N if Cv is not None else 0, _p(rr), 0 if rr is None else rr.size, _p(ref),
                               _p(bnd)))
    return ref, bnd
