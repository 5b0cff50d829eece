"""Thin ctypes binding over libspx (include/spx.h).

Every function here marshals arguments -- tensor pointers, sizes, the current
CUDA stream -- into one C-ABI call of the same name; all computation runs in
the library.  PyTorch supplies device memory and streams only.  There is no
fallback: if libspx.so is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspx.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "spx.h")

SPX_HOST, SPX_DEVICE = 0, 1
STATUS = {0: "SPX_OK", -1: "SPX_ERR_ARG", -2: "SPX_ERR_INDEX_RANGE", -3: "SPX_ERR_NOT_SORTED",
          -4: "SPX_ERR_DUPLICATE", -5: "SPX_ERR_CUDA", -6: "SPX_ERR_TIMEOUT", -7: "SPX_ERR_UNSUPPORTED",
          -8: "SPX_ERR_ALIGN", -9: "SPX_ERR_NOMEM", -10: "SPX_ERR_NOT_READY", -11: "SPX_ERR_SCRATCH_LIMIT"}
SPMM_VARIANTS = {0: "small-N", 1: "float4", 2: "float4-wide", 3: "scalar"}


class SpxError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        msg = _lib().spx_status_string(code).decode() if _LIB is not None else self.name
        super().__init__(f"{where}: {msg}")


class PlanOpts(ctypes.Structure):
    _fields_ = [("block_nnz", ctypes.c_int32), ("block_rows", ctypes.c_int32), ("pack_max", ctypes.c_int32),
                ("cta_max", ctypes.c_int32), ("seg_nnz", ctypes.c_int32), ("lanes_div", ctypes.c_int32)]


class RowStats(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("nnz", ctypes.c_int64), ("sumsq", ctypes.c_int64),
                ("min", ctypes.c_int32), ("max", ctypes.c_int32), ("p50", ctypes.c_int32),
                ("p95", ctypes.c_int32), ("p99", ctypes.c_int32), ("empty", ctypes.c_int32),
                ("mean", ctypes.c_double), ("var", ctypes.c_double), ("cv", ctypes.c_double)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class PlanInfo(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("K", ctypes.c_int64), ("nnz", ctypes.c_int64), ("tasks", ctypes.c_int64),
                ("long_rows", ctypes.c_int64), ("slots", ctypes.c_int64), ("packed_rows", ctypes.c_int64),
                ("cta_rows", ctypes.c_int64), ("split_rows", ctypes.c_int64), ("thread_groups", ctypes.c_int64),
                ("lane_groups", ctypes.c_int64), ("segmented_groups", ctypes.c_int64), ("table_bytes", ctypes.c_size_t),
                ("scratch_bytes", ctypes.c_size_t), ("stats", RowStats), ("opts", PlanOpts)]


class SellOpts(ctypes.Structure):
    _fields_ = [("sigma", ctypes.c_int32), ("piece", ctypes.c_int32)]


class SellInfo(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("K", ctypes.c_int64), ("nnz", ctypes.c_int64), ("slices", ctypes.c_int64),
                ("pseudo_rows", ctypes.c_int64), ("padded", ctypes.c_int64), ("long_rows", ctypes.c_int64),
                ("slots", ctypes.c_int64), ("image_bytes", ctypes.c_size_t), ("scratch_bytes", ctypes.c_size_t),
                ("opts", SellOpts)]


class WcsrPlanInfo(ctypes.Structure):
    _fields_ = [("windows", ctypes.c_int64), ("tasks", ctypes.c_int64), ("split_windows", ctypes.c_int64),
                ("slots", ctypes.c_int64), ("table_bytes", ctypes.c_size_t), ("max_chunks", ctypes.c_int32)]


LIB_CHECK_PATH = os.path.join(_HERE, "libspx_check.so")  # the bounds-checked build of the same sources

_LIB = None
_CHECKED = None
_use_checked = False


def _lib():
    """The library every call below goes through: libspx.so, or inside `checked_build()` libspx_check.so."""
    global _LIB, _CHECKED
    if _use_checked:
        if _CHECKED is None:
            if not os.path.exists(LIB_CHECK_PATH):
                raise ImportError(f"{LIB_CHECK_PATH} is not built; run __graft_entry__.build()")
            _CHECKED = _load(LIB_CHECK_PATH)
        return _CHECKED
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build()")
        _LIB = _load(LIB_PATH)
    return _LIB


class checked_build:
    """Context in which the calls of this module go to libspx_check.so, the build that tests every
    index it reads from the caller's arrays before using it and reports a bad one through
    spx_last_device_error (SPX_ERR_INDEX_RANGE) instead of reading out of bounds.  For finding bad
    inputs; objects (plans, SELL forms, task splits) made inside the context belong to it."""

    def __enter__(self):
        global _use_checked
        self._prev = _use_checked
        _use_checked = True
        return _lib()

    def __exit__(self, *exc):
        global _use_checked
        _use_checked = self._prev
        return False


def _load(path):
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    d = ctypes.POINTER(ctypes.c_double)
    sigs = {
        "spx_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "spx_launch_count": ([ctypes.POINTER(ctypes.c_uint64)], ctypes.c_int),
        "spx_build_csr": ([i32, i32, i64, vp, vp, vp, i32, vp, vp, vp, ctypes.c_int, vp], ctypes.c_int),
        "spx_transpose_csr": ([i32, i32, i64, vp, vp, vp, i32, vp, vp, vp, ctypes.c_int, vp], ctypes.c_int),
        "spx_build_bsr": ([i32, i32, vp, vp, vp, i32, i32, i32, vp, vp, vp, ctypes.POINTER(ctypes.c_int64), d,
                           ctypes.c_int, vp], ctypes.c_int),
        "spx_check_csr": ([i32, i32, i64, vp, vp, i32, ctypes.c_int, vp], ctypes.c_int),
        "spx_row_stats": ([i32, vp, ctypes.c_int, ctypes.POINTER(RowStats)], ctypes.c_int),
        "spx_plan_opts_default": ([ctypes.POINTER(PlanOpts)], ctypes.c_int),
        "spx_plan_opts_auto": ([ctypes.POINTER(RowStats), ctypes.POINTER(PlanOpts)], ctypes.c_int),
        "spx_plan_csr": ([i32, i32, i64, vp, ctypes.c_int, ctypes.POINTER(PlanOpts), ctypes.POINTER(vp)],
                         ctypes.c_int),
        "spx_plan_get_info": ([vp, ctypes.POINTER(PlanInfo)], ctypes.c_int),
        "spx_plan_get_tasks": ([vp, vp, vp], ctypes.c_int),
        "spx_plan_get_table": ([vp, vp], ctypes.c_int),
        "spx_plan_upload": ([vp, vp, sz, vp], ctypes.c_int),
        "spx_plan_destroy": ([vp], ctypes.c_int),
        "spx_plan_fingerprint": ([vp, ctypes.POINTER(ctypes.c_uint64)], ctypes.c_int),
        "spx_plan_validate": ([vp, i32, i32, i64, vp, ctypes.c_int, vp], ctypes.c_int),
        "spx_plan_autotune": ([i32, i32, i64, vp, vp, vp, vp, vp, vp, ctypes.POINTER(PlanOpts), i32, i32, vp,
                               ctypes.POINTER(PlanOpts), ctypes.POINTER(ctypes.c_float),
                               ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
        "spx_plan_autotune_forget": ([], ctypes.c_int),
        "spx_sell_opts_default": ([ctypes.POINTER(SellOpts)], ctypes.c_int),
        "spx_sell_build": ([i32, i32, i64, vp, vp, vp, ctypes.c_int, ctypes.POINTER(SellOpts),
                            ctypes.POINTER(vp)], ctypes.c_int),
        "spx_sell_get_info": ([vp, ctypes.POINTER(SellInfo)], ctypes.c_int),
        "spx_sell_get_arrays": ([vp, vp, vp, vp, vp, vp], ctypes.c_int),
        "spx_sell_upload": ([vp, vp, sz, vp], ctypes.c_int),
        "spx_sell_destroy": ([vp], ctypes.c_int),
        "spx_spmv_sell": ([vp, i32, i32, f32, vp, f32, vp, vp, sz, vp], ctypes.c_int),
        "spx_spmv_csr": ([vp, i32, i32, i64, vp, vp, vp, f32, vp, f32, vp, vp, sz, vp], ctypes.c_int),
        "spx_spmv_csr_noalloc": ([vp, i32, i32, i64, vp, vp, vp, f32, vp, f32, vp, vp], ctypes.c_int),
        "spx_spmv_csr_hostio_work_bytes": ([i32, i32], sz),
        "spx_spmv_csr_hostio": ([vp, i32, i32, i64, vp, vp, vp, f32, vp, i64, f32, vp, i64, i32, vp, sz, vp, sz, vp],
                                ctypes.c_int),
        "spx_spmv_coo_scratch_bytes": ([i64], sz),
        "spx_spmv_coo": ([i32, i32, i64, vp, vp, vp, f32, vp, f32, vp, vp, sz, vp], ctypes.c_int),
        "spx_spmv_csr_dual": ([vp, vp, i32, i32, i64, vp, vp, vp, vp, vp, vp, vp, f32, f32, vp, f32, f32, vp,
                               sz, vp], ctypes.c_int),
        "spx_spmm_csr": ([i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, vp], ctypes.c_int),
        "spx_spmm_csr_tiled": ([i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, i32, vp], ctypes.c_int),
        "spx_spmm_csr_variant": ([i32, vp, i64, vp, i64], ctypes.c_int32),
        "spx_spmm_csr_bf16": ([i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, vp], ctypes.c_int),
        "spx_spmm_csr_f16": ([i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, vp], ctypes.c_int),
        "spx_spmm_csr_planned_scratch_bytes": ([vp, i32], sz),
        "spx_spmm_csr_planned": ([vp, i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, vp, sz, vp],
                                 ctypes.c_int),
        "spx_spmm_csr_bf16_planned": ([vp, i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, vp, sz, vp],
                                      ctypes.c_int),
        "spx_spmm_csr_f16_planned": ([vp, i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, vp, sz, vp],
                                     ctypes.c_int),
        "spx_spmm_bsr": ([i32, i32, i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, vp], ctypes.c_int),
        "spx_build_wcsr": ([i32, i32, vp, vp, vp, i32, vp, vp, vp, ctypes.POINTER(ctypes.c_int64), d,
                            ctypes.c_int, vp], ctypes.c_int),
        "spx_spmm_wcsr": ([i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, vp], ctypes.c_int),
        "spx_wcsr_plan_build": ([i32, i64, vp, ctypes.c_int, i32, ctypes.POINTER(vp)], ctypes.c_int),
        "spx_wcsr_plan_info": ([vp, ctypes.POINTER(WcsrPlanInfo)], ctypes.c_int),
        "spx_wcsr_plan_get_tasks": ([vp, vp, vp], ctypes.c_int),
        "spx_wcsr_plan_upload": ([vp, vp, sz, vp], ctypes.c_int),
        "spx_wcsr_plan_destroy": ([vp], ctypes.c_int),
        "spx_spmm_wcsr_planned_scratch_bytes": ([vp, i32], sz),
        "spx_spmm_wcsr_planned": ([vp, i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, vp, sz, vp],
                                  ctypes.c_int),
        "spx_bsr_plan_build": ([i32, i64, vp, ctypes.c_int, i32, ctypes.POINTER(vp)], ctypes.c_int),
        "spx_spmm_bsr_planned_scratch_bytes": ([vp, i32], sz),
        "spx_spmm_bsr_planned": ([vp, i32, i32, i32, i32, i64, vp, vp, vp, i32, vp, i64, f32, f32, vp, i64, vp, sz,
                                  vp], ctypes.c_int),
        "spx_gather_probe_blocks": ([], ctypes.c_int32),
        "spx_gather_probe": ([i64, vp, vp, vp, i32, vp, i32, vp], ctypes.c_int),
        "spx_last_device_error": ([vp], ctypes.c_int),
        "spx_wait_probe": ([i64, vp], ctypes.c_int),
    }
    for name, (args, res) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def header_symbols() -> list[str]:
    """Function names declared in include/spx.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(spx_\w+)\s*\(", text, re.M)))


def _check(rc: int, where: str):
    if rc != 0:
        raise SpxError(rc, where)


def _ptr(t):
    """Address of an array's first element.  The library reads arrays densely,
    except the rows of 2-D operands, whose leading dimension is passed apart:
    anything else (a transposed or sliced view) is rejected, not copied."""
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        if not t.numel():
            return None
        if not (t.is_contiguous() or (t.dim() == 2 and t.stride(1) == 1)):
            raise ValueError(f"array with strides {tuple(t.stride())} is not laid out densely")
        return t.data_ptr()  # a plain address: the c_void_p argtypes take ints without building objects
    if isinstance(t, np.ndarray):
        if not t.size:
            return None
        if not (t.flags.c_contiguous or (t.ndim == 2 and t.strides[1] == t.itemsize)):
            raise ValueError(f"array with strides {t.strides} is not laid out densely")
        return t.ctypes.data  # the caller keeps the array alive for the call
    raise TypeError(type(t))


def _require(cond: bool, what: str):
    if not cond:
        raise ValueError(what)


_CUDA_OK = None


def _stream(stream=None):
    global _CUDA_OK
    if stream is None:
        if _CUDA_OK is None:
            _CUDA_OK = torch.cuda.is_available()
        if not _CUDA_OK:
            return None
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None  # the raw handle (0: the legacy default stream)


def _where(*arrays) -> int:
    dev = [isinstance(a, torch.Tensor) and a.is_cuda for a in arrays if a is not None]
    if any(dev) and not all(dev):
        raise ValueError("mix of host and device arrays")
    return SPX_DEVICE if dev and all(dev) else SPX_HOST


def _empty_like_loc(ref, n, dtype_np, dtype_t):
    if isinstance(ref, torch.Tensor) and ref.is_cuda:
        return torch.empty(int(n), dtype=dtype_t, device=ref.device)
    return np.empty(int(n), dtype=dtype_np)


_TDT = {np.dtype(np.float32): torch.float32, np.dtype(np.float64): torch.float64,
        np.dtype(np.uint16): torch.int16, np.dtype(np.int16): torch.int16, np.dtype(np.int32): torch.int32}


def _itemsize(a) -> int:
    return a.element_size() if isinstance(a, torch.Tensor) else a.itemsize


def launch_count() -> int:
    c = ctypes.c_uint64(0)
    _check(_lib().spx_launch_count(ctypes.byref(c)), "spx_launch_count")
    return c.value


# ------------------------------------------------------------------ builders

def spx_build_csr(M: int, K: int, coo_row, coo_col, coo_val, stream=None):
    """COO -> CSR; arrays all host (numpy) or all device (torch cuda)."""
    where = _where(coo_row, coo_col, coo_val)
    nnz = coo_row.numel() if isinstance(coo_row, torch.Tensor) else coo_row.size
    vb = _itemsize(coo_val)
    rp = _empty_like_loc(coo_row, M + 1, np.int32, torch.int32)
    col = _empty_like_loc(coo_row, nnz, np.int32, torch.int32)
    if isinstance(coo_val, torch.Tensor):
        val = torch.empty(nnz, dtype=coo_val.dtype, device=coo_val.device)
    else:
        val = np.empty(nnz, dtype=coo_val.dtype)
    _check(_lib().spx_build_csr(M, K, nnz, _ptr(coo_row), _ptr(coo_col), _ptr(coo_val), vb, _ptr(rp), _ptr(col),
                                _ptr(val), where, _stream(stream) if where == SPX_DEVICE else None), "spx_build_csr")
    return rp, col, val


def spx_transpose_csr(M: int, K: int, row_ptr, col, val, stream=None):
    where = _where(row_ptr, col, val)
    nnz = col.numel() if isinstance(col, torch.Tensor) else col.size
    trp = _empty_like_loc(row_ptr, K + 1, np.int32, torch.int32)
    tcol = _empty_like_loc(row_ptr, nnz, np.int32, torch.int32)
    if isinstance(val, torch.Tensor):
        tval = torch.empty(nnz, dtype=val.dtype, device=val.device)
    else:
        tval = np.empty(nnz, dtype=val.dtype)
    _check(_lib().spx_transpose_csr(M, K, nnz, _ptr(row_ptr), _ptr(col), _ptr(val), _itemsize(val), _ptr(trp),
                                    _ptr(tcol), _ptr(tval), where, _stream(stream) if where == SPX_DEVICE else None),
           "spx_transpose_csr")
    return trp, tcol, tval


def spx_build_bsr(M: int, K: int, row_ptr, col, val, br: int, bc: int, stream=None):
    """CSR -> BSR (two calls).  Returns (bsr_row_ptr, bsr_col, bsr_val[nnzb, br, bc], fill)."""
    where = _where(row_ptr, col, val)
    lib = _lib()
    MB = (M + br - 1) // br
    nnzb = ctypes.c_int64(0)
    fill = ctypes.c_double(0.0)
    st = _stream(stream) if where == SPX_DEVICE else None
    brp = _empty_like_loc(row_ptr, MB + 1, np.int32, torch.int32)
    _check(lib.spx_build_bsr(M, K, _ptr(row_ptr), _ptr(col), _ptr(val), _itemsize(val), br, bc, _ptr(brp), None,
                             None, ctypes.byref(nnzb), ctypes.byref(fill), where, st), "spx_build_bsr(count)")
    nb = nnzb.value
    bcol = _empty_like_loc(row_ptr, nb, np.int32, torch.int32)
    if isinstance(val, torch.Tensor):
        bval = torch.empty(nb * br * bc, dtype=val.dtype, device=val.device)
    else:
        bval = np.empty(nb * br * bc, dtype=val.dtype)
    if nb:
        _check(lib.spx_build_bsr(M, K, _ptr(row_ptr), _ptr(col), _ptr(val), _itemsize(val), br, bc, None,
                                 _ptr(bcol), _ptr(bval), ctypes.byref(nnzb), ctypes.byref(fill), where, st),
               "spx_build_bsr")
    return brp, bcol, bval.reshape(nb, br, bc), fill.value


def spx_build_wcsr(M: int, K: int, row_ptr, col, val, stream=None):
    """CSR -> WCSR with 64-row windows (two calls).
    Returns (win_ptr, win_col[nchunks*64], win_val[nchunks, 64, 64], fill)."""
    where = _where(row_ptr, col, val)
    lib = _lib()
    W = (M + 63) // 64
    nch = ctypes.c_int64(0)
    fill = ctypes.c_double(0.0)
    st = _stream(stream) if where == SPX_DEVICE else None
    wp = _empty_like_loc(row_ptr, W + 1, np.int32, torch.int32)
    _check(lib.spx_build_wcsr(M, K, _ptr(row_ptr), _ptr(col), _ptr(val), _itemsize(val), _ptr(wp), None, None,
                              ctypes.byref(nch), ctypes.byref(fill), where, st), "spx_build_wcsr(count)")
    nc = nch.value
    wc = _empty_like_loc(row_ptr, nc * 64, np.int32, torch.int32)
    if isinstance(val, torch.Tensor):
        wv = torch.empty(nc * 4096, dtype=val.dtype, device=val.device)
    else:
        wv = np.empty(nc * 4096, dtype=val.dtype)
    if nc:
        _check(lib.spx_build_wcsr(M, K, _ptr(row_ptr), _ptr(col), _ptr(val), _itemsize(val), None, _ptr(wc),
                                  _ptr(wv), ctypes.byref(nch), ctypes.byref(fill), where, st), "spx_build_wcsr")
    return wp, wc, wv.reshape(nc, 64, 64), fill.value


def spx_spmm_wcsr(M: int, K: int, win_ptr: torch.Tensor, win_col: torch.Tensor, win_val: torch.Tensor,
                  B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C <- alpha*A*B + beta*C, A in WCSR (bf16 bit patterns), B bf16 (K x N), C fp32 (M x N)."""
    N = B.shape[1]
    _require(B.dim() == 2 and C.dim() == 2 and B.stride(1) == 1 and C.stride(1) == 1,
             "B and C must be 2-D with unit column stride")
    nch = win_col.numel() // 64
    _check(_lib().spx_spmm_wcsr(M, K, nch, _ptr(win_ptr), _ptr(win_col), _ptr(win_val), N, _ptr(B), B.stride(0),
                                float(alpha), float(beta), _ptr(C), C.stride(0), _stream(stream)), "spx_spmm_wcsr")
    return C


class WcsrPlan:
    """Owns an spx_wcsr_plan* (the WCSR task split) and its uploaded device table."""

    _build = "spx_wcsr_plan_build"

    def __init__(self, M: int, nchunks: int, win_ptr, max_chunks: int = 0, device=None, upload=True, stream=None):
        lib = _lib()
        self._owner = lib  # the library that made this object also releases it
        h = ctypes.c_void_p()
        _check(getattr(lib, self._build)(M, nchunks, _ptr(win_ptr), _where(win_ptr), int(max_chunks), ctypes.byref(h)),
               self._build)
        self.handle, self.M, self.nchunks = h, M, nchunks
        info = WcsrPlanInfo()
        _check(lib.spx_wcsr_plan_info(h, ctypes.byref(info)), "spx_wcsr_plan_info")
        self.info = {f: getattr(info, f) for f, _ in WcsrPlanInfo._fields_}
        self.table = None
        if upload:
            dev = device or (win_ptr.device if isinstance(win_ptr, torch.Tensor) and win_ptr.is_cuda else "cuda")
            self.table = torch.empty(max(4, (self.info["table_bytes"] + 15) // 16 * 4), dtype=torch.int32, device=dev)
            _check(lib.spx_wcsr_plan_upload(h, _ptr(self.table), self.table.numel() * 4, _stream(stream)),
                   "spx_wcsr_plan_upload")

    def tasks(self):
        t = np.empty((self.info["tasks"], 4), np.int32)
        sp = np.empty((self.info["split_windows"], 4), np.int32)
        _check(_lib().spx_wcsr_plan_get_tasks(self.handle, _ptr(t), _ptr(sp)), "spx_wcsr_plan_get_tasks")
        return t, sp

    def close(self):
        if self.handle:
            self._owner.spx_wcsr_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BsrPlan(WcsrPlan):
    """The task split of BSR block-rows (spx_bsr_plan_build): same object as WcsrPlan,
    built from bsr_row_ptr with nnzb blocks and max_blocks (0: 64)."""
    _build = "spx_bsr_plan_build"


def spx_spmm_bsr_planned(plan: BsrPlan, M: int, K: int, br: int, bc: int, bsr_row_ptr: torch.Tensor,
                         bsr_col: torch.Tensor, bsr_val: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
                         alpha: float = 1.0, beta: float = 0.0, stream=None, scratch: torch.Tensor | None = None):
    """spx_spmm_bsr with the plan's long block-rows split (partial tiles + fixed-order fix-up)."""
    N = B.shape[1]
    _require(B.dim() == 2 and C.dim() == 2 and B.stride(1) == 1 and C.stride(1) == 1,
             "B and C must be 2-D with unit column stride")
    lib = _lib()
    need = int(lib.spx_spmm_bsr_planned_scratch_bytes(plan.handle, N))
    if scratch is None:
        scratch = torch.empty(max(4, (need + 15) // 16 * 4), dtype=torch.float32, device=C.device)
    _check(lib.spx_spmm_bsr_planned(plan.handle, M, K, br, bc, bsr_col.numel(), _ptr(bsr_row_ptr), _ptr(bsr_col),
                                    _ptr(bsr_val), N, _ptr(B), B.stride(0), float(alpha), float(beta), _ptr(C),
                                    C.stride(0), _ptr(scratch), scratch.numel() * scratch.element_size(),
                                    _stream(stream)), "spx_spmm_bsr_planned")
    return C


def spx_spmm_wcsr_planned(plan: WcsrPlan, M: int, K: int, win_ptr: torch.Tensor, win_col: torch.Tensor,
                          win_val: torch.Tensor, B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0,
                          beta: float = 0.0, stream=None, scratch: torch.Tensor | None = None):
    """spx_spmm_wcsr with the plan's wide windows split into pieces (partial tiles + fixed-order fix-up)."""
    N = B.shape[1]
    _require(B.dim() == 2 and C.dim() == 2 and B.stride(1) == 1 and C.stride(1) == 1,
             "B and C must be 2-D with unit column stride")
    lib = _lib()
    need = int(lib.spx_spmm_wcsr_planned_scratch_bytes(plan.handle, N))
    if scratch is None:
        scratch = torch.empty(max(4, (need + 15) // 16 * 4), dtype=torch.float32, device=C.device)
    nch = win_col.numel() // 64
    _check(lib.spx_spmm_wcsr_planned(plan.handle, M, K, nch, _ptr(win_ptr), _ptr(win_col), _ptr(win_val), N, _ptr(B),
                                     B.stride(0), float(alpha), float(beta), _ptr(C), C.stride(0), _ptr(scratch),
                                     scratch.numel() * scratch.element_size(), _stream(stream)),
           "spx_spmm_wcsr_planned")
    return C


def spx_check_csr(M: int, K: int, row_ptr, col, strict: bool = True, stream=None) -> int:
    """Returns the spx_status of the structural check (0 == valid)."""
    where = _where(row_ptr, col)
    nnz = col.numel() if isinstance(col, torch.Tensor) else col.size
    return _lib().spx_check_csr(M, K, nnz, _ptr(row_ptr), _ptr(col), int(strict), where,
                                _stream(stream) if where == SPX_DEVICE else None)


def spx_row_stats(M: int, row_ptr) -> dict:
    st = RowStats()
    _check(_lib().spx_row_stats(M, _ptr(row_ptr), _where(row_ptr), ctypes.byref(st)), "spx_row_stats")
    return st.as_dict()


def spx_plan_opts_default() -> dict:
    o = PlanOpts()
    _check(_lib().spx_plan_opts_default(ctypes.byref(o)), "spx_plan_opts_default")
    return {f: getattr(o, f) for f, _ in PlanOpts._fields_}


# ------------------------------------------------------------------ plan

class Plan:
    """Owns an spx_plan*, its device table and its scratch (torch tensors)."""

    def __init__(self, M: int, K: int, nnz: int, row_ptr, opts: dict | None = None, device=None, upload=True,
                 stream=None):
        lib = _lib()
        self._owner = lib  # the library that made this object also releases it
        o = None
        if opts:
            base = spx_plan_opts_default()
            base.update(opts)
            o = PlanOpts(**base)
        self.opts_given = dict(opts) if opts else None
        h = ctypes.c_void_p()
        _check(lib.spx_plan_csr(M, K, nnz, _ptr(row_ptr), _where(row_ptr), ctypes.byref(o) if o else None,
                                ctypes.byref(h)), "spx_plan_csr")
        self.handle = h
        self.M, self.K, self.nnz = M, K, nnz
        info = PlanInfo()
        _check(lib.spx_plan_get_info(h, ctypes.byref(info)), "spx_plan_get_info")
        self.info = {f: getattr(info, f) for f, _ in PlanInfo._fields_ if f not in ("stats", "opts")}
        self.stats = info.stats.as_dict()
        self.opts = {f: getattr(info.opts, f) for f, _ in PlanOpts._fields_}
        self.table = None
        self.scratch = None
        if upload:
            dev = device or (row_ptr.device if isinstance(row_ptr, torch.Tensor) and row_ptr.is_cuda else "cuda")
            self.table = torch.empty(max(1, (self.info["table_bytes"] + 15) // 16 * 4), dtype=torch.int32,
                                     device=dev)
            self.scratch = torch.empty(max(1, self.info["scratch_bytes"] // 4), dtype=torch.float32, device=dev)
            _check(lib.spx_plan_upload(h, _ptr(self.table), self.table.numel() * 4, _stream(stream)),
                   "spx_plan_upload")

    @property
    def fingerprint(self) -> int:
        """Structure fingerprint of the row_ptr the plan was built from (spx_plan_fingerprint)."""
        f = ctypes.c_uint64()
        _check(_lib().spx_plan_fingerprint(self.handle, ctypes.byref(f)), "spx_plan_fingerprint")
        return f.value

    def validate(self, row_ptr, stream=None) -> int:
        """spx_status of spx_plan_validate for this row_ptr (0: the plan still fits; -1: stale)."""
        where = _where(row_ptr)
        return _lib().spx_plan_validate(self.handle, self.M, self.K, self.nnz, _ptr(row_ptr), where,
                                        _stream(stream) if where == SPX_DEVICE else None)

    def tasks(self):
        t = np.empty((self.info["tasks"], 4), np.int32)
        lr = np.empty((self.info["long_rows"], 4), np.int32)
        _check(_lib().spx_plan_get_tasks(self.handle, _ptr(t), _ptr(lr)), "spx_plan_get_tasks")
        return t, lr

    def device_table(self) -> np.ndarray:
        """Host copy of the bytes spx_plan_upload writes (spx_plan_get_table), as uint8."""
        b = np.zeros(self.info["table_bytes"], np.uint8)
        _check(_lib().spx_plan_get_table(self.handle, _ptr(b) if b.size else None), "spx_plan_get_table")
        return b

    def first_rows(self) -> np.ndarray:
        """The per-thread first-row entries of the segmented groups (uint16, one row per group;
        empty when the plan's groups are not segmented)."""
        if self.opts["lanes_div"] != 0:
            return np.zeros((0, 0), np.uint16)
        B = self.opts["block_nnz"]
        T = B // 8 if B in (512, 1024, 2048, 4096) else 256
        off = 16 * (self.info["tasks"] + self.info["long_rows"])
        return self.device_table()[off:].view(np.uint16).reshape(-1, T)

    def close(self):
        if self.handle:
            self._owner.spx_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def spx_plan_csr(M: int, K: int, nnz: int, row_ptr, opts: dict | None = None, **kw) -> Plan:
    return Plan(M, K, nnz, row_ptr, opts, **kw)


class Sell:
    """Owns an spx_sell* (SELL-C-sigma form of a CSR), its device image and scratch."""

    def __init__(self, M: int, K: int, row_ptr, col, val, opts: dict | None = None, upload=True, device=None,
                 stream=None):
        lib = _lib()
        self._owner = lib  # the library that made this object also releases it
        o = None
        if opts:
            base = SellOpts()
            _check(lib.spx_sell_opts_default(ctypes.byref(base)), "spx_sell_opts_default")
            d = {f: getattr(base, f) for f, _ in SellOpts._fields_}
            d.update(opts)
            o = SellOpts(**d)
        h = ctypes.c_void_p()
        nnz = col.numel() if isinstance(col, torch.Tensor) else int(np.asarray(col).size)
        _check(lib.spx_sell_build(M, K, nnz, _ptr(row_ptr), _ptr(col), _ptr(val), _where(row_ptr, col, val),
                                  ctypes.byref(o) if o else None, ctypes.byref(h)), "spx_sell_build")
        self.handle = h
        self.M, self.K, self.nnz = M, K, nnz
        info = SellInfo()
        _check(lib.spx_sell_get_info(h, ctypes.byref(info)), "spx_sell_get_info")
        self.info = {f: getattr(info, f) for f, _ in SellInfo._fields_ if f != "opts"}
        self.opts = {f: getattr(info.opts, f) for f, _ in SellOpts._fields_}
        self.image = None
        self.scratch = None
        if upload:
            dev = device or (row_ptr.device if isinstance(row_ptr, torch.Tensor) and row_ptr.is_cuda else "cuda")
            self.image = torch.empty(max(1, (self.info["image_bytes"] + 15) // 16 * 4), dtype=torch.int32,
                                     device=dev)
            self.scratch = torch.empty(max(1, self.info["scratch_bytes"] // 4), dtype=torch.float32, device=dev)
            _check(lib.spx_sell_upload(h, _ptr(self.image), self.image.numel() * 4, _stream(stream)),
                   "spx_sell_upload")

    def arrays(self):
        i = self.info
        sp = np.empty(i["slices"] + 1, np.int32)
        pr = np.empty(32 * i["slices"], np.int32)
        lr = np.empty((i["long_rows"], 4), np.int32)
        sc = np.empty(i["padded"], np.int32)
        sv = np.empty(i["padded"], np.float32)
        _check(_lib().spx_sell_get_arrays(self.handle, _ptr(sp), _ptr(pr), _ptr(lr), _ptr(sc), _ptr(sv)),
               "spx_sell_get_arrays")
        return sp, pr, lr, sc, sv

    def close(self):
        if self.handle:
            self._owner.spx_sell_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def spx_spmv_sell(S: Sell, x: torch.Tensor, y: torch.Tensor, alpha: float = 1.0, beta: float = 0.0, stream=None,
                  scratch: torch.Tensor | None = None):
    """y <- alpha*A*x + beta*y with A in uploaded SELL-C-sigma form (scratch: the form's own by default)."""
    sc = S.scratch if scratch is None else scratch
    _check(_lib().spx_spmv_sell(S.handle, S.M, S.K, float(alpha), _ptr(x), float(beta), _ptr(y), _ptr(sc),
                                sc.numel() * 4, _stream(stream)), "spx_spmv_sell")
    return y


def spx_plan_autotune(A: "Csr", row_ptr_host, x: torch.Tensor, candidates: list[dict] | None = None, reps: int = 5,
                      stream=None, y_scratch: torch.Tensor | None = None):
    """Time candidate plan options on the device (cached per matrix profile).
    Returns (best options dict, per-candidate mean ms or -1 when cached, cached flag)."""
    rp = np.ascontiguousarray(row_ptr_host, dtype=np.int32)
    n = len(candidates) if candidates else 4
    cand = None
    if candidates:
        arr = (PlanOpts * n)()
        for i, c in enumerate(candidates):
            base = spx_plan_opts_default()
            base.update(c)
            arr[i] = PlanOpts(**base)
        cand = arr
    ys = torch.empty(max(A.M, 1), dtype=torch.float32, device=x.device) if y_scratch is None else y_scratch
    best = PlanOpts()
    times = (ctypes.c_float * n)()
    cached = ctypes.c_int32(0)
    _check(_lib().spx_plan_autotune(A.M, A.K, A.nnz, _ptr(rp), _ptr(A.row_ptr), _ptr(A.col), _ptr(A.val),
                                    _ptr(x), _ptr(ys), cand, n if cand is not None else 0, int(reps),
                                    _stream(stream), ctypes.byref(best), times, ctypes.byref(cached)),
           "spx_plan_autotune")
    return {f: getattr(best, f) for f, _ in PlanOpts._fields_}, [float(t) for t in times], bool(cached.value)


def spx_plan_autotune_forget():
    _check(_lib().spx_plan_autotune_forget(), "spx_plan_autotune_forget")


@dataclass
class Csr:
    """A CSR matrix held as device tensors (int32 row_ptr/col, fp32 val)."""
    M: int
    K: int
    row_ptr: torch.Tensor
    col: torch.Tensor
    val: torch.Tensor

    @property
    def nnz(self) -> int:
        return self.col.numel()


# ------------------------------------------------------------------ products

def spx_spmv_csr(plan: Plan, A: Csr, x: torch.Tensor, y: torch.Tensor, alpha: float = 1.0, beta: float = 0.0,
                 stream=None, scratch: torch.Tensor | None = None):
    """y <- alpha*A*x + beta*y (in place)."""
    sc = plan.scratch if scratch is None else scratch
    _check(_lib().spx_spmv_csr(plan.handle, A.M, A.K, A.nnz, _ptr(A.row_ptr), _ptr(A.col), _ptr(A.val),
                               float(alpha), _ptr(x), float(beta), _ptr(y), _ptr(sc), sc.numel() * 4,
                               _stream(stream)), "spx_spmv_csr")
    return y


def spx_spmv_csr_noalloc(plan: Plan, A: Csr, x: torch.Tensor, y: torch.Tensor, alpha: float = 1.0,
                         beta: float = 0.0, stream=None):
    """y <- alpha*A*x + beta*y without a caller scratch buffer, for callers that
    cannot allocate device memory: split-row partial sums use the library's
    fixed device array (see include/spx.h)."""
    _check(_lib().spx_spmv_csr_noalloc(plan.handle, A.M, A.K, A.nnz, _ptr(A.row_ptr), _ptr(A.col), _ptr(A.val),
                                       float(alpha), _ptr(x), float(beta), _ptr(y), _stream(stream)),
           "spx_spmv_csr_noalloc")
    return y


def spx_spmv_csr_hostio(plan: Plan, A: Csr, x_host: torch.Tensor, y_host: torch.Tensor, alpha: float = 1.0,
                        beta: float = 0.0, work: torch.Tensor | None = None, stream=None):
    """y_host[b] <- alpha*A*x_host[b] + beta*y_host[b] for every row b of the (batch x K) / (batch x M)
    host tensors (pinned for full speed); copies pipelined against the products.  Synchronises."""
    _require(not x_host.is_cuda and not y_host.is_cuda and x_host.dim() == 2 and y_host.dim() == 2,
             "x_host and y_host must be 2-D host tensors")
    _require(x_host.stride(1) == 1 and y_host.stride(1) == 1, "x_host and y_host need unit column stride")
    _require(x_host.shape[0] in (1, y_host.shape[0]), "x_host needs one row, or one row per batch")
    need = int(_lib().spx_spmv_csr_hostio_work_bytes(A.M, A.K))
    if work is None:
        work = torch.empty(max(1, need // 4), dtype=torch.float32, device=plan.table.device)
    sc = plan.scratch
    _check(_lib().spx_spmv_csr_hostio(plan.handle, A.M, A.K, A.nnz, _ptr(A.row_ptr), _ptr(A.col), _ptr(A.val),
                                      float(alpha), _ptr(x_host), x_host.stride(0) if x_host.shape[0] > 1 else 0,
                                      float(beta), _ptr(y_host), y_host.stride(0), y_host.shape[0], _ptr(work),
                                      work.numel() * 4, _ptr(sc),
                                      sc.numel() * 4, _stream(stream)), "spx_spmv_csr_hostio")
    (stream or torch.cuda.current_stream()).synchronize()
    return y_host


def spx_spmv_coo_scratch_bytes(nnz: int) -> int:
    return int(_lib().spx_spmv_coo_scratch_bytes(int(nnz)))


def spx_spmv_coo(M: int, K: int, row: torch.Tensor, col: torch.Tensor, val: torch.Tensor, x: torch.Tensor,
                 y: torch.Tensor, alpha: float = 1.0, beta: float = 0.0, stream=None,
                 scratch: torch.Tensor | None = None):
    """y <- alpha*A*x + beta*y for A given as row-sorted COO device tensors (int32 row/col, fp32 val)."""
    nnz = col.numel()
    need = spx_spmv_coo_scratch_bytes(nnz)
    if scratch is None:
        scratch = torch.empty(max(1, need // 4), dtype=torch.float32, device=y.device)
    _check(_lib().spx_spmv_coo(M, K, nnz, _ptr(row), _ptr(col), _ptr(val), float(alpha), _ptr(x), float(beta),
                               _ptr(y), _ptr(scratch), scratch.numel() * 4, _stream(stream)), "spx_spmv_coo")
    return y


def spx_spmv_csr_dual(plan_A: Plan, plan_At: Plan, A: Csr, At: Csr, v: torch.Tensor, u: torch.Tensor,
                      alpha_u: float, beta_u: float, alpha_v: float, beta_v: float, stream=None,
                      scratch: torch.Tensor | None = None):
    """u <- alpha_u*A v + beta_u*u, then v <- alpha_v*A^T u + beta_v*v (in place)."""
    if scratch is None:
        scratch = plan_A.scratch if plan_A.scratch.numel() >= plan_At.scratch.numel() else plan_At.scratch
    _check(_lib().spx_spmv_csr_dual(plan_A.handle, plan_At.handle, A.M, A.K, A.nnz, _ptr(A.row_ptr), _ptr(A.col),
                                    _ptr(A.val), _ptr(At.row_ptr), _ptr(At.col), _ptr(At.val), _ptr(v),
                                    float(alpha_u), float(beta_u), _ptr(u), float(alpha_v), float(beta_v),
                                    _ptr(scratch), scratch.numel() * 4, _stream(stream)), "spx_spmv_csr_dual")
    return u, v


def spx_spmm_csr(A: Csr, B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0, beta: float = 0.0, stream=None,
                 col_tile: int | None = None):
    """C <- alpha*A*B + beta*C; B (K x N) and C (M x N) row-major views (stride(1) == 1).
    col_tile: None = automatic (spx_spmm_csr), else spx_spmm_csr_tiled's column tile."""
    N = B.shape[1]
    _require(B.dim() == 2 and C.dim() == 2 and B.stride(1) == 1 and C.stride(1) == 1,
             "B and C must be 2-D with unit column stride")
    lib = _lib()
    args = (A.M, A.K, A.nnz, _ptr(A.row_ptr), _ptr(A.col), _ptr(A.val), N, _ptr(B), B.stride(0), float(alpha),
            float(beta), _ptr(C), C.stride(0))
    if col_tile is None:
        _check(lib.spx_spmm_csr(*args, _stream(stream)), "spx_spmm_csr")
    else:
        _check(lib.spx_spmm_csr_tiled(*args, int(col_tile), _stream(stream)), "spx_spmm_csr_tiled")
    return C


def spx_spmm_csr_bf16(A: Csr, B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C <- alpha*A*B + beta*C with A.val and B holding bf16 bit patterns (int16 tensors), C fp32."""
    N = B.shape[1]
    _require(B.dim() == 2 and C.dim() == 2 and B.stride(1) == 1 and C.stride(1) == 1,
             "B and C must be 2-D with unit column stride")
    _require(A.val.element_size() == 2 and B.element_size() == 2, "A values and B must be 16-bit (bf16 bit patterns)")
    _check(_lib().spx_spmm_csr_bf16(A.M, A.K, A.nnz, _ptr(A.row_ptr), _ptr(A.col), _ptr(A.val), N, _ptr(B),
                                    B.stride(0), float(alpha), float(beta), _ptr(C), C.stride(0), _stream(stream)),
           "spx_spmm_csr_bf16")
    return C


def spx_spmm_csr_f16(A: Csr, B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C <- alpha*A*B + beta*C with A.val and B holding fp16 values (float16 or int16 bit patterns), C fp32."""
    N = B.shape[1]
    _require(B.dim() == 2 and C.dim() == 2 and B.stride(1) == 1 and C.stride(1) == 1,
             "B and C must be 2-D with unit column stride")
    _require(A.val.element_size() == 2 and B.element_size() == 2, "A values and B must be 16-bit (fp16)")
    _check(_lib().spx_spmm_csr_f16(A.M, A.K, A.nnz, _ptr(A.row_ptr), _ptr(A.col), _ptr(A.val), N, _ptr(B),
                                   B.stride(0), float(alpha), float(beta), _ptr(C), C.stride(0), _stream(stream)),
           "spx_spmm_csr_f16")
    return C


def _spmm_planned(name: str, plan: Plan, A: Csr, B: torch.Tensor, C: torch.Tensor, alpha: float, beta: float,
                  stream, scratch):
    N = B.shape[1]
    _require(B.dim() == 2 and C.dim() == 2 and B.stride(1) == 1 and C.stride(1) == 1,
             "B and C must be 2-D with unit column stride")
    lib = _lib()
    need = int(lib.spx_spmm_csr_planned_scratch_bytes(plan.handle, N))
    if scratch is None:
        scratch = torch.empty(max(1, (need + 3) // 4), dtype=torch.float32, device=C.device)
    _check(getattr(lib, name)(plan.handle, A.M, A.K, A.nnz, _ptr(A.row_ptr), _ptr(A.col), _ptr(A.val), N, _ptr(B),
                              B.stride(0), float(alpha), float(beta), _ptr(C), C.stride(0), _ptr(scratch),
                              scratch.numel() * scratch.element_size(), _stream(stream)), name)
    return C


def spx_spmm_csr_planned(plan: Plan, A: Csr, B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0,
                         beta: float = 0.0, stream=None, scratch: torch.Tensor | None = None):
    """C <- alpha*A*B + beta*C with the plan's long rows split (CTA rows, segments + fix-up)."""
    return _spmm_planned("spx_spmm_csr_planned", plan, A, B, C, alpha, beta, stream, scratch)


def spx_spmm_csr_bf16_planned(plan: Plan, A: Csr, B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0,
                              beta: float = 0.0, stream=None, scratch: torch.Tensor | None = None):
    """spx_spmm_csr_planned with bf16 bit patterns for A.val and B."""
    _require(A.val.element_size() == 2 and B.element_size() == 2, "A values and B must be 16-bit (bf16)")
    return _spmm_planned("spx_spmm_csr_bf16_planned", plan, A, B, C, alpha, beta, stream, scratch)


def spx_spmm_csr_f16_planned(plan: Plan, A: Csr, B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0,
                             beta: float = 0.0, stream=None, scratch: torch.Tensor | None = None):
    """spx_spmm_csr_planned with fp16 values for A.val and B."""
    _require(A.val.element_size() == 2 and B.element_size() == 2, "A values and B must be 16-bit (fp16)")
    return _spmm_planned("spx_spmm_csr_f16_planned", plan, A, B, C, alpha, beta, stream, scratch)


def spx_spmm_csr_variant(B: torch.Tensor, C: torch.Tensor) -> str:
    v = _lib().spx_spmm_csr_variant(B.shape[1], _ptr(B), B.stride(0), _ptr(C), C.stride(0))
    return SPMM_VARIANTS[v]


def spx_spmm_bsr(M: int, K: int, br: int, bc: int, bsr_row_ptr, bsr_col, bsr_val, B: torch.Tensor,
                 C: torch.Tensor, stream=None, alpha: float = 1.0, beta: float = 0.0):
    """C <- alpha*A*B + beta*C, A BSR (bf16 blocks held as int16 bit patterns or bfloat16), B bf16, C fp32."""
    nnzb = bsr_col.numel()
    N = B.shape[1]
    _check(_lib().spx_spmm_bsr(M, K, br, bc, nnzb, _ptr(bsr_row_ptr), _ptr(bsr_col), _ptr(bsr_val), N, _ptr(B),
                               B.stride(0), float(alpha), float(beta), _ptr(C), C.stride(0), _stream(stream)),
           "spx_spmm_bsr")
    return C


def spx_gather_probe(A: Csr, x: torch.Tensor, partials: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The stream + gather floor kernel over A's col/val and x (see include/spx.h)."""
    nb = int(_lib().spx_gather_probe_blocks())
    if partials is None:
        partials = torch.empty(nb, dtype=torch.float32, device=x.device)
    _check(_lib().spx_gather_probe(A.nnz, _ptr(A.col), _ptr(A.val), _ptr(x), A.K, _ptr(partials), partials.numel(),
                                   _stream(stream)), "spx_gather_probe")
    return partials


def spx_wait_probe(limit_cycles: int, stream=None):
    """Arm a wait that nothing completes and let it run out after limit_cycles (see include/spx.h)."""
    _check(_lib().spx_wait_probe(int(limit_cycles), _stream(stream)), "spx_wait_probe")


def spx_last_device_error(stream=None) -> int:
    return _lib().spx_last_device_error(_stream(stream))
