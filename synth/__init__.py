"""Seeded synthetic inputs shaped like the workloads of the sparse x dense pages.

Both the oracle tests and the GPU path consume these arrays; this module holds
none of the products' arithmetic.  Matrices come out as COO triplets in
row-major order with distinct, sorted column indices per row -- turning them
into CSR/CSR(A^T)/BSR is the job of the builders under test.

The random numbers come from the counter-based SplitMix64 streams in
``synth.c``; every array is keyed by (seed, tag) and is the same on any host.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# stream tags (any distinct constants)
T_LEN, T_COL, T_VAL, T_X, T_Y, T_B, T_BLK, T_SCAL, T_PERM = range(101, 110)

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u64, _i64, _d = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double


def build(force: bool = False) -> str:
    """Compile libsynth.so with the host C compiler (plain C, no ISA flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            sig = {
                "synth_uniform_f32": ([_u64, _u64, _i64, _d, _d, _f32p], None),
                "synth_normal_f32": ([_u64, _u64, _i64, _d, _f32p], None),
                "synth_normal_bf16": ([_u64, _u64, _i64, _d, _u16p], None),
                "synth_f32_to_bf16": ([_i64, _f32p, _u16p], None),
                "synth_lengths_uniform": ([_u64, _u64, _i64, ctypes.c_int32, ctypes.c_int32, _i32p], _i64),
                "synth_lengths_poisson": ([_u64, _u64, _i64, _d, _i32p], _i64),
                "synth_lengths_zipf": ([_u64, _u64, _i64, _d, ctypes.c_int32, _d, _i32p,
                                        ctypes.POINTER(ctypes.c_double)], _i64),
                "synth_cols_uniform": ([_u64, _u64, _i64, _i64, _i32p, _i32p, _i32p], None),
                "synth_cols_band": ([_u64, _u64, _i64, _i64, _i32p, _i64, _d, _i64, _i64, _i32p, _i32p], None),
                "synth_cols_quads": ([_u64, _u64, _i64, _i64, _i32p, _i32p, _i32p], None),
                "synth_block_cols": ([_u64, _u64, _i64, _i64, _i64, _i32p], None),
                "synth_permutation": ([_u64, _u64, _i64, _i64p], None),
                "synth_raw": ([_u64, _u64, _u64], _u64),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


# ------------------------------------------------------------------ primitives

def uniform(seed: int, tag: int, n: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.float32)
    _load().synth_uniform_f32(seed, tag, int(n), lo, hi, out)
    return out


def normal_f32(seed: int, tag: int, n: int, sigma: float) -> np.ndarray:
    out = np.empty(int(n), dtype=np.float32)
    _load().synth_normal_f32(seed, tag, int(n), sigma, out)
    return out


def normal_bf16(seed: int, tag: int, n: int, sigma: float) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, sigma) draws, round-to-nearest-even."""
    out = np.empty(int(n), dtype=np.uint16)
    _load().synth_normal_bf16(seed, tag, int(n), sigma, out)
    return out


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32).ravel()
    out = np.empty(a.size, dtype=np.uint16)
    _load().synth_f32_to_bf16(a.size, a, out)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def lengths_uniform(seed: int, M: int, a: int, b: int, tag: int = T_LEN) -> np.ndarray:
    out = np.empty(int(M), dtype=np.int32)
    _load().synth_lengths_uniform(seed, tag, int(M), a, b, out)
    return out


def lengths_poisson(seed: int, M: int, lam: float, tag: int = T_LEN) -> np.ndarray:
    out = np.empty(int(M), dtype=np.int32)
    _load().synth_lengths_poisson(seed, tag, int(M), lam, out)
    return out


def lengths_zipf(seed: int, M: int, expo: float, lmax: int, mean: float, tag: int = T_LEN):
    out = np.empty(int(M), dtype=np.int32)
    s = ctypes.c_double(0.0)
    _load().synth_lengths_zipf(seed, tag, int(M), expo, int(lmax), mean, out, ctypes.byref(s))
    return out, s.value


def cols_uniform(seed: int, K: int, lengths: np.ndarray, tag: int = T_COL):
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    nnz = int(lengths.sum(dtype=np.int64))
    row = np.empty(nnz, dtype=np.int32)
    col = np.empty(nnz, dtype=np.int32)
    _load().synth_cols_uniform(seed, tag, lengths.size, int(K), lengths, row, col)
    return row, col


def cols_band(seed: int, K: int, lengths: np.ndarray, half: int, outlier: float, num: int, den: int,
              tag: int = T_COL):
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    nnz = int(lengths.sum(dtype=np.int64))
    row = np.empty(nnz, dtype=np.int32)
    col = np.empty(nnz, dtype=np.int32)
    _load().synth_cols_band(seed, tag, lengths.size, int(K), lengths, int(half), float(outlier),
                            int(num), int(den), row, col)
    return row, col


def cols_quads(seed: int, K: int, lengths: np.ndarray, tag: int = T_COL):
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    nnz = int(lengths.sum(dtype=np.int64))
    row = np.empty(nnz, dtype=np.int32)
    col = np.empty(nnz, dtype=np.int32)
    _load().synth_cols_quads(seed, tag, lengths.size, int(K), lengths, row, col)
    return row, col


def block_cols(seed: int, MB: int, KB: int, per_row: int, tag: int = T_BLK) -> np.ndarray:
    out = np.empty(int(MB) * int(per_row), dtype=np.int32)
    _load().synth_block_cols(seed, tag, int(MB), int(KB), int(per_row), out)
    return out.reshape(int(MB), int(per_row))


def permutation(seed: int, n: int, tag: int = T_PERM) -> np.ndarray:
    out = np.empty(int(n), dtype=np.int64)
    _load().synth_permutation(seed, tag, int(n), out)
    return out


def scalars(seed: int, n: int, lo: float, hi: float, tag: int = T_SCAL) -> np.ndarray:
    return uniform(seed, tag, n, lo, hi)


# ------------------------------------------------------------------ workloads

def random_coo(seed: int, M: int, K: int, lmin: int = 0, lmax: int = 8, values: str = "uniform"):
    """Small random matrix: row lengths uniform in [lmin, min(lmax, K)], distinct
    sorted columns.  values: 'uniform' (U[-1,1)), 'int' (small integers, so
    that fp64 sums are exact) or 'ones'."""
    lmax = min(lmax, K)
    lmin = min(lmin, lmax)
    lengths = lengths_uniform(seed, M, lmin, lmax)
    row, col = cols_uniform(seed, K, lengths)
    if values == "int":
        val = np.floor(uniform(seed, T_VAL, row.size, -4.0, 5.0)).astype(np.float32)
    elif values == "ones":
        val = np.ones(row.size, dtype=np.float32)
    else:
        val = uniform(seed, T_VAL, row.size)
    return dict(M=M, K=K, row=row, col=col, val=val, lengths=lengths)


def uniform_short_rows(seed: int = 1, M: int = 4096, K: int = 4096, lmin: int = 1, lmax: int = 16):
    """Uniform short rows: lengths U{lmin..lmax}, distinct sorted columns
    uniform over [0, K), values and x U[-1,1), y = 1*A*x + 0*y."""
    lengths = lengths_uniform(seed, M, lmin, lmax)
    row, col = cols_uniform(seed, K, lengths)
    return dict(name=f"uniform-rows {M}x{K} l~U{{{lmin}..{lmax}}}", M=M, K=K, row=row, col=col,
                val=uniform(seed, T_VAL, row.size), x=uniform(seed, T_X, K), y=uniform(seed, T_Y, M),
                alpha=1.0, beta=0.0, lengths=lengths)


def power_law_rows(seed: int = 2, M: int = 4_194_304, K: int | None = None, expo: float = 2.1,
                   lmax: int = 200_000, mean: float = 16.0):
    """Power-law rows: Zipf(expo) lengths clipped to [1, lmax] and rescaled to
    the given mean, distinct sorted uniform columns, values/x/y U[-1,1),
    y = 1*A*x + 0.5*y."""
    K = M if K is None else K
    lengths, s = lengths_zipf(seed, M, expo, lmax, mean)
    row, col = cols_uniform(seed, K, lengths)
    return dict(name=f"power-law {M}x{K} zipf({expo}) mean {mean}", M=M, K=K, row=row, col=col,
                val=uniform(seed, T_VAL, row.size), x=uniform(seed, T_X, K), y=uniform(seed, T_Y, M),
                alpha=1.0, beta=0.5, lengths=lengths, zipf_scale=s)


def banded_pair(seed: int = 3, m: int = 2_000_000, n: int = 1_000_000, lmin: int = 5, lmax: int = 15,
                half: int = 2048, outlier: float = 0.1, iters: int = 10):
    """Least-squares operator: m x n, lengths U{lmin..lmax}, columns in a band of
    width 2*half around floor(i*n/m) plus a fraction `outlier` of uniform
    columns; values, u0, v0 U[-1,1); per-iteration scalars alpha_k, beta_k
    U[0.5, 2)."""
    lengths = lengths_uniform(seed, m, lmin, lmax)
    row, col = cols_band(seed, n, lengths, half, outlier, n, m)
    sc = scalars(seed, 2 * iters, 0.5, 2.0).reshape(iters, 2)
    return dict(name=f"banded dual {m}x{n}", M=m, K=n, row=row, col=col, val=uniform(seed, T_VAL, row.size),
                u0=uniform(seed, T_Y, m), v0=uniform(seed, T_X, n), alphas=sc[:, 0].copy(),
                betas=sc[:, 1].copy(), lengths=lengths)


def clustered_spmm(seed: int = 4, M: int = 1_048_576, K: int | None = None, N: int = 32, lam: float = 32.0):
    """4x4-clustered Poisson rows with a dense row-major B (K x N), C = A*B."""
    K = M if K is None else K
    lengths = lengths_poisson(seed, M, lam)
    row, col = cols_quads(seed, K, lengths)
    return dict(name=f"clustered spmm {M}x{K} N={N}", M=M, K=K, N=N, row=row, col=col,
                val=uniform(seed, T_VAL, row.size), B=uniform(seed, T_B, K * N).reshape(K, N),
                alpha=1.0, beta=0.0, lengths=lengths)


def block_sparse(seed: int = 5, M: int = 16384, K: int | None = None, bs: int = 64, per_row: int = 26,
                 N: int = 1024, sigma_a: float = 0.02, sigma_b: float = 1.0):
    """Block-sparse weights: bs x bs dense blocks, `per_row` distinct block
    columns per block-row (uniform without replacement); entries bf16
    N(0, sigma_a); B is K x N bf16 N(0, sigma_b).  COO comes out row-major."""
    K = M if K is None else K
    MB, KB = M // bs, K // bs
    bcols = block_cols(seed, MB, KB, per_row)
    ar = np.arange(bs, dtype=np.int32)
    per_blockrow = (bcols[:, :, None] * bs + ar[None, None, :]).reshape(MB, per_row * bs)
    col = np.repeat(per_blockrow, bs, axis=0).reshape(-1)
    row = np.repeat(np.arange(M, dtype=np.int32), per_row * bs)
    val = normal_bf16(seed, T_VAL, row.size, sigma_a)
    Bm = normal_bf16(seed, T_B, K * N, sigma_b).reshape(K, N)
    return dict(name=f"bsr {M}x{K} {bs}x{bs} {per_row}/row N={N}", M=M, K=K, N=N, bs=bs, row=row, col=col,
                val_bf16=val, B_bf16=Bm, bcols=bcols)


def window_pool(seed: int = 6, M: int = 16384, K: int | None = None, win: int = 64, pool: int = 512,
                lmin: int = 32, lmax: int = 96, N: int = 1024, sigma_a: float = 0.02, sigma_b: float = 1.0):
    """Irregular sparsity with window locality: every window of `win` rows
    draws its own pool of `pool` distinct columns (the first `pool` of a
    permutation of K); each row takes l ~ U{lmin..lmax} distinct pool entries.
    Entries bf16 N(0, sigma_a), B is K x N bf16 N(0, sigma_b).  COO comes out
    sorted by (row, col)."""
    K = M if K is None else K
    W = (M + win - 1) // win
    lengths = lengths_uniform(seed, M, lmin, lmax)
    row, idx = cols_uniform(seed, pool, lengths)
    pools = np.stack([permutation(seed, K, tag=1000 + w)[:pool] for w in range(W)]).astype(np.int32)
    col = pools[row // win, idx]
    order = np.lexsort((col, row))
    row, col = row[order], col[order]
    val = normal_bf16(seed, T_VAL, row.size, sigma_a)
    Bm = normal_bf16(seed, T_B, K * N, sigma_b).reshape(K, N)
    return dict(name=f"window-pool {M}x{K} windows {win} pool {pool} l~U{{{lmin}..{lmax}}} N={N}", M=M, K=K, N=N,
                row=row, col=col, val_bf16=val, B_bf16=Bm)


def window_pool_skewed(seed: int = 7, M: int = 16384, K: int | None = None, win: int = 64, pool: int = 512,
                       big_pool: int = 8192, big_every: int = 16, lmin: int = 32, lmax: int = 96, N: int = 1024,
                       sigma_a: float = 0.02, sigma_b: float = 1.0):
    """window_pool with skewed windows: every `big_every`-th window draws its rows'
    columns from a pool of `big_pool` columns instead of `pool`, so its union of
    columns (and its WCSR chunk count) is many times larger."""
    K = M if K is None else K
    pool, big_pool = min(pool, K), min(big_pool, K)
    W = (M + win - 1) // win
    lengths = lengths_uniform(seed, M, lmin, min(lmax, pool))
    big = (np.arange(M) // win) % big_every == 0
    rs, ids = cols_uniform(seed, pool, np.where(big, 0, lengths).astype(np.int32))
    rb, idb = cols_uniform(seed + 1, big_pool, np.where(big, lengths, 0).astype(np.int32))
    pools = np.stack([permutation(seed, K, tag=1000 + w)[:pool] for w in range(W)]).astype(np.int32)
    bigw = np.arange(0, W, big_every)
    bpools = np.zeros((W, big_pool), np.int32)
    for w in bigw:
        bpools[w] = permutation(seed, K, tag=5000 + int(w))[:big_pool]
    row = np.concatenate([rs, rb])
    col = np.concatenate([pools[rs // win, ids], bpools[rb // win, idb]])
    order = np.lexsort((col, row))
    row, col = row[order].astype(np.int32), col[order].astype(np.int32)
    val = normal_bf16(seed, T_VAL, row.size, sigma_a)
    Bm = normal_bf16(seed, T_B, K * N, sigma_b).reshape(K, N)
    return dict(name=f"window-pool skewed {M}x{K} windows {win} pools {pool}/{big_pool} (every {big_every}th) "
                     f"l~U{{{lmin}..{lmax}}} N={N}", M=M, K=K, N=N, row=row, col=col, val_bf16=val, B_bf16=Bm)


def block_sparse_skewed(seed: int = 9, M: int = 16384, K: int | None = None, bs: int = 64, per_row: int = 26,
                        big_per_row: int = 208, big_every: int = 16, N: int = 1024, sigma_a: float = 0.02,
                        sigma_b: float = 1.0):
    """block_sparse with skewed block-rows: every `big_every`-th block-row holds
    `big_per_row` blocks instead of `per_row` (distinct block columns, uniform)."""
    K = M if K is None else K
    MB, KB = M // bs, K // bs
    per_row, big_per_row = min(per_row, KB), min(big_per_row, KB)
    small = block_cols(seed, MB, KB, per_row)
    big = block_cols(seed + 1, MB, KB, big_per_row)
    ar = np.arange(bs, dtype=np.int32)
    rows, cols = [], []
    for I in range(MB):
        bc = big[I] if I % big_every == 0 else small[I]
        per_blockrow = (bc[:, None] * bs + ar[None, :]).reshape(-1)
        cols.append(np.tile(per_blockrow, bs))
        rows.append(np.repeat(np.arange(I * bs, (I + 1) * bs, dtype=np.int32), per_blockrow.size))
    row, col = np.concatenate(rows), np.concatenate(cols).astype(np.int32)
    val = normal_bf16(seed, T_VAL, row.size, sigma_a)
    Bm = normal_bf16(seed, T_B, K * N, sigma_b).reshape(K, N)
    return dict(name=f"bsr skewed {M}x{K} {bs}x{bs} {per_row}/row, {big_per_row} every {big_every}th N={N}", M=M,
                K=K, N=N, bs=bs, row=row, col=col, val_bf16=val, B_bf16=Bm)
