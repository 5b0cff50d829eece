// spx_build.cu -- format builders on the GPU: COO -> CSR, CSR -> CSR(A^T),
// CSR -> BSR and CSR -> WCSR.
//
// [Formats] §3 (COO -> CSR: histogram of the row indices, prefix sum, stable
// scatter, entries of a row in column order) and [LSMR-dual] §2, §4 (CSR(A^T)
// = CSC(A): a counting sort by column that keeps rows ascending inside each
// output row).  Both are stable sorts of the entries by an integer key, done
// here as an LSD radix sort with 8-bit digits:
//   per tile of 2048 keys, a 256-bin histogram (shared-memory integer
//   atomics -- exact counts); an exclusive scan over (digit, tile); a scatter
//   that ranks each key among equal digits in input order (warp match + per-
//   warp counts), so every pass is stable and the result is the unique
//   stable order.
// COO -> CSR sorts by column, then by row (LSD over the pair); CSR -> CSR(A^T)
// sorts by column only (the entries already come in row order).  CSR -> BSR
// ([AsyncSparse] §2.2.1: every block holding an entry, stored dense, block
// columns ascending in a block-row) sorts by (block row, block column, place
// in the block); a scan of the block starts numbers the blocks, and each entry
// is scattered into its zeroed block.  CSR -> WCSR ([AsyncSparse] §2.2.2: per
// 64-row window the ascending union of its columns, cut into chunks of 64
// compressed columns) sorts by (window, column, row in the window); a scan of
// the (window, column) starts gives each column its compressed position.  The sort
// carries each entry's source index; columns and values (1, 2, 4 or 8 bytes)
// are gathered through it at the end.  Row offsets come from exact per-row
// counts and a scan.  Indices are validated first (SPX_ERR_INDEX_RANGE, like
// the host builders).  Temporary device memory is taken from the stream-
// ordered allocator and returned before the call ends.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>
#include <utility>
#include <vector>

#include "spx_internal.h"

namespace {

constexpr int kT = 256;              // threads per CTA
constexpr int kPer = 8;              // keys per thread per tile
constexpr int kTile = kT * kPer;     // 2048 keys per tile
constexpr int kScanBlock = 2048;     // elements per scan block (256 threads x 8)

// ---------------------------------------------------------------- validation
__global__ void check_indices(const int* __restrict__ a, long long n, int lim, int* __restrict__ bad) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int v = a[i];
        if (v < 0 || v >= lim) atomicOr(bad, 1);
    }
}

// row_ptr must start at 0, end at nnz and never decrease.
__global__ void check_row_ptr(const int* __restrict__ rp, int M, long long nnz, int* __restrict__ bad) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < M;
         i += static_cast<long long>(gridDim.x) * kT)
        if (rp[i + 1] < rp[i]) atomicOr(bad, 2);
    if (blockIdx.x == 0 && threadIdx.x == 0 && (rp[0] != 0 || static_cast<long long>(rp[M]) != nnz)) atomicOr(bad, 4);
}

// ---------------------------------------------------------------- scan (exclusive, uint32)
// Block b scans in[b*2048 .. +2048) into out and writes its total to sums[b].
__global__ void __launch_bounds__(kT) scan_blocks(const uint32_t* __restrict__ in, uint32_t* __restrict__ out,
                                                  long long n, uint32_t* __restrict__ sums) {
    __shared__ uint32_t s_w[kT / 32];
    const long long base = blockIdx.x * static_cast<long long>(kScanBlock) + threadIdx.x * kPer;
    uint32_t v[kPer], t = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        v[j] = base + j < n ? in[base + j] : 0u;
        t += v[j];
    }
    // exclusive scan of the per-thread totals across the block
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = t;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    uint32_t wp = 0;
    for (int w = 0; w < warp; ++w) wp += s_w[w];
    uint32_t run = wp + x - t;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (base + j < n) out[base + j] = run;
        run += v[j];
    }
    if (threadIdx.x == kT - 1) sums[blockIdx.x] = wp + x;
}

__global__ void __launch_bounds__(kT) scan_add(uint32_t* __restrict__ out, long long n,
                                               const uint32_t* __restrict__ offs) {
    const long long base = blockIdx.x * static_cast<long long>(kScanBlock) + threadIdx.x * kPer;
    const uint32_t o = offs[blockIdx.x];
#pragma unroll
    for (int j = 0; j < kPer; ++j)
        if (base + j < n) out[base + j] += o;
}

// ---------------------------------------------------------------- radix sort
// hist[d * ntiles + tile] = number of keys of this tile whose digit is d.
__global__ void __launch_bounds__(kT) radix_hist(const uint32_t* __restrict__ keys, long long n, int shift,
                                                 uint32_t* __restrict__ hist, int ntiles) {
    __shared__ uint32_t h[256];
    h[threadIdx.x] = 0;
    __syncthreads();
    const long long base = blockIdx.x * static_cast<long long>(kTile);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const long long i = base + j * kT + threadIdx.x;
        if (i < n) atomicAdd(&h[(keys[i] >> shift) & 255u], 1u);
    }
    __syncthreads();
    hist[static_cast<long long>(threadIdx.x) * ntiles + blockIdx.x] = h[threadIdx.x];
}

// Stable scatter of one tile: keys are taken in input order, 256 per round;
// a key's place = the tile's offset for its digit + keys of that digit in
// earlier rounds + in earlier warps of this round + in lower lanes of its warp.
__global__ void __launch_bounds__(kT) radix_scatter(const uint32_t* __restrict__ kin, const int* __restrict__ iin,
                                                    uint32_t* __restrict__ kout, int* __restrict__ iout, long long n,
                                                    int shift, const uint32_t* __restrict__ offs, int ntiles) {
    __shared__ uint32_t s_base[256];
    __shared__ uint32_t s_cnt[kT / 32][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    s_base[threadIdx.x] = offs[static_cast<long long>(threadIdx.x) * ntiles + blockIdx.x];
    const long long base = blockIdx.x * static_cast<long long>(kTile);
    const unsigned below = (1u << lane) - 1u;
    for (int r = 0; r < kPer; ++r) {
#pragma unroll
        for (int w = 0; w < kT / 32; ++w) s_cnt[w][threadIdx.x] = 0;
        __syncthreads();
        const long long i = base + r * kT + threadIdx.x;
        const bool valid = i < n;
        const uint32_t key = valid ? kin[i] : 0u;
        const int idx = valid ? iin[i] : 0;
        const uint32_t d = valid ? ((key >> shift) & 255u) : 256u;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        const int rank = __popc(peers & below);
        if (valid && rank == 0) s_cnt[warp][d] = __popc(peers);
        __syncthreads();
        if (valid) {
            uint32_t pos = s_base[d] + rank;
            for (int w = 0; w < warp; ++w) pos += s_cnt[w][d];
            kout[pos] = key;
            iout[pos] = idx;
        }
        __syncthreads();
        uint32_t add = 0;
#pragma unroll
        for (int w = 0; w < kT / 32; ++w) add += s_cnt[w][threadIdx.x];
        s_base[threadIdx.x] += add;
        __syncthreads();
    }
}

__global__ void iota_keys(const int* __restrict__ src, uint32_t* __restrict__ keys, int* __restrict__ idx, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        keys[i] = static_cast<uint32_t>(src[i]);
        idx[i] = static_cast<int>(i);
    }
}

// keys[i] = src[idx[i]] (the next, more significant key in source order of the current permutation)
__global__ void gather_keys(const int* __restrict__ src, const int* __restrict__ idx, uint32_t* __restrict__ keys,
                            long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT)
        keys[i] = static_cast<uint32_t>(src[idx[i]]);
}

// BSR sort keys of entry idx[i]: part 0 = its place inside the block
// ((row mod br) * bc + col mod bc), 1 = its block column, 2 = its block row.
__global__ void bsr_keys(const int* __restrict__ rowid, const int* __restrict__ col, const int* __restrict__ idx,
                         int br, int bc, int part, uint32_t* __restrict__ keys, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int p = idx[i];
        const int r = rowid[p], c = col[p];
        keys[i] = static_cast<uint32_t>(part == 0 ? (r % br) * bc + c % bc : part == 1 ? c / bc : r / br);
    }
}

template <class T>
__global__ void gather_values(const T* __restrict__ src, const int* __restrict__ idx, T* __restrict__ dst,
                              long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT)
        dst[i] = src[idx[i]];
}

__global__ void count_keys(const int* __restrict__ a, long long n, uint32_t* __restrict__ cnt) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT)
        atomicAdd(&cnt[a[i]], 1u);
}

// rowid[p] = the row holding entry p: the last i with rp[i] <= p (binary search).
__global__ void expand_rows(const int* __restrict__ rp, int M, long long n, int* __restrict__ rowid) {
    for (long long p = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; p < n;
         p += static_cast<long long>(gridDim.x) * kT) {
        int lo = 0, hi = M;  // rp[lo] <= p < rp[hi]
        while (hi - lo > 1) {
            const int mid = lo + (hi - lo) / 2;
            if (rp[mid] <= p) lo = mid;
            else hi = mid;
        }
        rowid[p] = lo;
    }
}

// BSR: entries sorted by (block row, block column, place in the block).
// flag[i] = 1 where a new block starts; bad |= 8 when two neighbours share (row, col).
__global__ void bsr_mark(const int* __restrict__ ix, const int* __restrict__ rowid, const int* __restrict__ col,
                         int br, int bc, long long n, uint32_t* __restrict__ flag, int* __restrict__ bad) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int p = ix[i];
        const int r = rowid[p], c = col[p];
        uint32_t f = 1;
        if (i > 0) {
            const int q = ix[i - 1];
            const int r2 = rowid[q], c2 = col[q];
            f = (r / br != r2 / br || c / bc != c2 / bc) ? 1u : 0u;
            if (r == r2 && c == c2) atomicOr(bad, 8);
        }
        flag[i] = f;
    }
}

// blocks per block row (from the block starts), for the block-row offsets
__global__ void bsr_count(const int* __restrict__ ix, const int* __restrict__ rowid, const uint32_t* __restrict__ flag,
                          int br, long long n, uint32_t* __restrict__ cnt) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT)
        if (flag[i]) atomicAdd(&cnt[rowid[ix[i]] / br], 1u);
}

// Entry i of the sorted order lands in block slot[i] (inclusive scan of the
// starts, minus one) at (row mod br, col mod bc); the block's column is
// written by its first entry.
template <class T>
__global__ void bsr_scatter(const int* __restrict__ ix, const int* __restrict__ rowid, const int* __restrict__ col,
                            const T* __restrict__ val, const uint32_t* __restrict__ flag,
                            const uint32_t* __restrict__ excl, int br, int bc, long long n, int* __restrict__ bcol,
                            T* __restrict__ bval) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int p = ix[i];
        const int r = rowid[p], c = col[p];
        const long long b = static_cast<long long>(excl[i]) + flag[i] - 1;
        if (flag[i]) bcol[b] = c / bc;
        bval[b * br * bc + static_cast<long long>(r % br) * bc + c % bc] = val[p];
    }
}

// WCSR (windows of 64 rows): entries sorted by (window, column, row in the
// window).  flag[i] = 1 where a new (window, column) starts, counted per
// window in cnt[w]; bad |= 8 when two neighbours share (row, col).
constexpr int kWin = 64;

__global__ void wcsr_keys(const int* __restrict__ rowid, const int* __restrict__ col, const int* __restrict__ idx,
                          int part, uint32_t* __restrict__ keys, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int p = idx[i];
        const int r = rowid[p];
        keys[i] = static_cast<uint32_t>(part == 0 ? r % kWin : part == 1 ? col[p] : r / kWin);
    }
}

__global__ void wcsr_mark(const int* __restrict__ ix, const int* __restrict__ rowid, const int* __restrict__ col,
                          long long n, uint32_t* __restrict__ flag, uint32_t* __restrict__ cnt, int* __restrict__ bad) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int p = ix[i];
        const int r = rowid[p], c = col[p];
        uint32_t f = 1;
        if (i > 0) {
            const int q = ix[i - 1];
            const int r2 = rowid[q], c2 = col[q];
            f = (r / kWin != r2 / kWin || c != c2) ? 1u : 0u;
            if (r == r2 && c == c2) atomicOr(bad, 8);
        }
        flag[i] = f;
        if (f) atomicAdd(&cnt[r / kWin], 1u);
    }
}

// chunks of window w = ceil(distinct columns / 64)
__global__ void wcsr_chunks(const uint32_t* __restrict__ cnt, long long W, uint32_t* __restrict__ nch) {
    for (long long w = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; w < W;
         w += static_cast<long long>(gridDim.x) * kT)
        nch[w] = (cnt[w] + kWin - 1) / kWin;
}

// Entry i has compressed position k = (distinct index) - (window's first
// distinct index); it lands in chunk wp[w] + k / 64 at (row mod 64, k mod 64).
// The first entry of each (window, column) writes the column.
template <class T>
__global__ void wcsr_scatter(const int* __restrict__ ix, const int* __restrict__ rowid, const int* __restrict__ col,
                             const T* __restrict__ val, const uint32_t* __restrict__ flag,
                             const uint32_t* __restrict__ excl, const uint32_t* __restrict__ dstart,
                             const uint32_t* __restrict__ wp, long long n, int* __restrict__ win_col,
                             T* __restrict__ win_val) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int p = ix[i];
        const int r = rowid[p], w = r / kWin;
        const long long k = static_cast<long long>(excl[i]) + flag[i] - 1 - dstart[w];
        const long long g0 = wp[w];
        if (flag[i]) win_col[g0 * kWin + k] = col[p];
        win_val[((g0 + k / kWin) * kWin + r % kWin) * kWin + k % kWin] = val[p];
    }
}

// Row statistics: len[i] = row_ptr[i+1] - row_ptr[i] (sort keys for the
// percentiles) and, per CTA, the sums S1, S2, min, max and empty rows, folded
// into acc64 = {S1, S2} and acc32 = {min, max, empty} with integer atomics
// (exact, so the order does not matter).
__global__ void __launch_bounds__(kT) row_len_stats(const int* __restrict__ rp, int M, uint32_t* __restrict__ len,
                                                    unsigned long long* __restrict__ acc64, int* __restrict__ acc32) {
    long long s1 = 0, s2 = 0;
    int mn = 0x7fffffff, mx = -0x7fffffff - 1, emp = 0;
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < M;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int l = rp[i + 1] - rp[i];
        len[i] = static_cast<uint32_t>(l);
        s1 += l;
        s2 += static_cast<long long>(l) * l;
        mn = min(mn, l);
        mx = max(mx, l);
        emp += l == 0;
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        s1 += __shfl_down_sync(0xffffffffu, s1, d);
        s2 += __shfl_down_sync(0xffffffffu, s2, d);
        mn = min(mn, __shfl_down_sync(0xffffffffu, mn, d));
        mx = max(mx, __shfl_down_sync(0xffffffffu, mx, d));
        emp += __shfl_down_sync(0xffffffffu, emp, d);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&acc64[0], static_cast<unsigned long long>(s1));
        atomicAdd(&acc64[1], static_cast<unsigned long long>(s2));
        atomicMin(&acc32[0], mn);
        atomicMax(&acc32[1], mx);
        atomicAdd(&acc32[2], emp);
    }
}

// ---------------------------------------------------------------- dispatch plan
// The plan of [SpMM-ops] §2.1-§2.4 built on the GPU, equal to the host
// builder's task for task.  Rows longer than pack_max are CTA rows (one task)
// or split rows (ceil(l / seg_nnz) segment tasks and partial-sum slots); the
// other rows are packed left to right into groups: a group starting at a short
// row s takes rows s .. e(s)-1, e(s) being the largest row end with at most
// block_rows rows, at most block_nnz nonzeros and no long row.  The groups are
// the chain run start, e(run start), e(e(run start)), ... of each run of short
// rows.  e is monotone, so the chain is marked by doubling: after round k
// every e^t(start) with t < 2^(k+1) is marked, and the rounds stop once e^(2^k)
// is a fixed point everywhere.

// per row: kind (0 short, 1 CTA row, 2 split row), long-row tasks, slots, flags
__global__ void plan_classify(const int* __restrict__ rp, int M, int pack_max, int cta_max, int seg_nnz,
                              uint32_t* __restrict__ ntl, uint32_t* __restrict__ nsl, uint32_t* __restrict__ fl,
                              uint32_t* __restrict__ fs, uint32_t* __restrict__ fshort) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < M;
         i += static_cast<long long>(gridDim.x) * kT) {
        const long long l = static_cast<long long>(rp[i + 1]) - rp[i];
        const int kind = l > pack_max ? (l <= cta_max ? 1 : 2) : 0;
        const uint32_t ns = kind == 2 ? static_cast<uint32_t>((l + seg_nnz - 1) / seg_nnz) : 0u;
        ntl[i] = kind == 1 ? 1u : ns;
        nsl[i] = ns;
        fl[i] = kind != 0;
        fs[i] = kind == 2;
        fshort[i] = kind == 0;
    }
}

// L[lidx[i]] = i for every long row (ascending)
__global__ void plan_compact(const uint32_t* __restrict__ fl, const uint32_t* __restrict__ lidx, int M,
                             int* __restrict__ L) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < M;
         i += static_cast<long long>(gridDim.x) * kT)
        if (fl[i]) L[lidx[i]] = static_cast<int>(i);
}

// E0[s] = e(s) for short rows, s itself for long rows and for s = M; on[s] = 1 at run starts
__global__ void plan_group_end(const int* __restrict__ rp, int M, const uint32_t* __restrict__ fl,
                               const int* __restrict__ L, int nL, int block_nnz, int block_rows, int* __restrict__ E0,
                               uint32_t* __restrict__ on) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i <= M;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int s = static_cast<int>(i);
        if (s == M || fl[s]) {
            E0[s] = s;
            on[s] = 0;
            continue;
        }
        int lo = 0, hi = nL;  // first long row after s
        while (lo < hi) {
            const int mid = lo + (hi - lo) / 2;
            if (L[mid] > s) hi = mid; else lo = mid + 1;
        }
        const int run_end = lo < nL ? L[lo] : M;
        const int lim = static_cast<int>(min(static_cast<long long>(run_end), static_cast<long long>(s) + block_rows));
        const int base = rp[s];
        int a = s + 1, b = lim;  // largest j in [s+1, lim] with rp[j] - rp[s] <= block_nnz (j = s+1 always fits)
        while (a < b) {
            const int mid = a + (b - a + 1) / 2;
            if (rp[mid] - base <= block_nnz) a = mid; else b = mid - 1;
        }
        E0[s] = a;
        on[s] = (s == 0 || fl[s - 1]) ? 1u : 0u;
    }
}

// one doubling round: mark E(s) for every marked s, then E2 = E o E (changed when any entry moved)
__global__ void plan_mark(const int* __restrict__ E, uint32_t* on, int M) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < M;
         i += static_cast<long long>(gridDim.x) * kT)
        if (on[i]) {
            const int t = E[i];
            if (t < M) on[t] = 1u;
        }
}

__global__ void plan_compose(const int* __restrict__ E, int* __restrict__ E2, int M, int* __restrict__ changed) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i <= M;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int a = E[i];
        const int b = E[a];
        E2[i] = b;
        if (b != a) *changed = 1;
    }
}

// group starts = marked short rows
__global__ void plan_starts(const uint32_t* __restrict__ on, const uint32_t* __restrict__ fshort, int M,
                            uint32_t* __restrict__ gs) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < M;
         i += static_cast<long long>(gridDim.x) * kT)
        gs[i] = on[i] & fshort[i];
}

__device__ __forceinline__ int plan_reduce_code(long long nnz_g, long long rows_g, int div) {
    if (div == 0) return kReduceSegmented;
    const long long per = (nnz_g + rows_g * div - 1) / (rows_g * div);
    int lg = 0;
    while (lg < 5 && (1ll << lg) < per) ++lg;
    return lg;
}

__device__ __forceinline__ void put4(int* d, long long pos, int a, int b, int c, int e) {
    reinterpret_cast<int4*>(d)[pos] = make_int4(a, b, c, e);
}

// Writes every task in both forms (host form: the documented one; device form:
// kind | code << 2 | aux << 8, row, p0, p1) and the split-row table; counts the
// groups by reduction code (cnt[0] thread groups, [1] lane groups, [2] segmented).
__global__ void plan_write(const int* __restrict__ rp, int M, int seg_nnz, int lanes_div,
                           const uint32_t* __restrict__ nsl,
                           const uint32_t* __restrict__ fl, const uint32_t* __restrict__ fs,
                           const uint32_t* __restrict__ toff, const uint32_t* __restrict__ soff,
                           const uint32_t* __restrict__ sidx, const uint32_t* __restrict__ gsf,
                           const uint32_t* __restrict__ gidx, const int* __restrict__ E0, long long nlongtasks,
                           int* __restrict__ htask, int* __restrict__ dtask, int* __restrict__ longrows,
                           unsigned long long* __restrict__ cnt) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < M;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int r = static_cast<int>(i);
        if (fl[r] && !fs[r]) {  // CTA row
            put4(htask, toff[r], kTaskCta, r, 0, 0);
            put4(dtask, toff[r], kTaskCta, r, rp[r], rp[r + 1]);
        } else if (fs[r]) {  // split row: its segments and its fix-up entry
            const int ns = static_cast<int>(nsl[r]), slot = static_cast<int>(soff[r]);
            put4(longrows, sidx[r], r, slot, ns, 0);
            for (int sg = 0; sg < ns; ++sg) {
                const long long lo = rp[r] + static_cast<long long>(sg) * seg_nnz;
                const long long hi = min(static_cast<long long>(rp[r + 1]), lo + seg_nnz);
                put4(htask, toff[r] + sg, kTaskSeg, r, sg, slot + sg);
                put4(dtask, toff[r] + sg, kTaskSeg | ((slot + sg) << 8), r, static_cast<int>(lo), static_cast<int>(hi));
            }
        } else if (gsf[r]) {  // a group starts here
            const int e = E0[r];
            const int c = plan_reduce_code(static_cast<long long>(rp[e]) - rp[r], e - r, lanes_div);
            const long long pos = nlongtasks + gidx[r];
            put4(htask, pos, kTaskGroup + 256 * c, r, e, 0);
            put4(dtask, pos, kTaskGroup | (c << 2) | ((e - r) << 8), r, rp[r], rp[e]);
            atomicAdd(&cnt[c == 0 ? 0 : c == kReduceSegmented ? 2 : 1], 1ull);
        }
    }
}

// Segmented groups: the first row of each thread (spx_first_entry), by a
// binary search of the group's row offsets; one entry per (group, thread).
__global__ void plan_first(const int* __restrict__ rp, const int4* __restrict__ groups, long long ngroups,
                           int nth, int per, uint16_t* __restrict__ first) {
    const long long total = ngroups * nth;
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int4 g = groups[i / nth];
        const long long a = (i % nth) * static_cast<long long>(per);
        const int nrows = g.x >> 8, r0 = g.y, p0 = g.z, n = g.w - g.z;
        uint16_t v = 0;
        if (a < n) {
            int lo = 0, hi = nrows;  // first index with rp[r0 + index] - p0 > a
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (rp[r0 + mid] - p0 > a) hi = mid; else lo = mid + 1;
            }
            v = spx_first_entry(lo - 1, rp[r0 + lo - 1] - p0 < a);
        }
        first[i] = v;
    }
}

// ---------------------------------------------------------------- SELL-C-sigma
// [SpMM-ops] §1.4, [Formats] §6: rows longer than `piece` are cut into pieces
// (pseudo-rows with a partial-sum slot); pseudo-rows are sorted longest first,
// stably, inside windows of sigma; slices of 32 take the length of their first
// (longest) pseudo-row and are stored column-major.  Same image as the host builder.
constexpr int kSellC = 32;

// per row: pseudo-rows n, long-row flag, slots (entry M stays 0 for the scans)
__global__ void sell_count(const int* __restrict__ rp, int M, int piece, uint32_t* __restrict__ n,
                           uint32_t* __restrict__ fl, uint32_t* __restrict__ ns) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < M;
         i += static_cast<long long>(gridDim.x) * kT) {
        const long long l = static_cast<long long>(rp[i + 1]) - rp[i];
        const bool lng = l > piece;
        const uint32_t k = lng ? static_cast<uint32_t>((l + piece - 1) / piece) : 1u;
        n[i] = k;
        fl[i] = lng;
        ns[i] = lng ? k : 0u;
    }
}

// pseudo-row arrays in row order (pieces in order) and the long-row table
__global__ void sell_pseudo(const int* __restrict__ rp, int M, int piece, const uint32_t* __restrict__ pst,
                            const uint32_t* __restrict__ fl, const uint32_t* __restrict__ lidx,
                            const uint32_t* __restrict__ lslot, int* __restrict__ plen, int* __restrict__ prow,
                            int* __restrict__ pstart, int* __restrict__ pslot, int* __restrict__ longrows) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < M;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int r = static_cast<int>(i);
        const int a = rp[r], l = rp[r + 1] - a;
        const uint32_t q0 = pst[r];
        if (!fl[r]) {
            plen[q0] = l;
            prow[q0] = r;
            pstart[q0] = a;
            pslot[q0] = -1;
            continue;
        }
        const int n = (l + piece - 1) / piece, slot = static_cast<int>(lslot[r]);
        reinterpret_cast<int4*>(longrows)[lidx[r]] = make_int4(r, slot, n, 0);
        for (int k = 0; k < n; ++k) {
            plen[q0 + k] = min(piece, l - k * piece);
            prow[q0 + k] = r;
            pstart[q0 + k] = a + k * piece;
            pslot[q0 + k] = slot + k;
        }
    }
}

// sort keys: descending length (piece - len), payload the pseudo-row index
__global__ void sell_len_keys(const int* __restrict__ plen, int piece, uint32_t* __restrict__ keys,
                              int* __restrict__ idx, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        keys[i] = static_cast<uint32_t>(piece - plen[i]);
        idx[i] = static_cast<int>(i);
    }
}

// window of the pseudo-row now at position i
__global__ void sell_win_keys(const int* __restrict__ idx, int sigma, uint32_t* __restrict__ keys, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT)
        keys[i] = static_cast<uint32_t>(idx[i] / sigma);
}

// padded entries of slice s = 32 x the length of its first pseudo-row; total in acc
__global__ void sell_slices(const int* __restrict__ idx, const int* __restrict__ plen, long long ns,
                            uint32_t* __restrict__ width, unsigned long long* __restrict__ acc) {
    for (long long s = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; s < ns;
         s += static_cast<long long>(gridDim.x) * kT) {
        const uint32_t w = static_cast<uint32_t>(plen[idx[s * kSellC]]) * kSellC;
        width[s] = w;
        atomicAdd(acc, static_cast<unsigned long long>(w));
    }
}

__global__ void fill_i32(int* __restrict__ a, long long n, int v) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT)
        a[i] = v;
}

// the pseudo-row at sorted position q: its row code and its entries, column-major in slice q / 32
__global__ void sell_scatter(const int* __restrict__ idx, const int* __restrict__ plen, const int* __restrict__ prow,
                             const int* __restrict__ pstart, const int* __restrict__ pslot,
                             const uint32_t* __restrict__ sp, const int* __restrict__ col,
                             const float* __restrict__ val, long long np, int* __restrict__ prow_out,
                             int* __restrict__ scol, float* __restrict__ sval) {
    for (long long q = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; q < np;
         q += static_cast<long long>(gridDim.x) * kT) {
        const int p = idx[q];
        const int slot = pslot[p];
        prow_out[q] = slot < 0 ? prow[p] : -1 - slot;
        const long long base = static_cast<long long>(sp[q / kSellC]) + q % kSellC;
        const int a = pstart[p], l = plen[p];
        for (int j = 0; j < l; ++j) {
            scol[base + static_cast<long long>(j) * kSellC] = col[a + j];
            sval[base + static_cast<long long>(j) * kSellC] = val[a + j];
        }
    }
}

int grid_for(long long n) {
    long long g = (n + kT - 1) / kT;
    if (g > 152 * 32) g = 152 * 32;
    return static_cast<int>(g < 1 ? 1 : g);
}

// ---------------------------------------------------------------- host helpers
struct Pool {
    cudaStream_t st;
    std::vector<void*> ptrs;
    cudaError_t err = cudaSuccess;
    explicit Pool(cudaStream_t s) : st(s) {}
    template <class T>
    T* get(long long n) {
        void* p = nullptr;
        if (err == cudaSuccess) err = cudaMallocAsync(&p, static_cast<size_t>(n > 0 ? n : 1) * sizeof(T), st);
        if (err == cudaSuccess) ptrs.push_back(p);
        return static_cast<T*>(p);
    }
    ~Pool() {
        for (void* p : ptrs) cudaFreeAsync(p, st);
    }
};

// Exclusive scan of n uint32 (in place allowed: out may equal in).
cudaError_t scan_exclusive(const uint32_t* in, uint32_t* out, long long n, Pool& pool) {
    if (n <= 0) return cudaSuccess;
    const long long nb = (n + kScanBlock - 1) / kScanBlock;
    uint32_t* sums = pool.get<uint32_t>(nb);
    if (pool.err != cudaSuccess) return pool.err;
    scan_blocks<<<static_cast<unsigned>(nb), kT, 0, pool.st>>>(in, out, n, sums);
    if (nb > 1) {
        cudaError_t e = scan_exclusive(sums, sums, nb, pool);
        if (e != cudaSuccess) return e;
        scan_add<<<static_cast<unsigned>(nb), kT, 0, pool.st>>>(out, n, sums);
    }
    return cudaGetLastError();
}

int bits_for(long long lim) {  // bits needed for keys in [0, lim)
    int b = 0;
    while (b < 32 && (1ll << b) < lim) ++b;
    return b;
}

// Stable LSD radix sort of (k, ix) by the low `bits` bits of the keys; the
// result ends in (k, ix) (the second buffers are scratch).
cudaError_t radix_sort(uint32_t*& k, int*& ix, uint32_t*& k2, int*& ix2, long long n, int bits, Pool& pool,
                       uint64_t& launches) {
    if (n <= 1) return cudaSuccess;
    const int ntiles = static_cast<int>((n + kTile - 1) / kTile);
    uint32_t* hist = pool.get<uint32_t>(256ll * ntiles);
    if (pool.err != cudaSuccess) return pool.err;
    for (int shift = 0; shift < bits; shift += 8) {
        radix_hist<<<ntiles, kT, 0, pool.st>>>(k, n, shift, hist, ntiles);
        cudaError_t e = scan_exclusive(hist, hist, 256ll * ntiles, pool);
        if (e != cudaSuccess) return e;
        radix_scatter<<<ntiles, kT, 0, pool.st>>>(k, ix, k2, ix2, n, shift, hist, ntiles);
        launches += 3;
        std::swap(k, k2);
        std::swap(ix, ix2);
    }
    return cudaGetLastError();
}

cudaError_t gather_vals(const void* src, const int* idx, void* dst, long long n, int vb, cudaStream_t st) {
    const int g = grid_for(n);
    switch (vb) {
        case 1: gather_values<uint8_t><<<g, kT, 0, st>>>(static_cast<const uint8_t*>(src), idx, static_cast<uint8_t*>(dst), n); break;
        case 2: gather_values<uint16_t><<<g, kT, 0, st>>>(static_cast<const uint16_t*>(src), idx, static_cast<uint16_t*>(dst), n); break;
        case 4: gather_values<uint32_t><<<g, kT, 0, st>>>(static_cast<const uint32_t*>(src), idx, static_cast<uint32_t*>(dst), n); break;
        default: gather_values<uint64_t><<<g, kT, 0, st>>>(static_cast<const uint64_t*>(src), idx, static_cast<uint64_t*>(dst), n); break;
    }
    return cudaGetLastError();
}

spx_status read_flag(const int* d_bad, cudaStream_t st, int* h) {
    if (cudaMemcpyAsync(h, d_bad, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SPX_ERR_CUDA;
    return SPX_OK;
}

// Row offsets from exact counts: ptr[0..lim] = exclusive scan of count(key == i), ptr[lim] = n.
cudaError_t offsets(const int* keys, long long n, int lim, int32_t* ptr, Pool& pool, uint64_t& launches) {
    uint32_t* cnt = reinterpret_cast<uint32_t*>(ptr);  // counted in place: lim + 1 slots
    cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(uint32_t) * (static_cast<size_t>(lim) + 1), pool.st);
    if (e != cudaSuccess) return e;
    if (n > 0) {
        count_keys<<<grid_for(n), kT, 0, pool.st>>>(keys, n, cnt);
        ++launches;
    }
    e = scan_exclusive(cnt, cnt, static_cast<long long>(lim) + 1, pool);
    ++launches;
    return e;
}

}  // namespace

spx_status spx_dev_build_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* coo_row, const int32_t* coo_col,
                             const void* coo_val, int32_t vb, int32_t* row_ptr, int32_t* col, void* val,
                             cudaStream_t st) {
    Pool pool(st);
    uint64_t launches = 0;
    int* bad = pool.get<int>(1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    if (cudaMemsetAsync(bad, 0, sizeof(int), st) != cudaSuccess) return SPX_ERR_CUDA;
    if (nnz > 0) {
        check_indices<<<grid_for(nnz), kT, 0, st>>>(coo_row, nnz, M, bad);
        check_indices<<<grid_for(nnz), kT, 0, st>>>(coo_col, nnz, K, bad);
        launches += 2;
    }
    int h = 0;
    spx_status s = read_flag(bad, st, &h);
    if (s != SPX_OK) return s;
    if (h) return SPX_ERR_INDEX_RANGE;
    uint32_t *k = pool.get<uint32_t>(nnz), *k2 = pool.get<uint32_t>(nnz);
    int *ix = pool.get<int>(nnz), *ix2 = pool.get<int>(nnz);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    cudaError_t e = cudaSuccess;
    if (nnz > 0) {
        // LSD over (row, col): stable by column first, then stable by row
        iota_keys<<<grid_for(nnz), kT, 0, st>>>(coo_col, k, ix, nnz);
        ++launches;
        e = radix_sort(k, ix, k2, ix2, nnz, bits_for(K), pool, launches);
        if (e == cudaSuccess) {
            gather_keys<<<grid_for(nnz), kT, 0, st>>>(coo_row, ix, k, nnz);
            ++launches;
            e = radix_sort(k, ix, k2, ix2, nnz, bits_for(M), pool, launches);
        }
        if (e == cudaSuccess) {
            gather_values<int32_t><<<grid_for(nnz), kT, 0, st>>>(coo_col, ix, col, nnz);
            e = gather_vals(coo_val, ix, val, nnz, vb, st);
            launches += 2;
        }
    }
    if (e == cudaSuccess) e = offsets(coo_row, nnz, M, row_ptr, pool, launches);
    if (e == cudaSuccess) e = cudaGetLastError();
    spx_note_launches(launches);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    return e == cudaSuccess ? SPX_OK : SPX_ERR_CUDA;
}

spx_status spx_dev_transpose_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                                 const void* val, int32_t vb, int32_t* t_row_ptr, int32_t* t_col, void* t_val,
                                 cudaStream_t st) {
    Pool pool(st);
    uint64_t launches = 0;
    int* bad = pool.get<int>(1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    if (cudaMemsetAsync(bad, 0, sizeof(int), st) != cudaSuccess) return SPX_ERR_CUDA;
    check_row_ptr<<<grid_for(M), kT, 0, st>>>(row_ptr, M, nnz, bad);
    ++launches;
    if (nnz > 0) {
        check_indices<<<grid_for(nnz), kT, 0, st>>>(col, nnz, K, bad);
        ++launches;
    }
    int h = 0;
    spx_status s = read_flag(bad, st, &h);
    if (s != SPX_OK) return s;
    if (h & 4) return SPX_ERR_ARG;
    if (h & 2) return SPX_ERR_NOT_SORTED;
    if (h & 1) return SPX_ERR_INDEX_RANGE;
    uint32_t *k = pool.get<uint32_t>(nnz), *k2 = pool.get<uint32_t>(nnz);
    int *ix = pool.get<int>(nnz), *ix2 = pool.get<int>(nnz), *rowid = pool.get<int>(nnz);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    cudaError_t e = cudaSuccess;
    if (nnz > 0) {
        expand_rows<<<grid_for(nnz), kT, 0, st>>>(row_ptr, M, nnz, rowid);
        iota_keys<<<grid_for(nnz), kT, 0, st>>>(col, k, ix, nnz);
        launches += 2;
        // entries come in row order: a stable sort by column keeps rows ascending in each column
        e = radix_sort(k, ix, k2, ix2, nnz, bits_for(K), pool, launches);
        if (e == cudaSuccess) {
            gather_values<int32_t><<<grid_for(nnz), kT, 0, st>>>(rowid, ix, t_col, nnz);
            e = gather_vals(val, ix, t_val, nnz, vb, st);
            launches += 2;
        }
    }
    if (e == cudaSuccess) e = offsets(col, nnz, K, t_row_ptr, pool, launches);
    if (e == cudaSuccess) e = cudaGetLastError();
    spx_note_launches(launches);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    return e == cudaSuccess ? SPX_OK : SPX_ERR_CUDA;
}

spx_status spx_dev_build_bsr(int32_t M, int32_t K, const int32_t* row_ptr, const int32_t* col, const void* val,
                             int32_t vb, int32_t br, int32_t bc, int32_t* bsr_row_ptr, int32_t* bsr_col,
                             void* bsr_val, int64_t* nnzb_out, double* fill_out, cudaStream_t st) {
    if (static_cast<long long>(br) * bc > kI32Max) return SPX_ERR_UNSUPPORTED;
    Pool pool(st);
    uint64_t launches = 0;
    int32_t nnz32 = 0;
    if (cudaMemcpyAsync(&nnz32, row_ptr + M, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SPX_ERR_CUDA;
    const long long nnz = nnz32;
    if (nnz < 0) return SPX_ERR_ARG;
    if (nnz > 0 && (!col || (bsr_val && !val))) return SPX_ERR_ARG;
    int* bad = pool.get<int>(1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    if (cudaMemsetAsync(bad, 0, sizeof(int), st) != cudaSuccess) return SPX_ERR_CUDA;
    check_row_ptr<<<grid_for(M), kT, 0, st>>>(row_ptr, M, nnz, bad);
    ++launches;
    if (nnz > 0) {
        check_indices<<<grid_for(nnz), kT, 0, st>>>(col, nnz, K, bad);
        ++launches;
    }
    int h = 0;
    spx_status s = read_flag(bad, st, &h);
    if (s != SPX_OK) return s;
    if (h & 4) return SPX_ERR_ARG;
    if (h & 2) return SPX_ERR_NOT_SORTED;
    if (h & 1) return SPX_ERR_INDEX_RANGE;
    const long long MB = (static_cast<long long>(M) + br - 1) / br;
    const long long KB = (static_cast<long long>(K) + bc - 1) / bc;
    uint32_t *k = pool.get<uint32_t>(nnz), *k2 = pool.get<uint32_t>(nnz), *flag = pool.get<uint32_t>(nnz);
    uint32_t* excl = pool.get<uint32_t>(nnz);
    int *ix = pool.get<int>(nnz), *ix2 = pool.get<int>(nnz), *rowid = pool.get<int>(nnz);
    uint32_t* cnt = pool.get<uint32_t>(MB + 1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    cudaError_t e = cudaSuccess;
    long long nnzb = 0;
    if (nnz > 0) {
        expand_rows<<<grid_for(nnz), kT, 0, st>>>(row_ptr, M, nnz, rowid);
        iota_keys<<<grid_for(nnz), kT, 0, st>>>(col, k, ix, nnz);  // ix = 0..nnz-1; the keys are set below
        launches += 2;
        // LSD over (block row, block column, place in the block): equal
        // (row, col) pairs end up next to each other whatever the column
        // order inside the CSR rows
        const long long lim[3] = {static_cast<long long>(br) * bc, KB, MB};
        for (int part = 0; part < 3 && e == cudaSuccess; ++part) {
            if (bits_for(lim[part]) == 0) continue;  // a single key value: nothing to order
            bsr_keys<<<grid_for(nnz), kT, 0, st>>>(rowid, col, ix, br, bc, part, k, nnz);
            ++launches;
            e = radix_sort(k, ix, k2, ix2, nnz, bits_for(lim[part]), pool, launches);
        }
        if (e == cudaSuccess) {
            bsr_mark<<<grid_for(nnz), kT, 0, st>>>(ix, rowid, col, br, bc, nnz, flag, bad);
            launches += 2;
            e = scan_exclusive(flag, excl, nnz, pool);
        }
        uint32_t last[2] = {0, 0};
        if (e == cudaSuccess) e = cudaMemcpyAsync(&last[0], excl + nnz - 1, 4, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(&last[1], flag + nnz - 1, 4, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(&h, bad, sizeof(int), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return SPX_ERR_CUDA;
        if (h & 8) return SPX_ERR_DUPLICATE;
        nnzb = static_cast<long long>(last[0]) + last[1];
        if (nnzb > kI32Max) return SPX_ERR_INDEX_RANGE;
    }
    if (bsr_row_ptr) {
        e = cudaMemsetAsync(cnt, 0, sizeof(uint32_t) * static_cast<size_t>(MB + 1), st);
        if (e == cudaSuccess && nnz > 0) {
            bsr_count<<<grid_for(nnz), kT, 0, st>>>(ix, rowid, flag, br, nnz, cnt);
            ++launches;
        }
        if (e == cudaSuccess) e = scan_exclusive(cnt, reinterpret_cast<uint32_t*>(bsr_row_ptr), MB + 1, pool);
    }
    if (e == cudaSuccess && bsr_col && bsr_val && nnzb > 0) {
        e = cudaMemsetAsync(bsr_val, 0, static_cast<size_t>(nnzb) * br * bc * vb, st);
        const int g = grid_for(nnz);
        if (e == cudaSuccess) {
            switch (vb) {
                case 1: bsr_scatter<uint8_t><<<g, kT, 0, st>>>(ix, rowid, col, static_cast<const uint8_t*>(val), flag, excl, br, bc, nnz, bsr_col, static_cast<uint8_t*>(bsr_val)); break;
                case 2: bsr_scatter<uint16_t><<<g, kT, 0, st>>>(ix, rowid, col, static_cast<const uint16_t*>(val), flag, excl, br, bc, nnz, bsr_col, static_cast<uint16_t*>(bsr_val)); break;
                case 4: bsr_scatter<uint32_t><<<g, kT, 0, st>>>(ix, rowid, col, static_cast<const uint32_t*>(val), flag, excl, br, bc, nnz, bsr_col, static_cast<uint32_t*>(bsr_val)); break;
                default: bsr_scatter<uint64_t><<<g, kT, 0, st>>>(ix, rowid, col, static_cast<const uint64_t*>(val), flag, excl, br, bc, nnz, bsr_col, static_cast<uint64_t*>(bsr_val)); break;
            }
            ++launches;
            e = cudaGetLastError();
        }
    }
    spx_note_launches(launches);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // the pool frees, and the caller's host sizes are final
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    if (nnzb_out) *nnzb_out = nnzb;
    if (fill_out) *fill_out = nnzb ? static_cast<double>(nnz) / (static_cast<double>(nnzb) * br * bc) : 0.0;
    return SPX_OK;
}

spx_status spx_dev_build_wcsr(int32_t M, int32_t K, const int32_t* row_ptr, const int32_t* col, const void* val,
                              int32_t vb, int32_t* win_ptr, int32_t* win_col, void* win_val, int64_t* nchunks_out,
                              double* fill_out, cudaStream_t st) {
    Pool pool(st);
    uint64_t launches = 0;
    int32_t nnz32 = 0;
    if (cudaMemcpyAsync(&nnz32, row_ptr + M, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SPX_ERR_CUDA;
    const long long nnz = nnz32;
    if (nnz < 0) return SPX_ERR_INDEX_RANGE;
    if (nnz > 0 && (!col || !val)) return SPX_ERR_ARG;
    int* bad = pool.get<int>(1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    if (cudaMemsetAsync(bad, 0, sizeof(int), st) != cudaSuccess) return SPX_ERR_CUDA;
    check_row_ptr<<<grid_for(M), kT, 0, st>>>(row_ptr, M, nnz, bad);
    ++launches;
    if (nnz > 0) {
        check_indices<<<grid_for(nnz), kT, 0, st>>>(col, nnz, K, bad);
        ++launches;
    }
    int h = 0;
    spx_status s = read_flag(bad, st, &h);
    if (s != SPX_OK) return s;
    if (h & 4) return SPX_ERR_ARG;
    if (h & 2) return SPX_ERR_NOT_SORTED;
    if (h & 1) return SPX_ERR_INDEX_RANGE;
    const long long W = (static_cast<long long>(M) + kWin - 1) / kWin;
    uint32_t *k = pool.get<uint32_t>(nnz), *k2 = pool.get<uint32_t>(nnz), *flag = pool.get<uint32_t>(nnz);
    uint32_t* excl = pool.get<uint32_t>(nnz);
    int *ix = pool.get<int>(nnz), *ix2 = pool.get<int>(nnz), *rowid = pool.get<int>(nnz);
    uint32_t *cnt = pool.get<uint32_t>(W + 1), *wp = pool.get<uint32_t>(W + 1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(uint32_t) * static_cast<size_t>(W + 1), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(wp, 0, sizeof(uint32_t) * static_cast<size_t>(W + 1), st);
    if (e == cudaSuccess && nnz > 0) {
        expand_rows<<<grid_for(nnz), kT, 0, st>>>(row_ptr, M, nnz, rowid);
        iota_keys<<<grid_for(nnz), kT, 0, st>>>(col, k, ix, nnz);  // ix = 0..nnz-1; the keys are set below
        launches += 2;
        // LSD over (window, column, row in the window)
        const long long lim[3] = {kWin, K, W};
        for (int part = 0; part < 3 && e == cudaSuccess; ++part) {
            if (bits_for(lim[part]) == 0) continue;
            wcsr_keys<<<grid_for(nnz), kT, 0, st>>>(rowid, col, ix, part, k, nnz);
            ++launches;
            e = radix_sort(k, ix, k2, ix2, nnz, bits_for(lim[part]), pool, launches);
        }
        if (e == cudaSuccess) {
            wcsr_mark<<<grid_for(nnz), kT, 0, st>>>(ix, rowid, col, nnz, flag, cnt, bad);
            wcsr_chunks<<<grid_for(W), kT, 0, st>>>(cnt, W, wp);
            launches += 2;
            e = scan_exclusive(flag, excl, nnz, pool);
        }
    }
    // wp[0..W] = first chunk of each window (wp[W] = chunks); cnt -> first distinct index per window
    if (e == cudaSuccess) e = scan_exclusive(wp, wp, W + 1, pool);
    if (e == cudaSuccess) e = scan_exclusive(cnt, cnt, W + 1, pool);
    uint32_t total = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&total, wp + W, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h, bad, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    if (h & 8) return SPX_ERR_DUPLICATE;
    const long long nch = total;
    if (nch * kWin > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (win_ptr) e = cudaMemcpyAsync(win_ptr, wp, sizeof(uint32_t) * static_cast<size_t>(W + 1),
                                     cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && win_col && win_val && nch > 0) {
        e = cudaMemsetAsync(win_col, 0xFF, sizeof(int32_t) * static_cast<size_t>(nch) * kWin, st);  // -1 = padding
        if (e == cudaSuccess) e = cudaMemsetAsync(win_val, 0, static_cast<size_t>(nch) * kWin * kWin * vb, st);
        const int g = grid_for(nnz);
        if (e == cudaSuccess && nnz > 0) {
            switch (vb) {
                case 1: wcsr_scatter<uint8_t><<<g, kT, 0, st>>>(ix, rowid, col, static_cast<const uint8_t*>(val), flag, excl, cnt, wp, nnz, win_col, static_cast<uint8_t*>(win_val)); break;
                case 2: wcsr_scatter<uint16_t><<<g, kT, 0, st>>>(ix, rowid, col, static_cast<const uint16_t*>(val), flag, excl, cnt, wp, nnz, win_col, static_cast<uint16_t*>(win_val)); break;
                case 4: wcsr_scatter<uint32_t><<<g, kT, 0, st>>>(ix, rowid, col, static_cast<const uint32_t*>(val), flag, excl, cnt, wp, nnz, win_col, static_cast<uint32_t*>(win_val)); break;
                default: wcsr_scatter<uint64_t><<<g, kT, 0, st>>>(ix, rowid, col, static_cast<const uint64_t*>(val), flag, excl, cnt, wp, nnz, win_col, static_cast<uint64_t*>(win_val)); break;
            }
            ++launches;
            e = cudaGetLastError();
        }
    }
    spx_note_launches(launches);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    if (nchunks_out) *nchunks_out = nch;
    if (fill_out) *fill_out = nch ? static_cast<double>(nnz) / (static_cast<double>(nch) * kWin * kWin) : 0.0;
    return SPX_OK;
}

// Structure fingerprint of row_ptr[0..M]: the sum of spx_fp_term(i, row_ptr[i])
// mod 2^64, summed per warp and added into one 64-bit word (integer sums: the
// value does not depend on the order).
__global__ void __launch_bounds__(kT) rp_fingerprint(const int* __restrict__ rp, int M,
                                                     unsigned long long* __restrict__ acc) {
    unsigned long long f = 0;
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i <= M;
         i += static_cast<long long>(gridDim.x) * kT)
        f += spx_fp_term(static_cast<uint64_t>(i), rp[i]);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) f += __shfl_down_sync(0xffffffffu, f, d);
    if ((threadIdx.x & 31) == 0) atomicAdd(acc, f);
}

spx_status spx_dev_rp_fingerprint(int32_t M, const int32_t* row_ptr, uint64_t* out, cudaStream_t st) {
    if (M < 0 || !row_ptr || !out) return SPX_ERR_ARG;
    Pool pool(st);
    unsigned long long* acc = pool.get<unsigned long long>(1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    unsigned long long h = 0;
    cudaError_t e = cudaMemsetAsync(acc, 0, sizeof(unsigned long long), st);
    if (e == cudaSuccess) {
        rp_fingerprint<<<grid_for(static_cast<long long>(M) + 1), kT, 0, st>>>(row_ptr, M, acc);
        spx_note_launches(1);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h, acc, sizeof(h), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    *out = h;
    return SPX_OK;
}

spx_status spx_dev_row_stats(int32_t M, const int32_t* row_ptr, spx_row_stats_t* out, cudaStream_t st) {
    std::memset(out, 0, sizeof(*out));
    out->rows = M;
    if (M == 0) return SPX_OK;
    Pool pool(st);
    uint64_t launches = 0;
    unsigned long long* acc64 = pool.get<unsigned long long>(2);
    int* acc32 = pool.get<int>(3);
    uint32_t *k = pool.get<uint32_t>(M), *k2 = pool.get<uint32_t>(M);
    int *ix = pool.get<int>(M), *ix2 = pool.get<int>(M);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    const int init32[3] = {0x7fffffff, -0x7fffffff - 1, 0};
    unsigned long long h64[2] = {0, 0};
    int h32[3] = {0, 0, 0};
    cudaError_t e = cudaMemsetAsync(acc64, 0, 2 * sizeof(unsigned long long), st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(acc32, init32, sizeof(init32), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ix, 0, sizeof(int) * static_cast<size_t>(M), st);  // payload unused
    if (e == cudaSuccess) {
        row_len_stats<<<grid_for(M), kT, 0, st>>>(row_ptr, M, k, acc64, acc32);
        ++launches;
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(h64, acc64, sizeof(h64), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h32, acc32, sizeof(h32), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    // nearest-rank percentiles: the ceil(q*M/100)-th smallest length of the sorted lengths
    const int hi = h32[1] < 0 ? 32 : bits_for(static_cast<long long>(h32[1]) + 1);
    e = radix_sort(k, ix, k2, ix2, M, hi, pool, launches);
    const long long rank[3] = {(50LL * M + 99) / 100, (95LL * M + 99) / 100, (99LL * M + 99) / 100};
    uint32_t q[3] = {0, 0, 0};
    for (int j = 0; j < 3 && e == cudaSuccess; ++j)
        e = cudaMemcpyAsync(&q[j], k + rank[j] - 1, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
    spx_note_launches(launches);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    const int64_t s1 = static_cast<int64_t>(h64[0]), s2 = static_cast<int64_t>(h64[1]);
    out->nnz = s1;
    out->sumsq = s2;
    out->min = h32[0];
    out->max = h32[1];
    out->empty = h32[2];
    out->p50 = static_cast<int32_t>(q[0]);
    out->p95 = static_cast<int32_t>(q[1]);
    out->p99 = static_cast<int32_t>(q[2]);
    spx_row_stats_finish(M, out);
    return SPX_OK;
}

spx_status spx_dev_check_rp(int32_t M, int64_t nnz, const int32_t* row_ptr, cudaStream_t st) {
    Pool pool(st);
    int* bad = pool.get<int>(1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    if (cudaMemsetAsync(bad, 0, sizeof(int), st) != cudaSuccess) return SPX_ERR_CUDA;
    check_row_ptr<<<grid_for(M), kT, 0, st>>>(row_ptr, M, nnz, bad);
    spx_note_launches(1);
    int h = 0;
    spx_status s = read_flag(bad, st, &h);
    if (s != SPX_OK) return s;
    if (h & 4) return SPX_ERR_ARG;
    if (h & 2) return SPX_ERR_NOT_SORTED;
    return SPX_OK;
}

spx_status spx_dev_make_plan(spx_plan* P, const int32_t* rp, cudaStream_t st) {
    const spx_plan_opts_t& o = P->opts;
    const int M = P->M;
    P->tasks.clear();
    P->dtasks.clear();
    P->longrows.clear();
    P->first.clear();
    std::memset(P->counts, 0, sizeof(P->counts));
    if (M == 0) {
        P->table_bytes = 0;
        P->scratch_bytes = 0;
        return SPX_OK;
    }
    Pool pool(st);
    uint64_t launches = 0;
    const long long n1 = static_cast<long long>(M) + 1;
    uint32_t *toff = pool.get<uint32_t>(n1), *nsl = pool.get<uint32_t>(n1), *soff = pool.get<uint32_t>(n1);
    uint32_t *fl = pool.get<uint32_t>(n1), *lidx = pool.get<uint32_t>(n1), *fs = pool.get<uint32_t>(n1);
    uint32_t *sidx = pool.get<uint32_t>(n1), *fsh = pool.get<uint32_t>(n1), *on = pool.get<uint32_t>(n1);
    uint32_t *gsf = pool.get<uint32_t>(n1), *gidx = pool.get<uint32_t>(n1);
    int *L = pool.get<int>(n1), *E0 = pool.get<int>(n1), *Ea = pool.get<int>(n1), *Eb = pool.get<int>(n1);
    int* changed = pool.get<int>(1);
    unsigned long long* gcnt = pool.get<unsigned long long>(3);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    const int g = grid_for(n1);
    cudaError_t e = cudaSuccess;
    for (uint32_t* a : {toff, nsl, fl, fs, fsh, gsf})  // entry M stays 0, so each scan's entry M is the total
        if (e == cudaSuccess) e = cudaMemsetAsync(a + M, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(gcnt, 0, 3 * sizeof(unsigned long long), st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    plan_classify<<<g, kT, 0, st>>>(rp, M, o.pack_max, o.cta_max, o.seg_nnz, toff, nsl, fl, fs, fsh);
    ++launches;
    e = scan_exclusive(toff, toff, n1, pool);
    if (e == cudaSuccess) e = scan_exclusive(nsl, soff, n1, pool);
    if (e == cudaSuccess) e = scan_exclusive(fl, lidx, n1, pool);
    if (e == cudaSuccess) e = scan_exclusive(fs, sidx, n1, pool);
    uint32_t tot[4] = {0, 0, 0, 0};  // long-row tasks, slots, long rows, split rows
    if (e == cudaSuccess) e = cudaMemcpyAsync(&tot[0], toff + M, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&tot[1], soff + M, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&tot[2], lidx + M, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&tot[3], sidx + M, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    if (tot[1] > (1u << 23)) return SPX_ERR_INDEX_RANGE;  // a slot must fit the task word
    const int nL = static_cast<int>(tot[2]);
    plan_compact<<<g, kT, 0, st>>>(fl, lidx, M, L);
    plan_group_end<<<g, kT, 0, st>>>(rp, M, fl, L, nL, o.block_nnz, o.block_rows, E0, on);
    launches += 2;
    e = cudaMemcpyAsync(Ea, E0, sizeof(int) * static_cast<size_t>(n1), cudaMemcpyDeviceToDevice, st);
    // doubling: at most ceil(log2(M + 1)) + 1 rounds
    for (int round = 0; round < 34 && e == cudaSuccess; ++round) {
        int h = 0;
        e = cudaMemsetAsync(changed, 0, sizeof(int), st);
        if (e != cudaSuccess) break;
        plan_mark<<<g, kT, 0, st>>>(Ea, on, M);
        plan_compose<<<g, kT, 0, st>>>(Ea, Eb, M, changed);
        launches += 2;
        e = cudaMemcpyAsync(&h, changed, sizeof(int), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess || !h) break;
        std::swap(Ea, Eb);
    }
    if (e == cudaSuccess) {
        plan_starts<<<g, kT, 0, st>>>(on, fsh, M, gsf);
        ++launches;
        e = scan_exclusive(gsf, gidx, n1, pool);
    }
    uint32_t ngroups = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&ngroups, gidx + M, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    const long long nt = static_cast<long long>(tot[0]) + ngroups;
    if (nt > kI32Max) return SPX_ERR_INDEX_RANGE;
    int *htask = pool.get<int>(4 * nt), *dtask = pool.get<int>(4 * nt), *lrows = pool.get<int>(4ll * tot[3]);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    plan_write<<<g, kT, 0, st>>>(rp, M, o.seg_nnz, o.lanes_div, nsl, fl, fs, toff, soff, sidx, gsf, gidx, E0,
                                 static_cast<long long>(tot[0]), htask, dtask, lrows, gcnt);
    ++launches;
    const int nth = spx_group_threads(o.block_nnz);
    const long long nfirst = o.lanes_div == 0 ? static_cast<long long>(ngroups) * nth : 0;
    uint16_t* first = nfirst ? pool.get<uint16_t>(nfirst) : nullptr;
    if (pool.err != cudaSuccess) {
        cudaStreamSynchronize(st);
        return SPX_ERR_NOMEM;
    }
    if (nfirst) {
        plan_first<<<grid_for(nfirst), kT, 0, st>>>(rp, reinterpret_cast<const int4*>(dtask) + tot[0], ngroups, nth,
                                                    spx_group_per(o.block_nnz), first);
        ++launches;
    }
    unsigned long long gc[3] = {0, 0, 0};
    try {
        P->tasks.resize(static_cast<size_t>(4 * nt));
        P->dtasks.resize(static_cast<size_t>(4 * nt));
        P->longrows.resize(static_cast<size_t>(4) * tot[3]);
        P->first.resize(static_cast<size_t>(nfirst));
    } catch (const std::bad_alloc&) {
        cudaStreamSynchronize(st);
        return SPX_ERR_NOMEM;
    }
    e = cudaGetLastError();
    if (e == cudaSuccess && nt)
        e = cudaMemcpyAsync(P->tasks.data(), htask, sizeof(int) * 4 * static_cast<size_t>(nt), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && nt)
        e = cudaMemcpyAsync(P->dtasks.data(), dtask, sizeof(int) * 4 * static_cast<size_t>(nt), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && tot[3])
        e = cudaMemcpyAsync(P->longrows.data(), lrows, sizeof(int) * 4 * static_cast<size_t>(tot[3]),
                            cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && nfirst)
        e = cudaMemcpyAsync(P->first.data(), first, sizeof(uint16_t) * static_cast<size_t>(nfirst),
                            cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(gc, gcnt, sizeof(gc), cudaMemcpyDeviceToHost, st);
    spx_note_launches(launches);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    const int64_t c[9] = {nt, static_cast<int64_t>(tot[3]), static_cast<int64_t>(tot[1]),
                          static_cast<int64_t>(M) - tot[2], static_cast<int64_t>(tot[2]) - tot[3],
                          static_cast<int64_t>(tot[3]), static_cast<int64_t>(gc[0]), static_cast<int64_t>(gc[1]),
                          static_cast<int64_t>(gc[2])};
    std::memcpy(P->counts, c, sizeof(c));
    P->table_bytes = (P->dtasks.size() + P->longrows.size()) * sizeof(int32_t) + P->first.size() * sizeof(uint16_t);
    P->scratch_bytes = static_cast<size_t>(tot[1]) * sizeof(float);
    return SPX_OK;
}

spx_status spx_dev_build_sell(int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col,
                              const float* val, int32_t sigma, int32_t piece, spx_sell_dev_image* out,
                              cudaStream_t st) {
    *out = spx_sell_dev_image{};
    Pool pool(st);
    uint64_t launches = 0;
    int* bad = pool.get<int>(1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    if (cudaMemsetAsync(bad, 0, sizeof(int), st) != cudaSuccess) return SPX_ERR_CUDA;
    check_row_ptr<<<grid_for(M), kT, 0, st>>>(rp, M, nnz, bad);
    ++launches;
    if (nnz > 0) {
        check_indices<<<grid_for(nnz), kT, 0, st>>>(col, nnz, K, bad);
        ++launches;
    }
    int h = 0;
    spx_status s = read_flag(bad, st, &h);
    if (s != SPX_OK) return s;
    if (h & 4) return SPX_ERR_ARG;
    if (h & 2) return SPX_ERR_NOT_SORTED;
    if (h & 1) return SPX_ERR_INDEX_RANGE;
    // pseudo-rows per row, long rows, slots
    const long long n1 = static_cast<long long>(M) + 1;
    uint32_t *cnt = pool.get<uint32_t>(n1), *fl = pool.get<uint32_t>(n1), *nsl = pool.get<uint32_t>(n1);
    uint32_t *pst = pool.get<uint32_t>(n1), *lidx = pool.get<uint32_t>(n1), *lslot = pool.get<uint32_t>(n1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    cudaError_t e = cudaSuccess;
    for (uint32_t* a : {cnt, fl, nsl})
        if (e == cudaSuccess) e = cudaMemsetAsync(a + M, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess && M > 0) {
        sell_count<<<grid_for(M), kT, 0, st>>>(rp, M, piece, cnt, fl, nsl);
        ++launches;
    }
    if (e == cudaSuccess) e = scan_exclusive(cnt, pst, n1, pool);
    if (e == cudaSuccess) e = scan_exclusive(fl, lidx, n1, pool);
    if (e == cudaSuccess) e = scan_exclusive(nsl, lslot, n1, pool);
    uint32_t tot[3] = {0, 0, 0};  // pseudo-rows, long rows, slots
    if (e == cudaSuccess) e = cudaMemcpyAsync(&tot[0], pst + M, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&tot[1], lidx + M, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&tot[2], lslot + M, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    const long long np = tot[0], nlong = tot[1], slots = tot[2];
    if (slots > kI32Max || np > kI32Max - kSellC) return SPX_ERR_INDEX_RANGE;
    const long long ns = (np + kSellC - 1) / kSellC;
    int *plen = pool.get<int>(np), *prow = pool.get<int>(np), *pstart = pool.get<int>(np), *pslot = pool.get<int>(np);
    int* lrows = pool.get<int>(4 * nlong);
    uint32_t *k = pool.get<uint32_t>(np), *k2 = pool.get<uint32_t>(np), *width = pool.get<uint32_t>(ns + 1);
    uint32_t* sp = pool.get<uint32_t>(ns + 1);
    int *ix = pool.get<int>(np), *ix2 = pool.get<int>(np);
    unsigned long long* acc = pool.get<unsigned long long>(1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    if (M > 0) {
        sell_pseudo<<<grid_for(M), kT, 0, st>>>(rp, M, piece, pst, fl, lidx, lslot, plen, prow, pstart, pslot, lrows);
        ++launches;
    }
    // longest first, stably, inside windows of sigma pseudo-rows (LSD: length, then window)
    if (np > 0) {
        sell_len_keys<<<grid_for(np), kT, 0, st>>>(plen, piece, k, ix, np);
        ++launches;
        e = radix_sort(k, ix, k2, ix2, np, bits_for(static_cast<long long>(piece) + 1), pool, launches);
        const long long nwin = (np + sigma - 1) / sigma;
        if (e == cudaSuccess && bits_for(nwin) > 0) {
            sell_win_keys<<<grid_for(np), kT, 0, st>>>(ix, sigma, k, np);
            ++launches;
            e = radix_sort(k, ix, k2, ix2, np, bits_for(nwin), pool, launches);
        }
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(width + ns, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(acc, 0, sizeof(unsigned long long), st);
    if (e == cudaSuccess && ns > 0) {
        sell_slices<<<grid_for(ns), kT, 0, st>>>(ix, plen, ns, width, acc);
        ++launches;
    }
    if (e == cudaSuccess) e = scan_exclusive(width, sp, ns + 1, pool);
    unsigned long long padded = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&padded, acc, sizeof(padded), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    if (padded > static_cast<unsigned long long>(kI32Max)) return SPX_ERR_INDEX_RANGE;
    // the image (same layout as the host builder's), allocated for the caller
    auto a16 = [](size_t n) { return (n + 15) & ~static_cast<size_t>(15); };
    spx_sell_dev_image img;
    img.off_prow = a16(sizeof(int32_t) * static_cast<size_t>(ns + 1));
    img.off_long = img.off_prow + a16(sizeof(int32_t) * static_cast<size_t>(ns * kSellC));
    img.off_col = img.off_long + a16(sizeof(int32_t) * static_cast<size_t>(4 * nlong));
    img.off_val = img.off_col + a16(sizeof(int32_t) * static_cast<size_t>(padded));
    img.bytes = img.off_val + a16(sizeof(float) * static_cast<size_t>(padded));
    if (cudaMalloc(&img.image, img.bytes) != cudaSuccess) {
        cudaGetLastError();  // clear the allocation error
        return SPX_ERR_NOMEM;
    }
    char* d = static_cast<char*>(img.image);
    int* prow_out = reinterpret_cast<int*>(d + img.off_prow);
    int* scol = reinterpret_cast<int*>(d + img.off_col);
    float* sval = reinterpret_cast<float*>(d + img.off_val);
    e = cudaMemcpyAsync(d, sp, sizeof(uint32_t) * static_cast<size_t>(ns + 1), cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && nlong)
        e = cudaMemcpyAsync(d + img.off_long, lrows, sizeof(int) * static_cast<size_t>(4 * nlong),
                            cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && padded) e = cudaMemsetAsync(scol, 0xFF, sizeof(int) * padded, st);  // -1: padding
    if (e == cudaSuccess && padded) e = cudaMemsetAsync(sval, 0, sizeof(float) * padded, st);
    if (e == cudaSuccess && ns > 0) {
        fill_i32<<<grid_for(ns * kSellC), kT, 0, st>>>(prow_out, ns * kSellC, INT32_MIN);  // unused tail lanes
        sell_scatter<<<grid_for(np), kT, 0, st>>>(ix, plen, prow, pstart, pslot, sp, col, val, np, prow_out, scol,
                                                  sval);
        launches += 2;
        e = cudaGetLastError();
    }
    spx_note_launches(launches);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        cudaFree(img.image);
        return SPX_ERR_CUDA;
    }
    img.nslices = ns;
    img.pseudo_rows = np;
    img.padded = static_cast<int64_t>(padded);
    img.nlong = nlong;
    img.slots = slots;
    *out = img;
    return SPX_OK;
}
