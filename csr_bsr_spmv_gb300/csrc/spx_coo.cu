// spx_coo.cu -- COO SpMV y = alpha*A*x + beta*y over row-sorted triplets on sm_103a.
//
// [Formats] §1 (COO: one (row, col, val) triplet per stored entry) and the
// COO row of the dispatch rule table of [SpMM-ops] §4: the work is split by
// nonzeros, not by rows, so a row's length never unbalances the launch.
//
// Launch 1 cuts the triplets into chunks of kChunk consecutive entries, one
// CTA each.  The CTA streams its chunk once (coalesced), multiplies by the
// gathered x, and thread t sums its kPer consecutive products run by run
// (a run = consecutive entries of one row).  Runs that cross threads are
// joined by a segmented block scan.  A run that both starts and ends in the
// chunk is finished in place (alpha/beta epilogue).  The chunk's first run,
// when its row began in an earlier chunk, leaves its sum in head[c]; the
// chunk's last run, when its row goes on into the next chunk, leaves its sum
// in tail[c].  Launch 2 (one thread per chunk) finishes every row that ended
// in chunk c but began before it: head[c] + tail[c-1] + tail[c-2] + ... back
// to the chunk where the row began, in that fixed order.  No floating-point
// atomics, so the result is bitwise reproducible.
//
// Rows without entries get y = beta*y (0 when beta == 0), written by the
// thread holding the first entry after the gap.  Out-of-range indices and
// rows out of order are skipped and recorded in an error word
// (spx_last_device_error); they never cause an out-of-bounds access.
#include <cuda_runtime.h>

#include "spx_carveout.cuh"
#include "spx_gather.cuh"
#include "spx_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kPer = 8;                   // consecutive entries per thread
constexpr int kChunk = kThreads * kPer;   // 2048 entries per CTA
constexpr unsigned kFull = 0xffffffffu;

__device__ int g_coo_error;

__device__ __forceinline__ void coo_error(int code) { atomicCAS(&g_coo_error, 0, code); }

// Skewed shared-memory slot: one padding word per 32, so both the strided
// fill (k = t + 256 j) and the blocked walk (k = 8 t .. 8 t + 7) are free of
// bank conflicts.
__device__ __forceinline__ int sk(int k) { return k + (k >> 5); }

__device__ __forceinline__ void finish_row(float* y, int r, float s, float alpha, float beta) {
    y[r] = beta != 0.f ? alpha * s + beta * y[r] : alpha * s;
}


// Register budget for 8 resident CTAs per SM (32 registers): more warps beat
// more registers here (measured 399 us against 419 us at 6 and 458 us at 4 CTAs).
constexpr int kMinBlocks = 8;
constexpr int kYCache = 512;  // rows of old y a chunk reads up front

__global__ void __launch_bounds__(kThreads, kMinBlocks) coo_chunk_kernel(int M, int K, long long nnz,
                                                             const int* __restrict__ row,
                                                             const int* __restrict__ col,
                                                             const float* __restrict__ val,
                                                             const float* __restrict__ x, float alpha, float beta,
                                                             float* y, float* __restrict__ head,
                                                             float* __restrict__ tail) {
    __shared__ int s_row[kChunk + kChunk / 32];
    __shared__ float s_prod[kChunk + kChunk / 32];
    __shared__ float s_sv[kThreads / 32];
    __shared__ int s_sf[kThreads / 32];
    __shared__ float s_y[kYCache];
    const long long c = blockIdx.x;
    const long long base = c * kChunk;
    const int n = static_cast<int>(min(static_cast<long long>(kChunk), nnz - base));
    const bool first_chunk = c == 0, last_chunk = base + n == nnz;
    // Rows just outside the chunk; -1 / M mean "none".
    const int prev_row = first_chunk ? -1 : __ldg(row + base - 1);
    const int next_row = last_chunk ? M : __ldg(row + base + n);
    // The old y of the chunk's rows [rfirst, rlast] is read up front, with the
    // entries, when the span is short: no row waits on it when it finishes.
    const int rfirst = __ldg(row + base), rlast = __ldg(row + base + n - 1);
    const bool ycache = beta != 0.f && rfirst >= 0 && rlast < M && rfirst <= rlast && rlast - rfirst < kYCache;
    if (ycache)
        for (int i = threadIdx.x; i <= rlast - rfirst; i += kThreads) s_y[i] = y[rfirst + i];
    auto old_y = [&](int r) { return ycache && r >= rfirst && r <= rlast ? s_y[r - rfirst] : y[r]; };
    auto finish = [&](int r, float total) { y[r] = beta != 0.f ? alpha * total + beta * old_y(r) : alpha * total; };
    auto empties = [&](int from, int to) {  // rows [from, to) without entries, clamped to [0, M)
        for (int r = max(from, 0); r < min(to, M); ++r) y[r] = beta != 0.f ? beta * old_y(r) : 0.f;
    };

    // 1. stage rows and products, coalesced: all loads of the thread first, then
    //    all its gathers, so kPer of each are in flight at once
    int rr[kPer], cc[kPer];
    float vv[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int k = threadIdx.x + j * kThreads;
        rr[j] = k < n ? spx_gather::ld_once(row + base + k) : 0;
        cc[j] = k < n ? spx_gather::ld_once(col + base + k) : 0;
        vv[j] = k < n ? spx_gather::ld_once(val + base + k) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const bool in = cc[j] >= 0 && cc[j] < K;
        vv[j] = in ? vv[j] * spx_gather::ld_x(x + cc[j]) : 0.f;
        if (!in && threadIdx.x + j * kThreads < n) coo_error(static_cast<int>(SPX_ERR_INDEX_RANGE));
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int k = threadIdx.x + j * kThreads;
        if (k < n) {
            s_row[sk(k)] = rr[j];
            s_prod[sk(k)] = vv[j];
        }
    }
    __syncthreads();

    // 2. walk this thread's entries [k0, k1) run by run
    const int k0 = threadIdx.x * kPer, k1 = min(k0 + kPer, n);
    float s = 0.f, first_part = 0.f;
    int flag = 1;                 // 1: the thread's trailing run started in this thread
    int first_run_row = -1;       // row of a first run that started before this thread and ends in it
    if (k0 < k1) {
        int prev = k0 > 0 ? s_row[sk(k0 - 1)] : prev_row;
        bool carry_in = true;     // the current run may have started before this thread
        for (int k = k0; k < k1; ++k) {
            const int r = s_row[sk(k)];
            if (r < 0 || r >= M) {  // out of range: skip the entry
                coo_error(static_cast<int>(SPX_ERR_INDEX_RANGE));
                continue;
            }
            if (r != prev) {
                if (r < prev) {  // out of order: skip the entry
                    coo_error(static_cast<int>(SPX_ERR_NOT_SORTED));
                    continue;
                }
                // the run of `prev` ended at k - 1
                if (k > k0) {
                    if (carry_in) {  // the run entering this thread: finished after the scan
                        first_part = s;
                        first_run_row = prev;
                    } else {         // began and ended in this thread
                        finish(prev, s);
                    }
                }
                carry_in = false;
                s = 0.f;
                empties(prev + 1, r);  // rows strictly between prev and r
                prev = r;
            }
            s += s_prod[sk(k)];
        }
        flag = carry_in ? 0 : 1;
        if (last_chunk && k1 == n) empties(prev + 1, M);
    }

    // 3. inclusive segmented scan of (flag, s) over the threads:
    //    (f1, v1) + (f2, v2) = (f1 | f2, f2 ? v2 : v1 + v2)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float v = s;
    int f = flag;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float v2 = __shfl_up_sync(kFull, v, d);
        const int f2 = __shfl_up_sync(kFull, f, d);
        if (lane >= d) {
            if (!f) v = v2 + v;
            f |= f2;
        }
    }
    if (lane == 31) {
        s_sv[warp] = v;
        s_sf[warp] = f;
    }
    __syncthreads();
    float wp = 0.f;  // carry from the earlier warps, in warp order
    for (int i = 0; i < warp; ++i) wp = s_sf[i] ? s_sv[i] : wp + s_sv[i];
    float ex = __shfl_up_sync(kFull, v, 1);
    int exf = __shfl_up_sync(kFull, f, 1);
    if (lane == 0) {
        ex = 0.f;
        exf = 0;
    }
    const float carry = exf ? ex : wp + ex;  // sum of the run entering this thread

    if (k0 >= k1) return;
    // 4. emit the run that entered this thread (if it ended here) and the trailing run
    auto emit = [&](int r, float total) {
        if (r == next_row) tail[c] = total;       // goes on into the next chunk
        else if (r == prev_row) head[c] = total;  // began in an earlier chunk
        else finish(r, total);
    };
    if (first_run_row >= 0) emit(first_run_row, carry + first_part);
    const int r_last = s_row[sk(k1 - 1)];
    const int r_after = k1 < n ? s_row[sk(k1)] : next_row;
    // the trailing run ends here unless the next thread of this chunk continues it
    if ((k1 == n || r_last != r_after) && r_last >= 0 && r_last < M) emit(r_last, flag ? s : carry + s);
}

// One thread per chunk: finish the row whose run ended in chunk c but began in an earlier chunk.
__global__ void __launch_bounds__(kThreads) coo_fixup_kernel(int M, long long nnz, long long nchunks,
                                                             const int* __restrict__ row,
                                                             const float* __restrict__ head,
                                                             const float* __restrict__ tail, float alpha, float beta,
                                                             float* y) {
    const long long c = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x;
    if (c == 0 || c >= nchunks) return;
    const long long base = c * kChunk;
    const int first = __ldg(row + base);
    if (first != __ldg(row + base - 1)) return;                 // no run entering this chunk
    if (c + 1 < nchunks && first == __ldg(row + base + kChunk)) return;  // the run also leaves it
    if (first < 0 || first >= M) return;
    float total = head[c];
    for (long long d = c - 1;; --d) {
        total += tail[d];
        const long long b = d * kChunk;
        if (d == 0 || __ldg(row + b) != first || __ldg(row + b - 1) != first) break;  // the row began in chunk d
    }
    finish_row(y, first, total, alpha, beta);
}

__global__ void __launch_bounds__(kThreads) coo_scale_kernel(int M, float beta, float* y) {
    const int i = blockIdx.x * kThreads + threadIdx.x;
    if (i < M) y[i] = beta != 0.f ? beta * y[i] : 0.f;
}

}  // namespace

int spx_coo_error_take() {
    int h = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_coo_error, sizeof(int)) != cudaSuccess) return static_cast<int>(SPX_ERR_CUDA);
    if (h != 0 && cudaMemcpyToSymbol(g_coo_error, &zero, sizeof(int)) != cudaSuccess)
        return static_cast<int>(SPX_ERR_CUDA);
    return h;
}

extern "C" {

size_t spx_spmv_coo_scratch_bytes(int64_t nnz) {
    if (nnz <= 0) return 0;
    return 2 * sizeof(float) * static_cast<size_t>((nnz + kChunk - 1) / kChunk);
}

spx_status spx_spmv_coo(int32_t M, int32_t K, int64_t nnz, const int32_t* coo_row, const int32_t* coo_col,
                        const float* coo_val, float alpha, const float* x, float beta, float* y, void* scratch,
                        size_t scratch_bytes, spx_stream_t stream) {
    if (M < 0 || K < 0 || nnz < 0) return SPX_ERR_ARG;
    if (nnz > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (M == 0) return nnz == 0 ? SPX_OK : SPX_ERR_INDEX_RANGE;
    if (!y || (nnz > 0 && (!coo_row || !coo_col || !coo_val || !x))) return SPX_ERR_ARG;
    if (!spx_aligned(y, 4) || (nnz > 0 && (!spx_aligned(coo_row, 4) || !spx_aligned(coo_col, 4) ||
                                           !spx_aligned(coo_val, 4) || !spx_aligned(x, 4))))
        return SPX_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (nnz == 0) {
        coo_scale_kernel<<<(M + kThreads - 1) / kThreads, kThreads, 0, st>>>(M, beta, y);
        spx_note_launches(1);
        return spx_cuda_status(cudaGetLastError());
    }
    const size_t need = spx_spmv_coo_scratch_bytes(nnz);
    if (!scratch || scratch_bytes < need) return SPX_ERR_ARG;
    if (!spx_aligned(scratch, 4)) return SPX_ERR_ALIGN;
    // x and y must not overlap: y is written while x is still being gathered
    const char* xb = reinterpret_cast<const char*>(x);
    const char* yb = reinterpret_cast<const char*>(y);
    if (xb < yb + 4 * static_cast<size_t>(M) && yb < xb + 4 * static_cast<size_t>(K)) return SPX_ERR_ARG;
    const long long nchunks = (nnz + kChunk - 1) / kChunk;
    float* head = static_cast<float*>(scratch);
    float* tail = head + nchunks;
    spx_carve::fit(coo_chunk_kernel, kThreads, 0);
    coo_chunk_kernel<<<static_cast<unsigned>(nchunks), kThreads, 0, st>>>(M, K, nnz, coo_row, coo_col, coo_val, x,
                                                                          alpha, beta, y, head, tail);
    uint64_t launches = 1;
    if (nchunks > 1) {
        coo_fixup_kernel<<<static_cast<unsigned>((nchunks + kThreads - 1) / kThreads), kThreads, 0, st>>>(
            M, nnz, nchunks, coo_row, head, tail, alpha, beta, y);
        ++launches;
    }
    spx_note_launches(launches);
    return spx_cuda_status(cudaGetLastError());
}

}  // extern "C"
