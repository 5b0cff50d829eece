// spx_spmv.cu -- CSR SpMV y = alpha*A*x + beta*y on sm_103a, and the
// two-direction operator pair u = A v ..., v = A^T u ... over CSR(A)/CSR(A^T).
//
// One launch serves the whole task table of the plan ([SpMM-ops] §2.1-§2.4):
//   group  : a run of consecutive short rows (<= B nonzeros).  The CTA streams
//            the group's values/column indices once, coalesced, gathers x
//            through the read-only path, parks the products in shared memory,
//            then reduces each row with w lanes (w = 1: thread per row,
//            w = 32: warp per row) and a shuffle tree.
//   cta    : one row of hundreds..thousands of nonzeros; all threads stride it,
//            warp shuffles then a fixed-order reduction of the warp sums.
//   seg    : one segment of a split long row; writes a partial sum.
// A second small launch (one warp per split row) adds the partial sums in a
// fixed order and applies the epilogue ([SpMM-ops] §2.4: partial buffer plus
// second-stage reduction; no floating-point atomics, so results are bitwise
// reproducible).
//
// Matrix streams (values, column indices) are read with the evict-first
// (streaming) cache hint so that x -- the gathered operand -- keeps its L2
// residency ([SpMM-ops] §2.5).
#include <cuda_runtime.h>

#include "spx_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float ld_stream(const float* p) { return __ldcs(p); }
__device__ __forceinline__ int ld_stream(const int* p) { return __ldcs(p); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_down_sync(0xffffffffu, v, d);
    return v;
}

// Sum of v over the NT threads of the CTA in a fixed order; result valid in thread 0.
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
    if (warp == 0) {
        s = lane < kWarps ? red[lane] : 0.f;
        s = warp_sum(s);
    }
    return s;
}

// Strided dot product of a nonzero range [a, b) with x; 4 loads in flight per thread.
__device__ __forceinline__ float range_dot(int a, int b, const int* __restrict__ col, const float* __restrict__ val,
                                           const float* __restrict__ x) {
    float s = 0.f;
    int p = a + threadIdx.x;
    for (; p + 3 * kThreads < b; p += 4 * kThreads) {
        int c0 = ld_stream(col + p), c1 = ld_stream(col + p + kThreads);
        int c2 = ld_stream(col + p + 2 * kThreads), c3 = ld_stream(col + p + 3 * kThreads);
        float v0 = ld_stream(val + p), v1 = ld_stream(val + p + kThreads);
        float v2 = ld_stream(val + p + 2 * kThreads), v3 = ld_stream(val + p + 3 * kThreads);
        float x0 = __ldg(x + c0), x1 = __ldg(x + c1), x2 = __ldg(x + c2), x3 = __ldg(x + c3);
        s += v0 * x0;
        s += v1 * x1;
        s += v2 * x2;
        s += v3 * x3;
    }
    for (; p < b; p += kThreads) s += ld_stream(val + p) * __ldg(x + ld_stream(col + p));
    return s;
}

__device__ __forceinline__ float epilogue(float s, float alpha, float beta, const float* y, int row) {
    float r = alpha * s;
    if (beta != 0.f) r += beta * y[row];
    return r;
}

// ITEMS = block_nnz / kThreads when it is a compile-time case, else 0 (loop).
template <int ITEMS>
__device__ __forceinline__ void group_task(int r0, int r1, int lg, const int* __restrict__ rp,
                                           const int* __restrict__ col, const float* __restrict__ val,
                                           const float* __restrict__ x, float alpha, float beta, float* y,
                                           float* s_prod, int* s_rp) {
    const int p0 = __ldg(rp + r0);
    const int nrows = r1 - r0;
    const int n = __ldg(rp + r1) - p0;
    for (int i = threadIdx.x; i <= nrows; i += kThreads) s_rp[i] = __ldg(rp + r0 + i) - p0;
    if (ITEMS > 0) {
        int c[ITEMS > 0 ? ITEMS : 1];
        float v[ITEMS > 0 ? ITEMS : 1];
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int k = threadIdx.x + j * kThreads;
            c[j] = k < n ? ld_stream(col + p0 + k) : 0;
            v[j] = k < n ? ld_stream(val + p0 + k) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int k = threadIdx.x + j * kThreads;
            if (k < n) s_prod[k] = v[j] * __ldg(x + c[j]);
        }
    } else {
        for (int k = threadIdx.x; k < n; k += kThreads) s_prod[k] = ld_stream(val + p0 + k) * __ldg(x + ld_stream(col + p0 + k));
    }
    __syncthreads();
    // reduce each row with w = 2^lg lanes; every lane of a warp runs the same trip count
    const int w = 1 << lg;
    const int sub = threadIdx.x >> lg, lane = threadIdx.x & (w - 1);
    const int nsub = kThreads >> lg;
    for (int base = 0; base < nrows; base += nsub) {
        const int r = base + sub;
        float s = 0.f;
        if (r < nrows) {
            const int a = s_rp[r], b = s_rp[r + 1];
            for (int k = a + lane; k < b; k += w) s += s_prod[k];
        }
        for (int d = 16; d > 0; d >>= 1)
            if (d < w) s += __shfl_down_sync(0xffffffffu, s, d, w);
        if (r < nrows && lane == 0) y[r0 + r] = epilogue(s, alpha, beta, y, r0 + r);
    }
}

template <int ITEMS>
__global__ void __launch_bounds__(kThreads) spmv_tasks_kernel(const int4* __restrict__ tasks,
                                                              const int* __restrict__ rp, const int* __restrict__ col,
                                                              const float* __restrict__ val,
                                                              const float* __restrict__ x, float alpha, float beta,
                                                              float* y, float* __restrict__ partials, int seg_nnz,
                                                              int block_nnz) {
    extern __shared__ __align__(16) float smem[];
    const int4 t = tasks[blockIdx.x];
    const int kind = t.x & 255;
    if (kind == kTaskGroup) {
        group_task<ITEMS>(t.y, t.z, t.x >> 8, rp, col, val, x, alpha, beta, y, smem,
                          reinterpret_cast<int*>(smem + block_nnz));
    } else if (kind == kTaskCta) {
        const int row = t.y;
        float s = range_dot(__ldg(rp + row), __ldg(rp + row + 1), col, val, x);
        s = block_sum(s, smem);
        if (threadIdx.x == 0) y[row] = epilogue(s, alpha, beta, y, row);
    } else {
        const int row = t.y;
        const int a = __ldg(rp + row), b = __ldg(rp + row + 1);
        const long long lo = (long long)a + (long long)t.z * seg_nnz;
        const int hi = (int)min((long long)b, lo + seg_nnz);
        float s = range_dot((int)lo, hi, col, val, x);
        s = block_sum(s, smem);
        if (threadIdx.x == 0) partials[t.w] = s;
    }
}

// One warp per split row: fixed-order sum of its segment partials, then the epilogue.
__global__ void __launch_bounds__(kThreads) spmv_fixup_kernel(const int4* __restrict__ longrows, int nlong,
                                                              const float* __restrict__ partials, float alpha,
                                                              float beta, float* y) {
    const int w = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= nlong) return;
    const int4 lr = longrows[w];
    float s = 0.f;
    for (int k = lane; k < lr.z; k += 32) s += partials[lr.y + k];
    s = warp_sum(s);
    if (lane == 0) y[lr.x] = epilogue(s, alpha, beta, y, lr.x);
}

spx_status launch_spmv(const spx_plan* P, const int* rp, const int* col, const float* val, float alpha,
                       const float* x, float beta, float* y, float* scratch, cudaStream_t st) {
    const int ntasks = static_cast<int>(P->counts[0]);
    const int nlong = static_cast<int>(P->counts[1]);
    if (ntasks == 0) return SPX_OK;
    const int4* tasks = static_cast<const int4*>(P->d_table);
    const int4* longrows = tasks + ntasks;
    const int B = P->opts.block_nnz;
    const size_t smem = sizeof(float) * static_cast<size_t>(B) + sizeof(int) * (static_cast<size_t>(P->opts.block_rows) + 1);
    const int seg = P->opts.seg_nnz;
    switch (B) {
        case kThreads * 4:
            spmv_tasks_kernel<4><<<ntasks, kThreads, smem, st>>>(tasks, rp, col, val, x, alpha, beta, y, scratch, seg, B);
            break;
        case kThreads * 8:
            spmv_tasks_kernel<8><<<ntasks, kThreads, smem, st>>>(tasks, rp, col, val, x, alpha, beta, y, scratch, seg, B);
            break;
        case kThreads * 16:
            spmv_tasks_kernel<16><<<ntasks, kThreads, smem, st>>>(tasks, rp, col, val, x, alpha, beta, y, scratch, seg, B);
            break;
        default:
            spmv_tasks_kernel<0><<<ntasks, kThreads, smem, st>>>(tasks, rp, col, val, x, alpha, beta, y, scratch, seg, B);
            break;
    }
    uint64_t launches = 1;
    if (nlong > 0) {
        spmv_fixup_kernel<<<(nlong + kWarps - 1) / kWarps, kThreads, 0, st>>>(longrows, nlong, scratch, alpha, beta, y);
        ++launches;
    }
    spx_note_launches(launches);
    return spx_cuda_status(cudaGetLastError());
}

spx_status check_call(const spx_plan* P, int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col,
                      const float* val, const float* x, const float* y, const void* scratch, size_t scratch_bytes) {
    if (!spx_plan_ok(P)) return SPX_ERR_ARG;
    if (P->M != M || P->K != K || P->nnz != nnz) return SPX_ERR_ARG;
    if (P->table_bytes > 0 && !P->d_table) return SPX_ERR_NOT_READY;
    if (M == 0) return SPX_OK;
    if (!rp || !y || (nnz > 0 && (!col || !val || !x))) return SPX_ERR_ARG;
    if (P->scratch_bytes > 0 && (!scratch || scratch_bytes < P->scratch_bytes)) return SPX_ERR_ARG;
    if (!spx_aligned(rp, 4) || !spx_aligned(col, 4) || !spx_aligned(val, 4) || !spx_aligned(x, 4) ||
        !spx_aligned(y, 4) || !spx_aligned(scratch, 4))
        return SPX_ERR_ALIGN;
    if (x && x < y + M && y < x + K) return SPX_ERR_ARG;  // x and y overlap
    return SPX_OK;
}

}  // namespace

extern "C" {

spx_status spx_spmv_csr(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr,
                        const int32_t* col, const float* val, float alpha, const float* x, float beta, float* y,
                        void* scratch, size_t scratch_bytes, spx_stream_t stream) {
    spx_status s = check_call(plan, M, K, nnz, row_ptr, col, val, x, y, scratch, scratch_bytes);
    if (s != SPX_OK || M == 0) return s;
    return launch_spmv(plan, row_ptr, col, val, alpha, x, beta, y, static_cast<float*>(scratch),
                       reinterpret_cast<cudaStream_t>(stream));
}

spx_status spx_spmv_csr_dual(const spx_plan* pA, const spx_plan* pAt, int32_t m, int32_t n, int64_t nnz,
                             const int32_t* A_rp, const int32_t* A_col, const float* A_val, const int32_t* At_rp,
                             const int32_t* At_col, const float* At_val, float* v, float alpha_u, float beta_u,
                             float* u, float alpha_v, float beta_v, void* scratch, size_t scratch_bytes,
                             spx_stream_t stream) {
    spx_status s = check_call(pA, m, n, nnz, A_rp, A_col, A_val, v, u, scratch, scratch_bytes);
    if (s == SPX_OK) s = check_call(pAt, n, m, nnz, At_rp, At_col, At_val, u, v, scratch, scratch_bytes);
    if (s != SPX_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (m > 0) s = launch_spmv(pA, A_rp, A_col, A_val, alpha_u, v, beta_u, u, static_cast<float*>(scratch), st);
    if (s == SPX_OK && n > 0)
        s = launch_spmv(pAt, At_rp, At_col, At_val, alpha_v, u, beta_v, v, static_cast<float*>(scratch), st);
    return s;
}

}  // extern "C"
