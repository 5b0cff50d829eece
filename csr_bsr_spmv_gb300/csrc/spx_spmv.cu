// spx_spmv.cu -- CSR SpMV y = alpha*A*x + beta*y on sm_103a, and the
// two-direction operator pair u = A v ..., v = A^T u ... over CSR(A)/CSR(A^T).
//
// One launch serves the whole task table of the plan ([SpMM-ops] §2.1-§2.4):
//   group  : a run of consecutive short rows (<= B nonzeros).  The CTA streams
//            the group's values/column indices once, coalesced, gathers x
//            through the read-only path and parks the products in shared
//            memory.  Then either
//              - lanes mode: each row is reduced by w lanes (w = 1: thread per
//                row, w = 32: warp per row) with a shuffle tree, or
//              - segmented mode: thread t sums the products [t*P, t*P + P)
//                whatever rows they belong to, rows that cross threads are
//                joined by a segmented block scan -- the same work per thread
//                however the row lengths vary ([Formats] §6, merge-based).
//   cta    : one row of hundreds..thousands of nonzeros; all threads stride it,
//            warp shuffles then a fixed-order reduction of the warp sums.
//   seg    : one segment of a split long row; writes a partial sum.
// A second small launch (one warp per split row) adds the partial sums in a
// fixed order and applies the epilogue ([SpMM-ops] §2.4: partial buffer plus
// second-stage reduction).  No floating-point atomics anywhere, so results are
// bitwise reproducible run to run.
//
// Each task carries its nonzero range, so a CTA issues its value/column loads
// right after reading the task.  Values and column indices are read with the
// streaming hint (no L1 allocation) so that x -- the gathered operand -- keeps
// its L1 and L2 residency ([SpMM-ops] §2.5).
#include <cuda_runtime.h>

#include <mutex>

#include "spx_carveout.cuh"
#include "spx_check.cuh"
#include "spx_gather.cuh"
#include "spx_internal.h"

namespace {

constexpr int kThreads = 256;  // fix-up kernel

SPX_CHECK_WORD(g_spmv_check)
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float ld_stream(const float* p) { return spx_gather::ld_once(p); }
__device__ __forceinline__ int ld_stream(const int* p) { return spx_gather::ld_once(p); }
using spx_gather::ld_x;

// Programmatic dependent launch (a kernel launched with programmatic stream
// serialization may start while the kernel before it on the stream is still
// running): let_dependents_start() lets the next kernel's CTAs be scheduled
// as this grid's SMs free up; predecessor_done() waits until the previous
// kernel has finished and its writes are visible.  Both are no-ops for a
// kernel launched the ordinary way.
__device__ __forceinline__ void let_dependents_start() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void predecessor_done() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_down_sync(kFull, v, d);
    return v;
}

// Sum of v over the CTA (NT threads) in a fixed order; result valid in thread 0.
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
    if (warp == 0) {
        s = lane < NT / 32 ? red[lane] : 0.f;
        s = warp_sum(s);
    }
    return s;
}

// x[c]; the checked build loads it only for a column inside [0, K) (else 0).
__device__ __forceinline__ float gather_x(const float* __restrict__ x, int c, int K) {
    if (SPX_CHECKED && (c < 0 || c >= K)) {
        check_fail();
        return 0.f;
    }
    return ld_x(x + c);
}

// Strided dot product of the nonzero range [a, b) with x: each thread takes its
// entries eight at a time (all eight loads, then all eight gathers in flight),
// the last batch predicated, and sums them in index order.
template <int NT>
__device__ __forceinline__ float range_dot(int a, int b, const int* __restrict__ col, const float* __restrict__ val,
                                           const float* __restrict__ x, int K) {
    float s = 0.f;
    for (int p = a + threadIdx.x; p < b; p += 8 * NT) {
        const int m = (b - p + NT - 1) / NT;  // entries of this batch (8 but in the last)
        int c[8];
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c[j] = j < m ? ld_stream(col + p + j * NT) : 0;
            v[j] = j < m ? ld_stream(val + p + j * NT) : 0.f;
        }
        float xv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) xv[j] = j < m ? gather_x(x, c[j], K) : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < m) s += v[j] * xv[j];
    }
    return s;
}

__device__ __forceinline__ void emit(float* y, int row, float s, float alpha, float beta) {
    float r = alpha * s;
    if (beta != 0.f) r += beta * y[row];
    y[row] = r;
}

// Group epilogue: the old y of the group's rows was prefetched into s_y with the
// products, so no row waits on a dependent global read here.
__device__ __forceinline__ void emit_g(float* y, const float* s_y, int r0, int r, float s, float alpha, float beta) {
    float v = alpha * s;
    if (beta != 0.f) v += beta * s_y[r];
    y[r0 + r] = v;
}

// Shared-memory slot of product k: one padding word after every 32 products,
// so both the strided writes (thread t: k = t + 256 j) and the blocked reads
// of the segmented mode (thread t: k = t*P .. t*P + P-1) hit 32 distinct banks.
__device__ __forceinline__ int sk(int k) { return k + (k >> 5); }

// Products val[p0+k] * x[col[p0+k]], k < n, into s_prod[sk(k)] (coalesced layout);
// ITEMS = block_nnz / NT as a compile-time case, 0 = runtime loop.
template <int NT, int ITEMS>
__device__ __forceinline__ void stage_products(int p0, int n, const int* __restrict__ col,
                                               const float* __restrict__ val, const float* __restrict__ x, int K,
                                               float* s_prod) {
    if (ITEMS > 0) {
        int c[ITEMS > 0 ? ITEMS : 1];
        float v[ITEMS > 0 ? ITEMS : 1];
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int k = threadIdx.x + j * NT;
            c[j] = k < n ? ld_stream(col + p0 + k) : 0;
            v[j] = k < n ? ld_stream(val + p0 + k) : 0.f;
        }
        predecessor_done();  // x may be the previous kernel's output: the matrix loads above are already in flight
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int k = threadIdx.x + j * NT;
            if (k < n) s_prod[sk(k)] = v[j] * gather_x(x, c[j], K);
        }
    } else {
        predecessor_done();
        for (int k = threadIdx.x; k < n; k += NT)
            s_prod[sk(k)] = ld_stream(val + p0 + k) * gather_x(x, ld_stream(col + p0 + k), K);
    }
}

// Lanes mode: each row reduced by w = 2^lg lanes; every lane of a warp runs the same trip count.
template <int NT>
__device__ __forceinline__ void reduce_lanes(int r0, int nrows, int lg, const float* s_prod, const int* s_rp,
                                             const float* s_y, float alpha, float beta, float* y) {
    const int w = 1 << lg;
    const int sub = threadIdx.x >> lg, lane = threadIdx.x & (w - 1);
    const int nsub = NT >> lg;
    for (int base = 0; base < nrows; base += nsub) {
        const int r = base + sub;
        float s = 0.f;
        if (r < nrows) {
            const int a = s_rp[r], b = s_rp[r + 1];
            for (int k = a + lane; k < b; k += w) s += s_prod[sk(k)];
        }
        for (int d = 16; d > 0; d >>= 1)
            if (d < w) s += __shfl_down_sync(kFull, s, d, w);
        if (r < nrows && lane == 0) emit_g(y, s_y, r0, r, s, alpha, beta);
    }
}

// Segmented mode: thread t owns products [t*per, t*per + per).  Rows that end
// inside a thread's run are written by that thread; a row crossing threads
// is finished by the thread holding its last product, which adds the carry
// from an inclusive segmented scan of the threads' trailing partial sums.
// The row holding the thread's first product, and whether that row started
// before it, come from the plan (fr = spx_first_entry), so no thread searches
// the row offsets between the product barrier and its sums.
template <int PER>
__device__ __forceinline__ void reduce_segmented(int r0, int nrows, int n, int per_rt, const float* s_prod,
                                                 const int* s_rp, const float* s_y, float alpha, float beta, float* y,
                                                 float* s_sv, int* s_sf, unsigned fr) {
    const int per = PER > 0 ? PER : per_rt;
    const int a = threadIdx.x * per;
    const int e = min(a + per, n);
    float s = 0.f, first_part = 0.f;
    int flag = 0, first_row = 0;
    bool first_ends = false;
    if (threadIdx.x == 0) {  // rows with no products before the first product
        for (int r = 0; r < nrows && s_rp[r + 1] == 0; ++r) emit_g(y, s_y, r0, r, 0.f, alpha, beta);
    }
    if (a < n) {
        int r = static_cast<int>(fr >> 1);  // the (non-empty) row holding position a
        bool carry_row = fr & 1u;
        first_row = r;
        int next = s_rp[r + 1];
        if (PER > 0 && a + PER <= n) {
#pragma unroll
            for (int j = 0; j < (PER > 0 ? PER : 1); ++j) {
                const int k = a + j;
                while (next == k) {
                    if (carry_row) { first_part = s; first_ends = true; carry_row = false; }
                    else emit_g(y, s_y, r0, r, s, alpha, beta);
                    s = 0.f;
                    ++r;
                    next = s_rp[r + 1];
                }
                s += s_prod[sk(k)];
            }
        } else {
            for (int k = a; k < e; ++k) {
                while (next == k) {
                    if (carry_row) { first_part = s; first_ends = true; carry_row = false; }
                    else emit_g(y, s_y, r0, r, s, alpha, beta);
                    s = 0.f;
                    ++r;
                    next = s_rp[r + 1];
                }
                s += s_prod[sk(k)];
            }
        }
        // rows ending exactly at this thread's boundary, and empty rows there
        while (r < nrows && next == e) {
            if (carry_row) { first_part = s; first_ends = true; carry_row = false; }
            else emit_g(y, s_y, r0, r, s, alpha, beta);
            s = 0.f;
            ++r;
            next = r < nrows ? s_rp[r + 1] : -1;
        }
        flag = carry_row ? 0 : 1;  // the trailing partial starts inside this thread
    }
    // inclusive segmented scan of (flag, s): (f1,v1) + (f2,v2) = (f1|f2, f2 ? v2 : v1 + v2)
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
    float wp = 0.f;
    for (int i = 0; i < warp; ++i) wp = s_sf[i] ? s_sv[i] : wp + s_sv[i];
    float ex = __shfl_up_sync(kFull, v, 1);
    int exf = __shfl_up_sync(kFull, f, 1);
    if (lane == 0) {
        ex = 0.f;
        exf = 0;
    }
    if (first_ends) emit_g(y, s_y, r0, first_row, (exf ? ex : wp + ex) + first_part, alpha, beta);
}

template <int NT, int ITEMS>
__global__ void __launch_bounds__(NT) spmv_tasks_kernel(const int4* __restrict__ tasks,
                                                              const int* __restrict__ rp, const int* __restrict__ col,
                                                              const float* __restrict__ val,
                                                              const float* __restrict__ x, float alpha, float beta,
                                                              float* y, float* __restrict__ partials, int block_nnz,
                                                              int block_rows, int K,
                                                              const uint16_t* __restrict__ first, int first_group) {
    extern __shared__ __align__(16) float smem[];
    let_dependents_start();
    // segmented groups (the last tasks): this thread's first row, read with the task
    const unsigned fr = (first && static_cast<int>(blockIdx.x) >= first_group)
                            ? __ldcs(first + static_cast<long long>(blockIdx.x - first_group) * NT + threadIdx.x)
                            : 0u;
    const int4 t = tasks[blockIdx.x];
    const int kind = t.x & 3;
    if (kind == kTaskGroup) {
        float* s_prod = smem;
        int* s_rp = reinterpret_cast<int*>(smem + block_nnz + block_nnz / 32 + 1);
        float* s_sv = reinterpret_cast<float*>(s_rp + block_rows + 1);
        int* s_sf = reinterpret_cast<int*>(s_sv + (NT / 32));
        float* s_y = reinterpret_cast<float*>(s_sf + (NT / 32));
        const int code = (t.x >> 2) & 63, nrows = t.x >> 8, r0 = t.y, p0 = t.z, n = t.w - t.z;
        for (int i = threadIdx.x; i <= nrows; i += NT) {
            s_rp[i] = __ldg(rp + r0 + i) - p0;
            if (beta != 0.f && i < nrows) s_y[i] = y[r0 + i];
        }
        stage_products<NT, ITEMS>(p0, n, col, val, x, K, s_prod);
        __syncthreads();
        if (SPX_CHECKED) {
            // the row offsets of this group, read from the caller's row_ptr, must fit the plan's range
            // [p0, p1) and rise; otherwise the rows are not reduced (no shared read outside the products)
            bool bad = false;
            for (int i = threadIdx.x; i <= nrows; i += NT)
                bad |= s_rp[i] < 0 || s_rp[i] > n || (i < nrows && s_rp[i + 1] < s_rp[i]) ||
                       (i == 0 && s_rp[0] != 0) || (i == nrows && s_rp[nrows] != n);
            if (code == kReduceSegmented) {
                // the plan's first row of this thread must hold its first product
                const int a = threadIdx.x * ((block_nnz + NT - 1) / NT), r = static_cast<int>(fr >> 1);
                if (!first) bad = true;
                else if (a < n && !bad)
                    bad = r >= nrows || s_rp[r] > a || s_rp[r + 1] <= a || ((fr & 1u) != 0) != (s_rp[r] < a);
            }
            if (__syncthreads_or(bad)) {
                if (threadIdx.x == 0) check_fail();
                return;
            }
        }
        if (code == kReduceSegmented)
            reduce_segmented<ITEMS>(r0, nrows, n, (block_nnz + NT - 1) / NT, s_prod, s_rp, s_y, alpha,
                                    beta, y, s_sv, s_sf, fr);
        else
            reduce_lanes<NT>(r0, nrows, code, s_prod, s_rp, s_y, alpha, beta, y);
    } else {
        // the old y of a CTA row is read up front, off the critical path
        const float y_old = (kind == kTaskCta && beta != 0.f && threadIdx.x == 0) ? y[t.y] : 0.f;
        predecessor_done();
        float s = range_dot<NT>(t.z, t.w, col, val, x, K);
        s = block_sum<NT>(s, smem);
        if (threadIdx.x == 0) {
            if (kind == kTaskCta) y[t.y] = alpha * s + (beta != 0.f ? beta * y_old : 0.f);
            else partials[t.x >> 8] = s;
        }
    }
}

// One warp per split row: fixed-order sum of its segment partials, then the epilogue.
__global__ void __launch_bounds__(kThreads) spmv_fixup_kernel(const int4* __restrict__ longrows, int nlong,
                                                              const float* __restrict__ partials, float alpha,
                                                              float beta, float* y) {
    const int w = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    predecessor_done();  // the partial sums are the main kernel's output
    if (w >= nlong) return;
    const int4 lr = longrows[w];
    float s = 0.f;
    for (int k = lane; k < lr.z; k += 32) s += partials[lr.y + k];
    s = warp_sum(s);
    if (lane == 0) emit(y, lr.x, s, alpha, beta);
}

// Stream + gather floor of a CSR SpMV: sum of val[p] * x[col[p]] over all
// nonzeros with no row structure at all (grid-stride, 8 gathers in flight per
// thread, one partial sum per CTA).  Measurement aid: the time this takes on a
// matrix is the floor for any SpMV kernel that reads each value and column
// once and gathers x once per nonzero.
__global__ void __launch_bounds__(kThreads) gather_probe_kernel(const int* __restrict__ col,
                                                                const float* __restrict__ val,
                                                                const float* __restrict__ x, long long n,
                                                                float* __restrict__ partials) {
    constexpr int U = 8;
    const long long stride = static_cast<long long>(gridDim.x) * kThreads;
    long long p = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x;
    float s = 0.f;
    for (; p + (U - 1) * stride < n; p += U * stride) {
        int c[U];
        float v[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            c[j] = ld_stream(col + p + j * stride);
            v[j] = ld_stream(val + p + j * stride);
        }
#pragma unroll
        for (int j = 0; j < U; ++j) s += v[j] * ld_x(x + c[j]);
    }
    for (; p < n; p += stride) s += ld_stream(val + p) * ld_x(x + ld_stream(col + p));
    __shared__ float red[kWarps];
    s = block_sum<kThreads>(s, red);
    if (threadIdx.x == 0) partials[blockIdx.x] = s;
}

// A launch of `kernel` on st; with pdl, one that may start while the kernel
// before it on st is still running (programmatic stream serialization): the
// kernel waits for it with predecessor_done() before reading its output.
template <typename... P, typename... A>
cudaError_t launch(void (*kernel)(P...), unsigned grid, unsigned block, size_t smem, cudaStream_t st, bool pdl,
                   A... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<P>(args)...);
}

template <int NT, int ITEMS>
cudaError_t launch_tasks(int ntasks, size_t smem, cudaStream_t st, bool pdl, const int4* tasks, const int* rp,
                         const int* col, const float* val, const float* x, float alpha, float beta, float* y,
                         float* scratch, int B, int R, int K, const uint16_t* first, int first_group) {
    spx_carve::fit(spmv_tasks_kernel<NT, ITEMS>, NT, smem);
    return launch(spmv_tasks_kernel<NT, ITEMS>, ntasks, NT, smem, st, pdl, tasks, rp, col, val, x, alpha, beta, y,
                  scratch, B, R, K, first, first_group);
}

// The SpMV of one plan: the task kernel, then (split rows) the fix-up.  pdl:
// the task kernel may start while the previous kernel on st runs (its matrix
// loads overlap that kernel's last CTAs; it reads x only once that kernel is
// done) -- the second product of the operator pair, whose x is the first's y.
// The fix-up always starts that way behind the task kernel.
spx_status launch_spmv(const spx_plan* P, const int* rp, const int* col, const float* val, float alpha,
                       const float* x, float beta, float* y, float* scratch, cudaStream_t st, bool pdl = false) {
    const int ntasks = static_cast<int>(P->counts[0]);
    const int nlong = static_cast<int>(P->counts[1]);
    if (ntasks == 0) return SPX_OK;
    const int4* tasks = static_cast<const int4*>(P->d_table);
    const int4* longrows = tasks + ntasks;
    const int B = P->opts.block_nnz, R = P->opts.block_rows, K = static_cast<int>(P->K);
    // Eight products per thread: block_nnz 512 / 1024 / 2048 / 4096 runs 64 /
    // 128 / 256 / 512-thread CTAs (smaller CTAs, more of them resident: measured
    // better on skewed rows); other sizes take the runtime-loop form with 256
    // threads.
    const int NT = spx_group_threads(B);
    // the groups are the last tasks; their threads' first rows follow the split-row table
    const int ngroups = static_cast<int>(P->counts[6] + P->counts[7] + P->counts[8]);
    const int first_group = ntasks - ngroups;
    const uint16_t* first =
        P->first.empty() ? nullptr : reinterpret_cast<const uint16_t*>(longrows + nlong);
    const size_t smem = sizeof(float) * static_cast<size_t>(B + B / 32 + 1) +
                        sizeof(int) * (static_cast<size_t>(R) + 1) + 2 * (NT / 32) * sizeof(float) +
                        sizeof(float) * static_cast<size_t>(R);
    cudaError_t e = cudaSuccess;
    switch (B) {
        case 512: e = launch_tasks<64, 8>(ntasks, smem, st, pdl, tasks, rp, col, val, x, alpha, beta, y, scratch, B, R, K, first, first_group); break;
        case 1024: e = launch_tasks<128, 8>(ntasks, smem, st, pdl, tasks, rp, col, val, x, alpha, beta, y, scratch, B, R, K, first, first_group); break;
        case 2048: e = launch_tasks<256, 8>(ntasks, smem, st, pdl, tasks, rp, col, val, x, alpha, beta, y, scratch, B, R, K, first, first_group); break;
        case 4096: e = launch_tasks<512, 8>(ntasks, smem, st, pdl, tasks, rp, col, val, x, alpha, beta, y, scratch, B, R, K, first, first_group); break;
        default: e = launch_tasks<256, 0>(ntasks, smem, st, pdl, tasks, rp, col, val, x, alpha, beta, y, scratch, B, R, K, first, first_group); break;
    }
    uint64_t launches = 1;
    if (e == cudaSuccess && nlong > 0) {
        e = launch(spmv_fixup_kernel, (nlong + kWarps - 1) / kWarps, kThreads, 0, st, true, longrows, nlong, scratch,
                   alpha, beta, y);
        ++launches;
    }
    spx_note_launches(launches);
    return spx_cuda_status(e != cudaSuccess ? e : cudaGetLastError());
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

int spx_spmv_check_take() { return spx_check_take(g_spmv_check); }

extern "C" {

int32_t spx_gather_probe_blocks(void) {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return 8 * nsm;
}

spx_status spx_gather_probe(int64_t nnz, const int32_t* col, const float* val, const float* x, int32_t K,
                            float* partials, int32_t nblocks, spx_stream_t stream) {
    if (nnz < 0 || K < 0 || nblocks < 1 || !partials || (nnz > 0 && (!col || !val || !x))) return SPX_ERR_ARG;
    if (nnz > 0) {
        gather_probe_kernel<<<nblocks, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(col, val, x, nnz,
                                                                                            partials);
        spx_note_launches(1);
    }
    return spx_cuda_status(cudaGetLastError());
}


spx_status spx_spmv_csr(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr,
                        const int32_t* col, const float* val, float alpha, const float* x, float beta, float* y,
                        void* scratch, size_t scratch_bytes, spx_stream_t stream) {
    spx_status s = check_call(plan, M, K, nnz, row_ptr, col, val, x, y, scratch, scratch_bytes);
    if (s != SPX_OK || M == 0) return s;
    return launch_spmv(plan, row_ptr, col, val, alpha, x, beta, y, static_cast<float*>(scratch),
                       reinterpret_cast<cudaStream_t>(stream));
}

size_t spx_spmv_csr_hostio_work_bytes(int32_t M, int32_t K) {
    if (M < 0 || K < 0) return 0;
    const size_t xb = (4 * static_cast<size_t>(K) + 255) & ~static_cast<size_t>(255);
    const size_t yb = (4 * static_cast<size_t>(M) + 255) & ~static_cast<size_t>(255);
    return 2 * (xb + yb);
}

spx_status spx_spmv_csr_hostio(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr,
                               const int32_t* col, const float* val, float alpha, const float* x_host,
                               int64_t x_stride, float beta, float* y_host, int64_t y_stride, int32_t nbatch,
                               void* work, size_t work_bytes, void* scratch, size_t scratch_bytes,
                               spx_stream_t stream) {
    if (!spx_plan_ok(plan) || nbatch < 0 || (x_stride != 0 && x_stride < K) || y_stride < M) return SPX_ERR_ARG;
    if (nbatch == 0 || M == 0) return SPX_OK;
    if (!x_host || !y_host || !work || work_bytes < spx_spmv_csr_hostio_work_bytes(M, K)) return SPX_ERR_ARG;
    if (!spx_aligned(work, 256)) return SPX_ERR_ALIGN;
    const size_t xb = (4 * static_cast<size_t>(K) + 255) & ~static_cast<size_t>(255);
    const size_t yb = (4 * static_cast<size_t>(M) + 255) & ~static_cast<size_t>(255);
    float* xs[2] = {static_cast<float*>(work), reinterpret_cast<float*>(static_cast<char*>(work) + xb + yb)};
    float* ys[2] = {reinterpret_cast<float*>(static_cast<char*>(work) + xb),
                    reinterpret_cast<float*>(static_cast<char*>(work) + 2 * xb + yb)};
    spx_status s = check_call(plan, M, K, nnz, row_ptr, col, val, xs[0], ys[0], scratch, scratch_bytes);
    if (s != SPX_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // Two copy streams and the caller's stream: batch b's inputs go up while
    // batch b-1 computes and batch b-2's result comes down (two device slots).
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t ev[8] = {};  // start, up_done[2], k_done[2], down_done[2], end
    cudaError_t e = cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&down, cudaStreamNonBlocking);
    for (int i = 0; i < 8 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    cudaEvent_t& start = ev[0];
    cudaEvent_t* up_done = ev + 1;
    cudaEvent_t* k_done = ev + 3;
    cudaEvent_t* down_done = ev + 5;
    cudaEvent_t& end = ev[7];
    if (e == cudaSuccess) e = cudaEventRecord(start, st);  // the copies follow the caller's earlier work
    if (e == cudaSuccess) e = cudaStreamWaitEvent(up, start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(down, start, 0);
    for (int32_t b = 0; b < nbatch && e == cudaSuccess && s == SPX_OK; ++b) {
        const int sl = b & 1;
        const float* xh = x_host + static_cast<int64_t>(b) * x_stride;
        float* yh = y_host + static_cast<int64_t>(b) * y_stride;
        if (b >= 2) e = cudaStreamWaitEvent(up, down_done[sl], 0);  // slot free: batch b-2 is home
        if (e == cudaSuccess) e = cudaMemcpyAsync(xs[sl], xh, 4 * static_cast<size_t>(K), cudaMemcpyHostToDevice, up);
        if (e == cudaSuccess && beta != 0.f)
            e = cudaMemcpyAsync(ys[sl], yh, 4 * static_cast<size_t>(M), cudaMemcpyHostToDevice, up);
        if (e == cudaSuccess) e = cudaEventRecord(up_done[sl], up);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, up_done[sl], 0);
        if (e == cudaSuccess) s = launch_spmv(plan, row_ptr, col, val, alpha, xs[sl], beta, ys[sl],
                                              static_cast<float*>(scratch), st);
        if (e == cudaSuccess && s == SPX_OK) e = cudaEventRecord(k_done[sl], st);
        if (e == cudaSuccess && s == SPX_OK) e = cudaStreamWaitEvent(down, k_done[sl], 0);
        if (e == cudaSuccess && s == SPX_OK)
            e = cudaMemcpyAsync(yh, ys[sl], 4 * static_cast<size_t>(M), cudaMemcpyDeviceToHost, down);
        if (e == cudaSuccess && s == SPX_OK) e = cudaEventRecord(down_done[sl], down);
    }
    // the caller's stream resumes once every result is home
    if (e == cudaSuccess) e = cudaEventRecord(end, down);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, end, 0);
    for (int i = 0; i < 8; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);
    if (up) cudaStreamDestroy(up);
    if (down) cudaStreamDestroy(down);
    if (s != SPX_OK) return s;
    return e == cudaSuccess ? SPX_OK : SPX_ERR_CUDA;
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
    if (s == SPX_OK && n > 0)  // starts while the first product finishes; gathers u once it is done
        s = launch_spmv(pAt, At_rp, At_col, At_val, alpha_v, u, beta_v, v, static_cast<float*>(scratch), st, m > 0);
    return s;
}

}  // extern "C"

// ---------------------------------------------------------------- no-alloc variant
// Partial sums of split rows for spx_spmv_csr_noalloc, for callers that cannot
// allocate device memory.  One copy per device, alive until the process exits;
// every call on a device shares it (see include/spx.h).
namespace {
static __device__ __align__(256) float g_noalloc_partials[SPX_NOALLOC_MAX_SLOTS];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the array on the current device, with that device
// current (host code must not use the symbol itself).  Looked up again on
// every call made outside stream capture -- a cheap host call -- so a device
// reset by the caller between calls cannot leave a stale address behind; a
// call on a capturing stream reuses the address of the last call outside
// capture, and the first call on a device must come before any capture.
spx_status noalloc_partials(cudaStream_t st, float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPX_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SPX_ERR_UNSUPPORTED;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const bool capturing = cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone;
    if (capturing) cudaGetLastError();  // a refused query leaves no sticky error behind
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!capturing) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || !p) return SPX_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    if (!g_noalloc_ptr[dev]) return SPX_ERR_NOT_READY;
    *out = g_noalloc_ptr[dev];
    return SPX_OK;
}
}  // namespace

extern "C" spx_status spx_spmv_csr_noalloc(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz,
                                           const int32_t* row_ptr, const int32_t* col, const float* val, float alpha,
                                           const float* x, float beta, float* y, spx_stream_t stream) {
    if (!spx_plan_ok(plan)) return SPX_ERR_ARG;
    if (plan->counts[2] > SPX_NOALLOC_MAX_SLOTS) return SPX_ERR_SCRATCH_LIMIT;
    float* partials = nullptr;
    spx_status s = noalloc_partials(reinterpret_cast<cudaStream_t>(stream), &partials);
    if (s != SPX_OK) return s;
    s = check_call(plan, M, K, nnz, row_ptr, col, val, x, y, partials, sizeof(float) * SPX_NOALLOC_MAX_SLOTS);
    if (s != SPX_OK || M == 0) return s;
    return launch_spmv(plan, row_ptr, col, val, alpha, x, beta, y, partials, reinterpret_cast<cudaStream_t>(stream));
}
