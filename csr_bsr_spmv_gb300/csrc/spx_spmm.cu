// spx_spmm.cu -- CSR SpMM C = alpha*A*B + beta*C on sm_103a, B and C dense
// row-major.  [SpMM-ops] §3: for each stored A(i,k), the contiguous run
// B(k, n:n+N_TILE) updates register accumulators; C is written once.
// The variant is chosen by N ([SpMM-ops] §3.1-§3.3):
//   small   N <= 8     : lanes split the row's nonzeros, N accumulators per lane,
//                        warp-shuffle reduction of each column;
//   float4  N%4 == 0 : columns are cut into tiles of T = pow2ceil(N) up to 128
//                        (or the caller's choice, 8..128); a sub-warp of
//                        L = T/4 lanes owns (row, tile), each lane 4 adjacent
//                        columns (float4 loads of B); 32/L rows per warp, so a
//                        4-row cluster shares one warp and its B rows hit in
//                        L1.  The tile index is the outer grid dimension, the
//                        CTA's run of A is staged in shared memory, B loads
//                        carry an L2 evict-last hint and A / C stream through
//                        with evict-first hints;
//   scalar  otherwise  : a warp per row, lanes over columns.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "spx_check.cuh"
#include "spx_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

SPX_CHECK_WORD(g_spmm_check)

// The checked build's tests: a column inside [0, K) (else the term is skipped)
// and a row range inside [lo, hi] (else the row is skipped).
__device__ __forceinline__ bool col_ok(int c, int K) {
    if (!SPX_CHECKED || (c >= 0 && c < K)) return true;
    check_fail();
    return false;
}
__device__ __forceinline__ bool range_ok(long long a, long long b, long long lo, long long hi) {
    if (!SPX_CHECKED || (lo <= a && a <= b && b <= hi)) return true;
    check_fail();
    return false;
}

__device__ __forceinline__ float ld_stream(const float* p) { return __ldcs(p); }
__device__ __forceinline__ int ld_stream(const int* p) { return __ldcs(p); }

// B rows are the reused operand: keep them in L2 ahead of the streamed A and C.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ float4 ld_keep(const float* p, uint64_t pol) {
    float4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

// ------------------------------------------------------------- small N
template <int N>
__global__ void __launch_bounds__(kThreads) spmm_small_kernel(int M, const int* __restrict__ rp,
                                                              const int* __restrict__ col,
                                                              const float* __restrict__ val,
                                                              const float* __restrict__ B, long long ldb,
                                                              float alpha, float beta, float* C, long long ldc, int K,
                                                              long long nnz) {
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= M) return;
    float acc[N];
#pragma unroll
    for (int c = 0; c < N; ++c) acc[c] = 0.f;
    const int a = __ldg(rp + row), b = __ldg(rp + row + 1);
    if (!range_ok(a, b, 0, nnz)) return;
    for (int p = a + lane; p < b; p += 32) {
        const float v = ld_stream(val + p);
        const int cp = ld_stream(col + p);
        if (!col_ok(cp, K)) continue;
        const float* brow = B + (long long)cp * ldb;
#pragma unroll
        for (int c = 0; c < N; ++c) acc[c] += v * __ldg(brow + c);
    }
#pragma unroll
    for (int c = 0; c < N; ++c)
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) acc[c] += __shfl_down_sync(0xffffffffu, acc[c], d);
    if (lane == 0) {
        float* crow = C + (long long)row * ldc;
#pragma unroll
        for (int c = 0; c < N; ++c) {
            float r = alpha * acc[c];
            if (beta != 0.f) r += beta * crow[c];
            crow[c] = r;
        }
    }
}

// ------------------------------------------------------------- float4 sub-warp / tiled
// L lanes per row, each lane 4 columns; the warp holds 32/L rows.  Column
// tile origin = blockIdx.y * 4 * L (gridDim.y tiles).  One template serves
// fp32 storage and 16-bit storage (A's values and B as bf16 or fp16, widened
// exactly to fp32: [SpMM-ops] §5 keeps storage and accumulation precision
// apart; halving B halves the gathered bytes, the term that dominates SpMM).
//
// The CTA's rows are consecutive, so their nonzeros are one contiguous run of
// col/val.  Up to kStageCap of them are first copied into shared memory with
// coalesced loads by the whole CTA; the row loops then wait only on B rows,
// not on a dependent col -> B chain through DRAM for every batch of U
// nonzeros.  A CTA whose run is longer reads col/val from global memory.
constexpr int kStageCap = 2048;
#ifndef SPX_SPMM_UNROLL
#define SPX_SPMM_UNROLL 8
#endif

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint16_t ld_stream(const uint16_t* p) {
    return static_cast<uint16_t>(__ldcs(reinterpret_cast<const unsigned short*>(p)));
}

// kMinBlocks: resident CTAs per SM the register budget is sized for.  Measured
// on the clustered 1M x 1M matrix at N = 32 and 128: fp32 runs fastest at 6
// (42 registers: 8 B rows of 16 bytes in flight per lane), bf16 at 8 (32).
struct StoreF32 {
    using V = float;
    using Bt = float;
    static constexpr int kMinBlocks = 6;
    static constexpr bool kBatchTail = true;  // the last partial batch of a row loads in parallel
    __device__ static float widen(float v) { return v; }
    __device__ static float4 brow(const float* p, uint64_t pol) { return ld_keep(p, pol); }
};
struct StoreBF16 {
    using V = uint16_t;
    using Bt = uint16_t;
    static constexpr int kMinBlocks = 8;
    static constexpr bool kBatchTail = false;  // at 32 registers the batched tail spills
    __device__ static float widen(uint16_t v) { return __uint_as_float(static_cast<uint32_t>(v) << 16); }
    __device__ static float4 brow(const uint16_t* p, uint64_t pol) {  // 4 bf16 = 8 bytes
        uint2 w;
        asm volatile("ld.global.nc.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;" : "=r"(w.x), "=r"(w.y) : "l"(p), "l"(pol));
        return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
    }
};

struct StoreF16 {  // IEEE binary16 values; widened with the hardware conversion (exact)
    using V = uint16_t;
    using Bt = uint16_t;
    static constexpr int kMinBlocks = 8;
    static constexpr bool kBatchTail = false;
    __device__ static float widen(uint16_t v) { return __half2float(__ushort_as_half(v)); }
    __device__ static float4 brow(const uint16_t* p, uint64_t pol) {  // 4 fp16 = 8 bytes
        uint2 w;
        asm volatile("ld.global.nc.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;" : "=r"(w.x), "=r"(w.y) : "l"(p), "l"(pol));
        return make_float4(widen(static_cast<uint16_t>(w.x & 0xffffu)), widen(static_cast<uint16_t>(w.x >> 16)),
                           widen(static_cast<uint16_t>(w.y & 0xffffu)), widen(static_cast<uint16_t>(w.y >> 16)));
    }
};

template <bool SMEM>
__device__ __forceinline__ int ld_a(const int* p) { return SMEM ? *p : ld_stream(p); }
template <bool SMEM, class V>
__device__ __forceinline__ V ld_a(const V* p) { return SMEM ? *p : ld_stream(p); }

// Sum over the nonzeros [a, b) of cols/vals of val * B(col, n0 .. n0+3); U B rows in flight.
template <class T, bool SMEM>
__device__ __forceinline__ float4 row_dot(const int* cols, const typename T::V* vals, int a, int b,
                                          const typename T::Bt* Bc, long long ldb, uint64_t pol, int K) {
    constexpr int U = SPX_SPMM_UNROLL;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int p = a;
    for (; p + U - 1 < b; p += U) {
        int c[U];
        float v[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            c[j] = ld_a<SMEM>(cols + p + j);
            v[j] = T::widen(ld_a<SMEM>(vals + p + j));
        }
        float4 bv[U];
#pragma unroll
        for (int j = 0; j < U; ++j)
            bv[j] = col_ok(c[j], K) ? T::brow(Bc + (long long)c[j] * ldb, pol) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < U; ++j) {
            acc.x += v[j] * bv[j].x; acc.y += v[j] * bv[j].y; acc.z += v[j] * bv[j].z; acc.w += v[j] * bv[j].w;
        }
    }
    if (T::kBatchTail && p < b) {  // the last partial batch, its loads issued together (no serial tail)
        int c[U];
        float v[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            c[j] = p + j < b ? ld_a<SMEM>(cols + p + j) : 0;
            v[j] = p + j < b ? T::widen(ld_a<SMEM>(vals + p + j)) : 0.f;
        }
        float4 bv[U];
#pragma unroll
        for (int j = 0; j < U; ++j)
            bv[j] = p + j < b && col_ok(c[j], K) ? T::brow(Bc + (long long)c[j] * ldb, pol)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < U; ++j) {
            acc.x += v[j] * bv[j].x; acc.y += v[j] * bv[j].y; acc.z += v[j] * bv[j].z; acc.w += v[j] * bv[j].w;
        }
        p = b;
    }
    for (; p < b; ++p) {
        const int c0 = ld_a<SMEM>(cols + p);
        const float v0 = T::widen(ld_a<SMEM>(vals + p));
        const float4 b0 = col_ok(c0, K) ? T::brow(Bc + (long long)c0 * ldb, pol) : make_float4(0.f, 0.f, 0.f, 0.f);
        acc.x += v0 * b0.x; acc.y += v0 * b0.y; acc.z += v0 * b0.z; acc.w += v0 * b0.w;
    }
    return acc;
}

template <int L, class T>
__global__ void __launch_bounds__(kThreads, T::kMinBlocks)
    spmm_vec_kernel(int M, int N, const int* __restrict__ rp, const int* __restrict__ col,
                    const typename T::V* __restrict__ val, const typename T::Bt* __restrict__ B, long long ldb,
                    float alpha, float beta, float* C, long long ldc, int long_min, int K, long long nnz) {
    constexpr int RPW = 32 / L;         // rows per warp
    constexpr int R = kWarps * RPW;     // rows per CTA
    constexpr int IT = kStageCap / kThreads;
    __shared__ int s_col[kStageCap];
    __shared__ typename T::V s_val[kStageCap];
    const int lane = threadIdx.x & 31;
    const int r0 = blockIdx.x * R;
    const int row = r0 + (threadIdx.x >> 5) * RPW + lane / L;
    const int n0 = blockIdx.y * 4 * L + 4 * (lane % L);
    const int ca = __ldg(rp + r0);
    const int cn = __ldg(rp + min(r0 + R, M)) - ca;
    // (checked build: a run outside [0, nnz] is not staged; its rows fail the range test below)
    const bool staged = cn <= kStageCap && (!SPX_CHECKED || (ca >= 0 && cn >= 0 && ca + (long long)cn <= nnz));
    if (staged) {
        int c[IT];
        typename T::V v[IT];
#pragma unroll
        for (int j = 0; j < IT; ++j) {
            const int k = threadIdx.x + j * kThreads;
            if (k < cn) {
                c[j] = ld_stream(col + ca + k);
                v[j] = ld_stream(val + ca + k);
            }
        }
#pragma unroll
        for (int j = 0; j < IT; ++j) {
            const int k = threadIdx.x + j * kThreads;
            if (k < cn) {
                s_col[k] = c[j];
                s_val[k] = v[j];
            }
        }
        __syncthreads();
    }
    if (row >= M || n0 >= N) return;
    const uint64_t pol = l2_evict_last_policy();
    const int a = __ldg(rp + row), b = __ldg(rp + row + 1);
    if (b - a > long_min) return;  // a long row: its CTA task or segments (planned call) produce it
    if (!range_ok(a, b, staged ? ca : 0, staged ? (long long)ca + cn : nnz)) return;
    const typename T::Bt* Bc = B + n0;
    const float4 acc = staged ? row_dot<T, true>(s_col, s_val, a - ca, b - ca, Bc, ldb, pol, K)
                              : row_dot<T, false>(col, val, a, b, Bc, ldb, pol, K);
    float4* cp = reinterpret_cast<float4*>(C + (long long)row * ldc + n0);
    float4 r = make_float4(alpha * acc.x, alpha * acc.y, alpha * acc.z, alpha * acc.w);
    if (beta != 0.f) {
        const float4 o = *cp;
        r.x += beta * o.x; r.y += beta * o.y; r.z += beta * o.z; r.w += beta * o.w;
    }
    __stcs(cp, r);  // C is written once: evict-first
}

// ------------------------------------------------------------- long rows (planned call)
// One CTA per long task of an SpMV plan and per column tile ([SpMM-ops] §2.4:
// split a long row, combine the partial sums in a second pass).  The kT/L
// sub-warps stride the task's nonzeros; their float4 sums are combined in a
// fixed order through shared memory.  A CTA row writes C; a segment of a split
// row writes its partial row to partials[slot][0..N).
template <int L, class T>
__global__ void __launch_bounds__(kThreads) spmm_long_kernel(const int4* __restrict__ tasks, int N,
                                                            const int* __restrict__ col,
                                                            const typename T::V* __restrict__ val,
                                                            const typename T::Bt* __restrict__ B, long long ldb,
                                                            float alpha, float beta, float* C, long long ldc,
                                                            float* __restrict__ partials, int K) {
    constexpr int NSUB = kThreads / L;
    constexpr int U = 4;
    __shared__ float4 red[NSUB][L];
    const int4 t = tasks[blockIdx.x];
    const int kind = t.x & 3, row = t.y, p0 = t.z, p1 = t.w;
    const int q = threadIdx.x / L, l = threadIdx.x % L;
    const int n0 = blockIdx.y * 4 * L + 4 * l;
    const uint64_t pol = l2_evict_last_policy();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (n0 < N) {
        const typename T::Bt* Bc = B + n0;
        int p = p0 + q;
        for (; p + (U - 1) * NSUB < p1; p += U * NSUB) {
            int c[U];
            float v[U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                c[j] = ld_stream(col + p + j * NSUB);
                v[j] = T::widen(ld_stream(val + p + j * NSUB));
            }
            float4 bv[U];
#pragma unroll
            for (int j = 0; j < U; ++j)
                bv[j] = col_ok(c[j], K) ? T::brow(Bc + (long long)c[j] * ldb, pol) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < U; ++j) {
                acc.x += v[j] * bv[j].x; acc.y += v[j] * bv[j].y; acc.z += v[j] * bv[j].z; acc.w += v[j] * bv[j].w;
            }
        }
        for (; p < p1; p += NSUB) {
            const float v0 = T::widen(ld_stream(val + p));
            const int c0 = ld_stream(col + p);
            const float4 b0 = col_ok(c0, K) ? T::brow(Bc + (long long)c0 * ldb, pol) : make_float4(0.f, 0.f, 0.f, 0.f);
            acc.x += v0 * b0.x; acc.y += v0 * b0.y; acc.z += v0 * b0.z; acc.w += v0 * b0.w;
        }
    }
    red[q][l] = acc;
    __syncthreads();
    if (threadIdx.x >= 4 * L) return;
    // thread c sums column c of the tile over the sub-warps, in sub-warp order
    const int c = threadIdx.x, n = blockIdx.y * 4 * L + c;
    if (n >= N) return;
    const float* rf = reinterpret_cast<const float*>(&red[0][0]);
    float s = 0.f;
    for (int k = 0; k < NSUB; ++k) s += rf[k * 4 * L + c];
    if (kind == 1) {  // a CTA row: the whole row is here
        float* cp = C + (long long)row * ldc + n;
        *cp = beta != 0.f ? alpha * s + beta * *cp : alpha * s;
    } else {  // a segment: its partial row
        partials[(long long)(t.x >> 8) * N + n] = s;
    }
}

// One thread per (split row, column): the row's segment partials in segment order, then alpha/beta.
__global__ void __launch_bounds__(kThreads) spmm_long_fixup_kernel(const int4* __restrict__ longrows, int nlong,
                                                                  int N, const float* __restrict__ partials,
                                                                  float alpha, float beta, float* C, long long ldc) {
    for (int r = blockIdx.y; r < nlong; r += gridDim.y) {
        const int4 lr = longrows[r];
        for (int n = blockIdx.x * kThreads + threadIdx.x; n < N; n += gridDim.x * kThreads) {
            float s = 0.f;
            for (int k = 0; k < lr.z; ++k) s += partials[(long long)(lr.y + k) * N + n];
            float* cp = C + (long long)lr.x * ldc + n;
            *cp = beta != 0.f ? alpha * s + beta * *cp : alpha * s;
        }
    }
}

// ------------------------------------------------------------- scalar fallback
__global__ void __launch_bounds__(kThreads) spmm_scalar_kernel(int M, int N, const int* __restrict__ rp,
                                                               const int* __restrict__ col,
                                                               const float* __restrict__ val,
                                                               const float* __restrict__ B, long long ldb,
                                                               float alpha, float beta, float* C, long long ldc, int K,
                                                               long long nnz) {
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= M) return;
    const int a = __ldg(rp + row), b = __ldg(rp + row + 1);
    if (!range_ok(a, b, 0, nnz)) return;
    for (int n = blockIdx.y * 32 + lane; n < N; n += 32 * gridDim.y) {
        float acc = 0.f;
        for (int p = a; p < b; ++p) {
            const int c = __ldg(col + p);
            if (col_ok(c, K)) acc += __ldg(val + p) * __ldg(B + (long long)c * ldb + n);
        }
        float r = alpha * acc;
        float* cp = C + (long long)row * ldc + n;
        if (beta != 0.f) r += beta * *cp;
        *cp = r;
    }
}

int pick_variant(int32_t N, const float* B, int64_t ldb, const float* C, int64_t ldc) {
    if (N <= 8) return 0;
    const bool vec = (N % 4 == 0) && (ldb % 4 == 0) && (ldc % 4 == 0) && spx_aligned(B, 16) && spx_aligned(C, 16);
    if (!vec) return 3;
    return N <= 128 ? 1 : 2;
}

// Column tile of the float4 variants: the whole of N up to 128 columns (a
// sub-warp of N/4 lanes per row), tiles of 128 beyond.  Narrower tiles keep
// less of B per pass but were slower on GB300 (1M x 1M clustered matrix,
// N = 128: 1.11 ms at 128 columns, 1.18 / 1.29 / 1.93 ms at 64 / 32 / 16):
// every tile re-streams the matrix, and below 32 fp32 columns a B-row
// fragment is smaller than the 128-byte lines L2 fills from DRAM, so DRAM
// traffic grows (5.1 GB at 128 columns, 10.6 GB at 16).  They are only taken
// on request.
int auto_col_tile(int32_t N) {
    int t = 8;
    while (t < N && t < 128) t <<= 1;
    return t;
}

// Long-row work of a planned call: the plan's CTA-row and segment tasks (the
// first nlong_tasks entries of its device table), then the split-row fix-up.
struct LongWork {
    int K = 0;          // columns of A (the checked build tests every column against it)
    long long nnz = 0;  // entries of A (and every row range against it)
    const int4* tasks = nullptr;
    int ntasks = 0;
    const int4* longrows = nullptr;
    int nlongrows = 0;
    float* partials = nullptr;
    int long_min = 0x7fffffff;  // rows longer than this are long (skipped by the row kernel)
};

template <int L, class T>
void launch_vec(int M, int N, const int* rp, const int* col, const typename T::V* val, const typename T::Bt* B,
                long long ldb, float alpha, float beta, float* C, long long ldc, cudaStream_t st,
                const LongWork& lw) {
    constexpr int rows_per_cta = kWarps * (32 / L);
    const int tiles = (N + 4 * L - 1) / (4 * L);
    dim3 grid((M + rows_per_cta - 1) / rows_per_cta, tiles);
    spmm_vec_kernel<L, T><<<grid, kThreads, 0, st>>>(M, N, rp, col, val, B, ldb, alpha, beta, C, ldc, lw.long_min, lw.K,
                                                    lw.nnz);
    if (lw.ntasks > 0)
        spmm_long_kernel<L, T><<<dim3(lw.ntasks, tiles), kThreads, 0, st>>>(lw.tasks, N, col, val, B, ldb, alpha,
                                                                             beta, C, ldc, lw.partials, lw.K);
    if (lw.nlongrows > 0)
        spmm_long_fixup_kernel<<<dim3((N + kThreads - 1) / kThreads, lw.nlongrows < 65535 ? lw.nlongrows : 65535),
                                 kThreads, 0, st>>>(lw.longrows, lw.nlongrows, N, lw.partials, alpha, beta, C, ldc);
}

template <class T>
void launch_vec_tile(int tile, int M, int N, const int* rp, const int* col, const typename T::V* val,
                     const typename T::Bt* B, long long ldb, float alpha, float beta, float* C, long long ldc,
                     cudaStream_t st, const LongWork& lw) {
    switch (tile) {
        case 8: launch_vec<2, T>(M, N, rp, col, val, B, ldb, alpha, beta, C, ldc, st, lw); break;
        case 16: launch_vec<4, T>(M, N, rp, col, val, B, ldb, alpha, beta, C, ldc, st, lw); break;
        case 32: launch_vec<8, T>(M, N, rp, col, val, B, ldb, alpha, beta, C, ldc, st, lw); break;
        case 64: launch_vec<16, T>(M, N, rp, col, val, B, ldb, alpha, beta, C, ldc, st, lw); break;
        default: launch_vec<32, T>(M, N, rp, col, val, B, ldb, alpha, beta, C, ldc, st, lw); break;
    }
}

// 16-bit A values and B (bf16 or fp16 bit patterns), fp32 products and sums, fp32 C.
template <class T>
spx_status spmm_16bit(int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col, const uint16_t* val,
                      int32_t N, const uint16_t* B, int64_t ldb, float alpha, float beta, float* C, int64_t ldc,
                      cudaStream_t st) {
    if (M < 0 || K < 0 || nnz < 0 || N < 0) return SPX_ERR_ARG;
    if (nnz > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (M == 0 || N == 0) return SPX_OK;
    if (!rp || !C || (nnz > 0 && (!col || !val || !B))) return SPX_ERR_ARG;
    if (ldb < N || ldc < N) return SPX_ERR_ARG;
    if (N % 4 || ldb % 4 || ldc % 4) return SPX_ERR_UNSUPPORTED;
    if (!spx_aligned(rp, 4) || !spx_aligned(col, 4) || !spx_aligned(val, 2) || !spx_aligned(B, 8) ||
        !spx_aligned(C, 16))
        return SPX_ERR_ALIGN;
    LongWork lw;
    lw.K = K;
    lw.nnz = nnz;
    launch_vec_tile<T>(auto_col_tile(N), M, N, rp, col, val, B, ldb, alpha, beta, C, ldc, st, lw);
    spx_note_launches(1);
    return spx_cuda_status(cudaGetLastError());
}

// A planned call: the plan's long rows (CTA rows and split rows, as for the
// SpMV) get whole CTAs and segment partials; the other rows run as usual.
template <class T>
spx_status spmm_planned(const spx_plan* P, int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col,
                        const typename T::V* val, int32_t N, const typename T::Bt* B, int64_t ldb, float alpha,
                        float beta, float* C, int64_t ldc, void* scratch, size_t scratch_bytes, cudaStream_t st) {
    if (!spx_plan_ok(P) || M < 0 || K < 0 || nnz < 0 || N < 0) return SPX_ERR_ARG;
    if (P->M != M || P->K != K || P->nnz != nnz) return SPX_ERR_ARG;
    if (M == 0 || N == 0) return SPX_OK;
    if (P->table_bytes > 0 && !P->d_table) return SPX_ERR_NOT_READY;
    if (!rp || !C || (nnz > 0 && (!col || !val || !B))) return SPX_ERR_ARG;
    if (ldb < N || ldc < N) return SPX_ERR_ARG;
    if (N % 4 || ldb % 4 || ldc % 4) return SPX_ERR_UNSUPPORTED;
    if (!spx_aligned(rp, 4) || !spx_aligned(col, 4) || !spx_aligned(val, sizeof(typename T::V)) ||
        !spx_aligned(B, 4 * sizeof(typename T::Bt)) || !spx_aligned(C, 16) || !spx_aligned(scratch, 4))
        return SPX_ERR_ALIGN;
    const int64_t slots = P->counts[2];
    const size_t need = sizeof(float) * static_cast<size_t>(slots) * static_cast<size_t>(N);
    if (need && (!scratch || scratch_bytes < need)) return SPX_ERR_ARG;
    LongWork lw;
    lw.K = K;
    lw.nnz = nnz;
    const int64_t ngroups = P->counts[6] + P->counts[7] + P->counts[8];
    lw.tasks = static_cast<const int4*>(P->d_table);
    lw.ntasks = static_cast<int>(P->counts[0] - ngroups);  // long-row tasks come first in the table
    lw.longrows = lw.tasks + P->counts[0];
    lw.nlongrows = static_cast<int>(P->counts[1]);
    lw.partials = static_cast<float*>(scratch);
    lw.long_min = P->opts.pack_max;
    launch_vec_tile<T>(auto_col_tile(N), M, N, rp, col, val, B, ldb, alpha, beta, C, ldc, st, lw);
    spx_note_launches(1 + (lw.ntasks > 0) + (lw.nlongrows > 0));
    return spx_cuda_status(cudaGetLastError());
}

spx_status spmm_impl(int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col, const float* val,
                     int32_t N, const float* B, int64_t ldb, float alpha, float beta, float* C, int64_t ldc,
                     int32_t col_tile, cudaStream_t st) {
    if (M < 0 || K < 0 || nnz < 0 || N < 0 || col_tile < 0) return SPX_ERR_ARG;
    if (nnz > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (M == 0 || N == 0) return SPX_OK;
    if (!rp || !C || (nnz > 0 && (!col || !val || !B))) return SPX_ERR_ARG;
    if (ldb < N || ldc < N) return SPX_ERR_ARG;
    if (col_tile && (col_tile < 8 || col_tile > 128 || (col_tile & (col_tile - 1)))) return SPX_ERR_ARG;
    if (!spx_aligned(rp, 4) || !spx_aligned(col, 4) || !spx_aligned(val, 4) || !spx_aligned(B, 4) ||
        !spx_aligned(C, 4))
        return SPX_ERR_ALIGN;
    const int v = pick_variant(N, B, ldb, C, ldc);
    if (v == 0) {
        const int grid = (M + kWarps - 1) / kWarps;
        switch (N) {
#define SPX_SMALL(n) case n: spmm_small_kernel<n><<<grid, kThreads, 0, st>>>(M, rp, col, val, B, ldb, alpha, beta, C, ldc, K, nnz); break;
            SPX_SMALL(1) SPX_SMALL(2) SPX_SMALL(3) SPX_SMALL(4) SPX_SMALL(5) SPX_SMALL(6) SPX_SMALL(7) SPX_SMALL(8)
#undef SPX_SMALL
        }
    } else if (v == 3) {
        dim3 grid((M + kWarps - 1) / kWarps, (N + 31) / 32 < 4 ? (N + 31) / 32 : 4);
        spmm_scalar_kernel<<<grid, kThreads, 0, st>>>(M, N, rp, col, val, B, ldb, alpha, beta, C, ldc, K, nnz);
    } else {
        const int t = col_tile ? col_tile : auto_col_tile(N);
        LongWork lw;
        lw.K = K;
        lw.nnz = nnz;
        launch_vec_tile<StoreF32>(t, M, N, rp, col, val, B, ldb, alpha, beta, C, ldc, st, lw);
    }
    spx_note_launches(1);
    return spx_cuda_status(cudaGetLastError());
}

}  // namespace

int spx_spmm_check_take() { return spx_check_take(g_spmm_check); }

extern "C" {

int32_t spx_spmm_csr_variant(int32_t N, const float* B, int64_t ldb, const float* C, int64_t ldc) {
    return pick_variant(N, B, ldb, C, ldc);
}

spx_status spx_spmm_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col, const float* val,
                        int32_t N, const float* B, int64_t ldb, float alpha, float beta, float* C, int64_t ldc,
                        spx_stream_t stream) {
    return spmm_impl(M, K, nnz, rp, col, val, N, B, ldb, alpha, beta, C, ldc, 0, reinterpret_cast<cudaStream_t>(stream));
}

spx_status spx_spmm_csr_bf16(int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col,
                             const uint16_t* val, int32_t N, const uint16_t* B, int64_t ldb, float alpha, float beta,
                             float* C, int64_t ldc, spx_stream_t stream) {
    return spmm_16bit<StoreBF16>(M, K, nnz, rp, col, val, N, B, ldb, alpha, beta, C, ldc,
                                 reinterpret_cast<cudaStream_t>(stream));
}

spx_status spx_spmm_csr_f16(int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col,
                            const uint16_t* val, int32_t N, const uint16_t* B, int64_t ldb, float alpha, float beta,
                            float* C, int64_t ldc, spx_stream_t stream) {
    return spmm_16bit<StoreF16>(M, K, nnz, rp, col, val, N, B, ldb, alpha, beta, C, ldc,
                                reinterpret_cast<cudaStream_t>(stream));
}

size_t spx_spmm_csr_planned_scratch_bytes(const spx_plan* plan, int32_t N) {
    if (!spx_plan_ok(plan) || N < 0) return 0;
    return sizeof(float) * static_cast<size_t>(plan->counts[2]) * static_cast<size_t>(N);
}

spx_status spx_spmm_csr_planned(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* rp,
                                const int32_t* col, const float* val, int32_t N, const float* B, int64_t ldb,
                                float alpha, float beta, float* C, int64_t ldc, void* scratch, size_t scratch_bytes,
                                spx_stream_t stream) {
    return spmm_planned<StoreF32>(plan, M, K, nnz, rp, col, val, N, B, ldb, alpha, beta, C, ldc, scratch,
                                  scratch_bytes, reinterpret_cast<cudaStream_t>(stream));
}

spx_status spx_spmm_csr_bf16_planned(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* rp,
                                     const int32_t* col, const uint16_t* val, int32_t N, const uint16_t* B,
                                     int64_t ldb, float alpha, float beta, float* C, int64_t ldc, void* scratch,
                                     size_t scratch_bytes, spx_stream_t stream) {
    return spmm_planned<StoreBF16>(plan, M, K, nnz, rp, col, val, N, B, ldb, alpha, beta, C, ldc, scratch,
                                   scratch_bytes, reinterpret_cast<cudaStream_t>(stream));
}

spx_status spx_spmm_csr_f16_planned(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* rp,
                                    const int32_t* col, const uint16_t* val, int32_t N, const uint16_t* B,
                                    int64_t ldb, float alpha, float beta, float* C, int64_t ldc, void* scratch,
                                    size_t scratch_bytes, spx_stream_t stream) {
    return spmm_planned<StoreF16>(plan, M, K, nnz, rp, col, val, N, B, ldb, alpha, beta, C, ldc, scratch,
                                  scratch_bytes, reinterpret_cast<cudaStream_t>(stream));
}

spx_status spx_spmm_csr_tiled(int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col,
                              const float* val, int32_t N, const float* B, int64_t ldb, float alpha, float beta,
                              float* C, int64_t ldc, int32_t col_tile, spx_stream_t stream) {
    return spmm_impl(M, K, nnz, rp, col, val, N, B, ldb, alpha, beta, C, ldc, col_tile,
                     reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
