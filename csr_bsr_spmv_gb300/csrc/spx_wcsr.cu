// spx_wcsr.cu -- WCSR (window CSR) format and its tensor-core SpMM on sm_103a.
//
// [AsyncSparse] §2.2.2: rows are grouped into windows of fixed height (64
// here); a window stores the union of the columns its rows use
// (window_col_idx, -1 = padding) and, for those compressed columns, a dense
// 64-row block of values -- finer than BSR for scattered nonzeros, at the
// price of an indirect load of B.  Here the compressed columns of a window
// are cut into chunks of 64, and each chunk's values are one 64 x 64 bf16
// block stored row-major (8 KB, the BSR block layout), so a chunk is a
// "BSR block whose B rows are gathered".
//
// Kernel ([AsyncSparse] §4.1: TMA for A, cooperative gather of B rows into a
// 128-byte-swizzled shared tile, tensor-core MMA; mapped to Blackwell): one
// CTA per (128-column tile of N, window), 192 threads:
//   warp 0, lane 0: TMA of the chunk's A block into the ring stage;
//   warp 1, lane 0: tcgen05.mma of the stage into a TMEM accumulator
//                   (transposed: M = 128 output columns, N = 64 window rows,
//                   K = 16), tcgen05.commit frees the stage;
//   warps 2-5     : gather the chunk's 64 B rows (128 columns, 256 bytes each)
//                   with 16-byte cp.async straight into the swizzled B tile
//                   (zero-fill for padding columns), several stages in
//                   flight per thread; then they run the epilogue.
// Each window is one CTA (no split, no atomics): the product is deterministic.
// Every mbarrier wait is bounded; on expiry the CTA records an error word
// (spx_last_device_error), stops, drains its copies, frees TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <type_traits>
#include <new>
#include <vector>

#include "spx_check.cuh"
#include "spx_internal.h"
#include "spx_tc.cuh"

using namespace spx_tc;

namespace {

constexpr int kWin = 64;                       // window height = chunk width
constexpr int kThreads = 192;
constexpr uint32_t kABytes = kWin * kWin * 2;  // 8 KB A block
constexpr uint32_t kBBox = kWin * 64 * 2;      // 64 k-rows x 64 n, 8 KB
constexpr uint32_t kIdesc = idesc_bf16_mn_k(128, 64);
constexpr long long kSpinLimit = 2000000000LL;  // cycles (~1 s)

// A 2-deep ring (four CTAs per SM) measured fastest; deeper rings and
// 256-column tiles were slower.  A stage holds one A chunk and the gathered B
// rows for 128 output columns (HALVES M = 128 halves).
constexpr int STAGES = 2;
constexpr int HALVES = 1;
constexpr uint32_t kStageBytesW = kABytes + 2 * HALVES * kBBox;  // 24 KB
constexpr size_t kSmemW = STAGES * kStageBytesW + 1024 + 256;

enum : int { kErrFull = 1, kErrEmpty = 2, kErrAcc = 3, kErrDrain = 4 };

__device__ int g_wcsr_error;
__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_wcsr_error, 0, code); }

// The checked build's word: a column outside [-1, K) (read as padding in
// either build, reported here) or a window whose chunks leave [0, nchunks)
// (treated as empty here).
SPX_CHECK_WORD(g_wcsr_check)

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <bool TASKS>
__global__ void __launch_bounds__(kThreads)
    wcsr_spmm_kernel(const __grid_constant__ CUtensorMap tmA, const int* __restrict__ win_ptr,
                     const int* __restrict__ win_col, const uint16_t* __restrict__ B, long long ldb,
                     float* __restrict__ C, long long ldc, int M, int K, float alpha, float beta,
                     long long spin_limit, const int4* __restrict__ tasks, float* __restrict__ partials, int N,
                     long long nchunks) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_issued, s_consumed;

    constexpr int kStages = STAGES;
    constexpr uint32_t kStageBytes = kStageBytesW;
    constexpr uint32_t kTmemCols = 64 * HALVES;
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t bars = base + kStages * kStageBytes;
    auto afull = [&](int s) { return bars + 8u * s; };                 // TMA bytes of the A block
    auto gfull = [&](int s) { return bars + 8u * (kStages + s); };     // 128 gather threads
    auto empty = [&](int s) { return bars + 8u * (2 * kStages + s); }; // MMA commit
    const uint32_t acc_bar = bars + 8u * (3 * kStages);
    auto stage_a = [&](int s) { return base + s * kStageBytes; };
    auto stage_b = [&](int s) { return base + s * kStageBytes + kABytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * 128 * HALVES;
    // one window per CTA row of the grid, or (planned call) one task: a piece
    // of a window's chunks {window, first chunk, chunks, partial slot or -1}
    int w, g0, nch, slot = -1;
    if (TASKS) {
        const int4 t = tasks[blockIdx.y];
        w = t.x;
        g0 = t.y;
        nch = t.z;
        slot = t.w;
    } else {
        w = blockIdx.y;
        g0 = __ldg(win_ptr + w);
        nch = __ldg(win_ptr + w + 1) - g0;
    }
    if (SPX_CHECKED && !(g0 >= 0 && nch >= 0 && g0 + static_cast<long long>(nch) <= nchunks)) {
        if (threadIdx.x == 0) check_fail();
        nch = 0;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(afull(s), 1);
            mbar_init(gfull(s), 128);
            mbar_init(empty(s), 1);
        }
        mbar_init(acc_bar, 1);
        s_abort = 0;
        s_issued = 0;
        s_consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = s_tmem;

    if (warp == 0) {
        if (lane == 0) {
            int b = 0;
            for (; b < nch; ++b) {
                const int s = b % kStages;
                if (!mbar_wait(empty(s), ((b / kStages) & 1u) ^ 1u, spin_limit) || s_abort) {
                    record_error(kErrEmpty);
                    s_abort = 1;
                    break;
                }
                mbar_expect_tx(afull(s), kABytes);
                tma_load_2d(stage_a(s), &tmA, 0, (g0 + b) * kWin, afull(s));
            }
            s_issued = b;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int b = 0;
            for (; b < nch; ++b) {
                const int s = b % kStages;
                const uint32_t ph = (b / kStages) & 1u;
                if (!mbar_wait(afull(s), ph, spin_limit) || !mbar_wait(gfull(s), ph, spin_limit)) {
                    record_error(kErrFull);
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kWin / 16; ++ks) {
                    const uint64_t bdesc = sw128_desc(stage_a(s) + ks * 32u, 16u, 1024u);
#pragma unroll
                    for (int hh = 0; hh < HALVES; ++hh) {
                        const uint64_t adesc = sw128_desc(stage_b(s) + 2 * hh * kBBox + ks * 2048u, kBBox, 1024u);
                        mma_bf16(tmem_d + 64 * hh, adesc, bdesc, kIdesc, (b > 0 || ks > 0) ? 1u : 0u);
                    }
                }
                mma_commit(empty(s));
            }
            s_consumed = b;
            if (b > 0) mma_commit(acc_bar);
            else mbar_arrive(acc_bar);
        }
    } else {
        // Gather: per stage 64 B rows x 64 columns per box (128 bytes = 8 pieces
        // of 16 bytes).  Eight consecutive threads copy one row's 128 bytes, so
        // each warp-wide copy covers four whole 128-byte lines.  Thread t copies
        // piece j = t%8 of box h = (t/8)%2 for rows k = 8i + t/16, i = 0..7, into
        // the 128-byte-swizzled tile: row k at k*128, piece j at (j ^ (k & 7)).
        const int t = threadIdx.x - 64;
        const int j = t & 7, h = (t >> 3) & 1, k0 = t >> 4;
        const uint32_t piece_off = h * kBBox + (static_cast<uint32_t>(j ^ (k0 & 7)) << 4);
        // this thread's eight column indices of the next chunk, loaded one chunk ahead so that their
        // latency overlaps the current chunk's wait and copies
        int cnext[8];
        if (nch > 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) cnext[i] = __ldg(win_col + static_cast<long long>(g0) * kWin + 8 * i + k0);
        }
        int b = 0;
        for (; b < nch; ++b) {
            const int s = b % kStages;
            int cur[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) cur[i] = cnext[i];
            if (b + 1 < nch) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    cnext[i] = __ldg(win_col + static_cast<long long>(g0 + b + 1) * kWin + 8 * i + k0);
            }
            int ok = 1;
            if (lane == 0) ok = (mbar_wait(empty(s), ((b / kStages) & 1u) ^ 1u, spin_limit) && !s_abort) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    record_error(kErrEmpty);
                    s_abort = 1;
                }
                break;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = 8 * i + k0;
                const int cr = cur[i];
                if (SPX_CHECKED && (cr < -1 || cr >= K)) check_fail();
                const int c = cr < K ? cr : -1;  // a column outside B is read as padding, never dereferenced
                const uint16_t* row = c >= 0 ? B + static_cast<long long>(c) * ldb : B;
                const uint32_t dst = stage_b(s) + k * 128u + piece_off;
#pragma unroll
                for (int hh = 0; hh < HALVES; ++hh) {
                    // padding, or a piece past column N (a ragged last tile): zero-fill, no read
                    const int cc = n0 + 128 * hh + 64 * h + 8 * j;
                    const bool in = c >= 0 && cc < N;
                    cp_async16(dst + 2 * hh * kBBox, in ? row + cc : B, in ? 16u : 0u);
                }
            }
            cp_async_commit();
            if (b >= kStages - 1) {  // the copies of stage b - (kStages - 1) have landed: publish them
                cp_async_wait<kStages - 1>();
                fence_proxy_async();
                mbar_arrive(gfull((b - (kStages - 1)) % kStages));
            }
        }
        // publish the stages still in flight, oldest first
        cp_async_wait<0>();
        fence_proxy_async();
        for (int q = max(0, b - (kStages - 1)); q < b; ++q) mbar_arrive(gfull(q % kStages));
    }
    __syncwarp();

    if (warp >= 2) {  // epilogue: TMEM lanes 32*(warp%4) .. +31 = output columns n0 + that range
        int ok = 1;
        if (lane == 0) ok = mbar_wait(acc_bar, 0, spin_limit) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok && lane == 0) record_error(kErrAcc);
        tc_fence_after();
        const int q = warp & 3;
        const int rows = min(kWin, M - w * kWin);
#pragma unroll
        for (int hh = 0; hh < HALVES; ++hh) {
            const int cn = n0 + 128 * hh + 32 * q + lane;  // this thread's column; columns >= N are not stored
            const bool cok = cn < N;
            float* cp = C + static_cast<long long>(w) * kWin * ldc + cn;
            // a piece of a split window writes its raw partial tile (1 * sum, exact; the fix-up applies alpha/beta)
            const bool raw = TASKS && slot >= 0;
            float* dst = raw ? partials + static_cast<long long>(slot) * kWin * N + cn : cp;
            const long long dstride = raw ? N : ldc;
            const float ealpha = raw ? 1.f : alpha, ebeta = raw ? 0.f : beta;
            if (nch == 0) {
                if (cok)
                    for (int r = 0; r < rows; ++r) __stcs(cp + r * ldc, beta != 0.f ? beta * cp[r * ldc] : 0.f);
            } else if (ok && !s_abort) {
                // GUARD: the tile reaches past row M or column N (a ragged edge), so each store is
                // checked; whole tiles (CTA-uniform test) take the unchecked copy of the loop
                auto drain = [&](auto guard) {
                    constexpr bool GUARD = decltype(guard)::value;
#pragma unroll
                    for (int c0 = 0; c0 < kWin; c0 += 32) {
                        uint32_t v[32];
                        tmem_ld32(tmem_d + (static_cast<uint32_t>(32 * q) << 16) + 64 * hh + c0, v);
                        float old[32];  // beta != 0: all 32 old values are loaded before any store
                        if (ebeta != 0.f) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                old[j] = (!GUARD || (cok && c0 + j < rows)) ? dst[static_cast<long long>(c0 + j) * dstride] : 0.f;
                        }
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (!GUARD || (cok && c0 + j < rows)) {
                                float* p = dst + static_cast<long long>(c0 + j) * dstride;
                                const float acc = ealpha * __uint_as_float(v[j]);
                                __stcs(p, ebeta != 0.f ? acc + ebeta * old[j] : acc);
                            }
                        }
                    }
                };
                if (rows == kWin && n0 + 128 * (hh + 1) <= N) drain(std::false_type{});
                else drain(std::true_type{});
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0) {  // A blocks issued but never consumed: wait (bounded) until they landed
        for (int b = s_consumed; b < s_issued; ++b)
            if (!mbar_wait(afull(b % kStages), (b / kStages) & 1u, spin_limit)) {
                record_error(kErrDrain);
                break;
            }
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_d), "r"(kTmemCols) : "memory");
}

// Split windows of a planned call: C rows of window w = alpha * (sum of its
// pieces' partial tiles, in piece order) + beta * C.  One thread per (row of
// the window, column): grid (column blocks, 64 rows, split windows).
__global__ void __launch_bounds__(256) wcsr_fixup_kernel(const int4* __restrict__ splits, int nsplit,
                                                        const float* __restrict__ partials, int M, int N, float alpha,
                                                        float beta, float* C, long long ldc) {
    const int n = blockIdx.x * 256 + threadIdx.x, r = blockIdx.y;
    if (n >= N) return;
    for (int i = blockIdx.z; i < nsplit; i += gridDim.z) {
        const int4 sp = splits[i];  // {window, first slot, pieces, 0}
        if (r >= M - sp.x * kWin) continue;
        float s = 0.f;
        for (int k = 0; k < sp.z; ++k) s += __ldcs(partials + (static_cast<long long>(sp.y + k) * kWin + r) * N + n);
        float* q = C + (static_cast<long long>(sp.x) * kWin + r) * ldc + n;
        *q = beta != 0.f ? alpha * s + beta * *q : alpha * s;
    }
}

__global__ void wcsr_scale_kernel(float* C, long long ldc, int M, int N, float beta) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= N) return;
    for (int r = blockIdx.y; r < M; r += gridDim.y) {
        float* q = C + static_cast<long long>(r) * ldc + c;
        *q = beta != 0.f ? beta * *q : 0.f;
    }
}

// ---------------------------------------------------------------- host builder
spx_status build_wcsr_host(int32_t M, int32_t K, const int32_t* rp, const int32_t* col, const char* val, int32_t vb,
                           int32_t* win_ptr, int32_t* win_col, char* win_val, int64_t* nchunks_out, double* fill_out) {
    if (rp[0] != 0) return SPX_ERR_ARG;
    for (int32_t i = 0; i < M; ++i)
        if (rp[i + 1] < rp[i]) return SPX_ERR_NOT_SORTED;
    const int64_t W = (static_cast<int64_t>(M) + kWin - 1) / kWin;
    std::vector<int32_t> pos(static_cast<size_t>(K), -1);  // column -> compressed position in this window
    std::vector<int32_t> cols;
    std::vector<uint8_t> seen;
    int64_t g = 0;
    if (win_ptr) win_ptr[0] = 0;
    for (int64_t w = 0; w < W; ++w) {
        const int64_t r0 = w * kWin, r1 = std::min<int64_t>(r0 + kWin, M);
        cols.clear();
        for (int64_t p = rp[r0]; p < rp[r1]; ++p) {
            if (col[p] < 0 || col[p] >= K) return SPX_ERR_INDEX_RANGE;
            if (pos[col[p]] < 0) {
                pos[col[p]] = 0;
                cols.push_back(col[p]);
            }
        }
        std::sort(cols.begin(), cols.end());
        for (size_t t = 0; t < cols.size(); ++t) pos[cols[t]] = static_cast<int32_t>(t);
        const int64_t nch = (static_cast<int64_t>(cols.size()) + kWin - 1) / kWin;
        seen.assign(static_cast<size_t>(nch) * kWin * kWin, 0);
        for (int64_t i = r0; i < r1; ++i)
            for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
                const int64_t k = pos[col[p]];
                const int64_t slot = (k / kWin) * kWin * kWin + (i - r0) * kWin + k % kWin;
                if (seen[slot]) {
                    for (int32_t c : cols) pos[c] = -1;
                    return SPX_ERR_DUPLICATE;
                }
                seen[slot] = 1;
            }
        if (win_col && win_val) {
            for (int64_t k = 0; k < nch * kWin; ++k)
                win_col[g * kWin + k] = k < static_cast<int64_t>(cols.size()) ? cols[k] : -1;
            std::memset(win_val + g * kWin * kWin * vb, 0, static_cast<size_t>(nch * kWin * kWin * vb));
            for (int64_t i = r0; i < r1; ++i)
                for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
                    const int64_t k = pos[col[p]];
                    const int64_t e = (g + k / kWin) * kWin * kWin + (i - r0) * kWin + k % kWin;
                    std::memcpy(win_val + e * vb, val + p * vb, static_cast<size_t>(vb));
                }
        }
        for (int32_t c : cols) pos[c] = -1;
        g += nch;
        if (g * kWin > kI32Max) return SPX_ERR_INDEX_RANGE;
        if (win_ptr) win_ptr[w + 1] = static_cast<int32_t>(g);
    }
    if (nchunks_out) *nchunks_out = g;
    if (fill_out) *fill_out = g ? static_cast<double>(rp[M]) / (static_cast<double>(g) * kWin * kWin) : 0.0;
    return SPX_OK;
}

constexpr int32_t kDefaultTaskChunks = 16;  // chunks per task before a window is split

}  // namespace

namespace {

inline bool wplan_ok(const spx_wcsr_plan* P) { return P && P->magic == kWcsrPlanMagic; }

// One WCSR product: all windows (P == nullptr), or the plan's tasks followed
// by the fix-up of its split windows.
spx_status wcsr_run(const spx_wcsr_plan* P, int32_t M, int32_t K, int64_t nchunks, const int32_t* win_ptr,
                    const int32_t* win_col, const uint16_t* win_val, int32_t N, const uint16_t* B, int64_t ldb,
                    float alpha, float beta, float* C, int64_t ldc, void* scratch, size_t scratch_bytes,
                    cudaStream_t st) {
    if (M < 0 || K < 0 || N < 0 || nchunks < 0) return SPX_ERR_ARG;
    if (nchunks * kWin > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (N % 8) return SPX_ERR_UNSUPPORTED;  // B rows are gathered in 16-byte pieces
    if (M == 0 || N == 0) return SPX_OK;
    if (!win_ptr || !C || (nchunks > 0 && (!win_col || !win_val || !B))) return SPX_ERR_ARG;
    if (ldb < N || ldc < N) return SPX_ERR_ARG;
    if (ldb % 8 || !spx_aligned(win_val, 16) || !spx_aligned(B, 16) || !spx_aligned(C, 4) ||
        !spx_aligned(win_ptr, 4) || !spx_aligned(win_col, 4))
        return SPX_ERR_ALIGN;
    const int W = static_cast<int>((static_cast<int64_t>(M) + kWin - 1) / kWin);
    const int64_t ntasks = P ? static_cast<int64_t>(P->tasks.size() / 4) : W;
    const int nsplit = P ? static_cast<int>(P->splits.size() / 4) : 0;
    if (ntasks > 65535) return SPX_ERR_UNSUPPORTED;  // windows (tasks) map to gridDim.y
    const int4* tasks = P ? static_cast<const int4*>(P->d_table) : nullptr;
    const int4* splits = tasks ? tasks + ntasks : nullptr;
    float* partials = static_cast<float*>(scratch);
    if (nsplit > 0) {
        const size_t need = sizeof(float) * static_cast<size_t>(P->slots) * kWin * static_cast<size_t>(N);
        if (!scratch || scratch_bytes < need) return SPX_ERR_ARG;
        if (!spx_aligned(scratch, 16)) return SPX_ERR_ALIGN;
    }
    if (nchunks == 0) {
        dim3 grid((N + 255) / 256, M < 65535 ? M : 65535);
        wcsr_scale_kernel<<<grid, 256, 0, st>>>(C, ldc, M, N, beta);
        spx_note_launches(1);
        return spx_cuda_status(cudaGetLastError());
    }
    CUtensorMap tmA;
    if (!make_map(&tmA, win_val, kWin, static_cast<uint64_t>(nchunks) * kWin, kWin * 2)) return SPX_ERR_CUDA;
#define SPX_WCSR_LAUNCH(T)                                                                                     \
    do {                                                                                                       \
        if (set_smem_limit(wcsr_spmm_kernel<T>, kSmemW) != cudaSuccess) return SPX_ERR_CUDA;                   \
        wcsr_spmm_kernel<T><<<dim3((N + 127) / 128, static_cast<unsigned>(ntasks)), kThreads, kSmemW, st>>>(   \
            tmA, win_ptr, win_col, B, ldb, C, ldc, M, K, alpha, beta, kSpinLimit, tasks, partials, N, nchunks); \
    } while (0)
    if (tasks) SPX_WCSR_LAUNCH(true);
    else SPX_WCSR_LAUNCH(false);
#undef SPX_WCSR_LAUNCH
    uint64_t launches = 1;
    if (nsplit > 0) {
        wcsr_fixup_kernel<<<dim3((N + 255) / 256, kWin, nsplit < 65535 ? nsplit : 65535), 256, 0, st>>>(
            splits, nsplit, partials, M, N, alpha, beta, C, ldc);
        ++launches;
    }
    spx_note_launches(launches);
    return spx_cuda_status(cudaGetLastError());
}

}  // namespace

int spx_wcsr_check_take() { return spx_check_take(g_wcsr_check); }

int spx_wcsr_error_take() {
    int h = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_wcsr_error, sizeof(int)) != cudaSuccess) return static_cast<int>(SPX_ERR_CUDA);
    if (h != 0 && cudaMemcpyToSymbol(g_wcsr_error, &zero, sizeof(int)) != cudaSuccess)
        return static_cast<int>(SPX_ERR_CUDA);
    return h ? static_cast<int>(SPX_ERR_TIMEOUT) : 0;
}

extern "C" {

spx_status spx_build_wcsr(int32_t M, int32_t K, const int32_t* row_ptr, const int32_t* col, const void* val,
                          int32_t val_bytes, int32_t* win_ptr, int32_t* win_col, void* win_val, int64_t* nchunks_out,
                          double* fill_out, spx_loc where, spx_stream_t stream) {
    if (M < 0 || K < 0 || !row_ptr) return SPX_ERR_ARG;
    if (!(val_bytes == 1 || val_bytes == 2 || val_bytes == 4 || val_bytes == 8)) return SPX_ERR_ARG;
    if ((win_col == nullptr) != (win_val == nullptr)) return SPX_ERR_ARG;
    if (where == SPX_DEVICE)
        return spx_dev_build_wcsr(M, K, row_ptr, col, val, val_bytes, win_ptr, win_col, win_val, nchunks_out, fill_out,
                                  reinterpret_cast<cudaStream_t>(stream));
    if (where != SPX_HOST) return SPX_ERR_ARG;
    if (row_ptr[M] > 0 && (!col || !val)) return SPX_ERR_ARG;
    try {
        return build_wcsr_host(M, K, row_ptr, col, static_cast<const char*>(val), val_bytes, win_ptr, win_col,
                               static_cast<char*>(win_val), nchunks_out, fill_out);
    } catch (const std::bad_alloc&) {
        return SPX_ERR_NOMEM;
    }
}

spx_status spx_spmm_wcsr(int32_t M, int32_t K, int64_t nchunks, const int32_t* win_ptr, const int32_t* win_col,
                         const uint16_t* win_val, int32_t N, const uint16_t* B, int64_t ldb, float alpha, float beta,
                         float* C, int64_t ldc, spx_stream_t stream) {
    return wcsr_run(nullptr, M, K, nchunks, win_ptr, win_col, win_val, N, B, ldb, alpha, beta, C, ldc, nullptr, 0,
                    reinterpret_cast<cudaStream_t>(stream));
}

spx_status spx_wcsr_plan_build(int32_t M, int64_t nchunks, const int32_t* win_ptr, spx_loc where, int32_t max_chunks,
                               spx_wcsr_plan** out) {
    if (!out) return SPX_ERR_ARG;
    *out = nullptr;
    if (M < 0 || nchunks < 0 || !win_ptr || max_chunks < 0) return SPX_ERR_ARG;
    if (nchunks * kWin > kI32Max) return SPX_ERR_INDEX_RANGE;
    const int64_t W = (static_cast<int64_t>(M) + kWin - 1) / kWin;
    std::vector<int32_t> wp;
    try {
        wp.resize(static_cast<size_t>(W) + 1);
    } catch (const std::bad_alloc&) {
        return SPX_ERR_NOMEM;
    }
    if (where == SPX_DEVICE) {
        if (cudaMemcpy(wp.data(), win_ptr, sizeof(int32_t) * wp.size(), cudaMemcpyDeviceToHost) != cudaSuccess)
            return SPX_ERR_CUDA;
    } else if (where == SPX_HOST) {
        std::memcpy(wp.data(), win_ptr, sizeof(int32_t) * wp.size());
    } else {
        return SPX_ERR_ARG;
    }
    if (wp[0] != 0 || wp[W] != nchunks) return SPX_ERR_ARG;
    for (int64_t w = 0; w < W; ++w)
        if (wp[w + 1] < wp[w]) return SPX_ERR_NOT_SORTED;
    spx_wcsr_plan* P = new (std::nothrow) spx_wcsr_plan();
    if (!P) return SPX_ERR_NOMEM;
    P->M = M;
    P->nchunks = nchunks;
    P->max_chunks = max_chunks > 0 ? max_chunks : kDefaultTaskChunks;
    try {
        for (int64_t w = 0; w < W; ++w) {
            const int32_t g0 = wp[w], nch = wp[w + 1] - wp[w];
            if (nch <= P->max_chunks) {
                P->tasks.insert(P->tasks.end(), {static_cast<int32_t>(w), g0, nch, -1});
                continue;
            }
            const int32_t np = (nch + P->max_chunks - 1) / P->max_chunks, q = nch / np, r = nch % np;
            if (P->slots + np > kI32Max) {
                delete P;
                return SPX_ERR_INDEX_RANGE;
            }
            P->splits.insert(P->splits.end(), {static_cast<int32_t>(w), static_cast<int32_t>(P->slots), np, 0});
            int32_t start = g0;
            for (int32_t k = 0; k < np; ++k) {  // balanced pieces in chunk order
                const int32_t len = q + (k < r ? 1 : 0);
                P->tasks.insert(P->tasks.end(), {static_cast<int32_t>(w), start, len, static_cast<int32_t>(P->slots + k)});
                start += len;
            }
            P->slots += np;
        }
        // longest tasks first (stable): CTAs start in task order, so the long pieces run early and the
        // last wave holds short ones
        const size_t nt = P->tasks.size() / 4;
        std::vector<int32_t> order(nt);
        for (size_t i = 0; i < nt; ++i) order[i] = static_cast<int32_t>(i);
        std::stable_sort(order.begin(), order.end(),
                         [&](int32_t x, int32_t y) { return P->tasks[4 * x + 2] > P->tasks[4 * y + 2]; });
        std::vector<int32_t> sorted(P->tasks.size());
        for (size_t i = 0; i < nt; ++i)
            for (int f = 0; f < 4; ++f) sorted[4 * i + f] = P->tasks[4 * static_cast<size_t>(order[i]) + f];
        P->tasks.swap(sorted);
    } catch (const std::bad_alloc&) {
        delete P;
        return SPX_ERR_NOMEM;
    }
    P->table_bytes = sizeof(int32_t) * (P->tasks.size() + P->splits.size());
    P->magic = kWcsrPlanMagic;
    *out = P;
    return SPX_OK;
}

spx_status spx_wcsr_plan_info(const spx_wcsr_plan* P, spx_wcsr_plan_info_t* out) {
    if (!wplan_ok(P) || !out) return SPX_ERR_ARG;
    out->windows = (static_cast<int64_t>(P->M) + kWin - 1) / kWin;
    out->tasks = static_cast<int64_t>(P->tasks.size() / 4);
    out->split_windows = static_cast<int64_t>(P->splits.size() / 4);
    out->slots = P->slots;
    out->table_bytes = P->table_bytes;
    out->max_chunks = P->max_chunks;
    return SPX_OK;
}

spx_status spx_wcsr_plan_get_tasks(const spx_wcsr_plan* P, int32_t* tasks, int32_t* splits) {
    if (!wplan_ok(P)) return SPX_ERR_ARG;
    if (tasks && !P->tasks.empty()) std::memcpy(tasks, P->tasks.data(), sizeof(int32_t) * P->tasks.size());
    if (splits && !P->splits.empty()) std::memcpy(splits, P->splits.data(), sizeof(int32_t) * P->splits.size());
    return SPX_OK;
}

spx_status spx_wcsr_plan_upload(spx_wcsr_plan* P, void* table, size_t table_bytes, spx_stream_t stream) {
    if (!wplan_ok(P)) return SPX_ERR_ARG;
    if (P->table_bytes == 0) return SPX_OK;
    if (!table || table_bytes < P->table_bytes) return SPX_ERR_ARG;
    if (!spx_aligned(table, 16)) return SPX_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* d = static_cast<char*>(table);
    cudaError_t e = cudaMemcpyAsync(d, P->tasks.data(), sizeof(int32_t) * P->tasks.size(), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && !P->splits.empty())
        e = cudaMemcpyAsync(d + sizeof(int32_t) * P->tasks.size(), P->splits.data(), sizeof(int32_t) * P->splits.size(),
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    P->d_table = table;
    return SPX_OK;
}

spx_status spx_wcsr_plan_destroy(spx_wcsr_plan* P) {
    if (!P) return SPX_OK;
    if (!wplan_ok(P)) return SPX_ERR_ARG;
    P->magic = 0;
    delete P;
    return SPX_OK;
}

size_t spx_spmm_wcsr_planned_scratch_bytes(const spx_wcsr_plan* P, int32_t N) {
    if (!wplan_ok(P) || N < 0) return 0;
    return sizeof(float) * static_cast<size_t>(P->slots) * kWin * static_cast<size_t>(N);
}

spx_status spx_spmm_wcsr_planned(const spx_wcsr_plan* P, int32_t M, int32_t K, int64_t nchunks,
                                 const int32_t* win_ptr, const int32_t* win_col, const uint16_t* win_val, int32_t N,
                                 const uint16_t* B, int64_t ldb, float alpha, float beta, float* C, int64_t ldc,
                                 void* scratch, size_t scratch_bytes, spx_stream_t stream) {
    if (!wplan_ok(P)) return SPX_ERR_ARG;
    if (P->M != M || P->nchunks != nchunks) return SPX_ERR_ARG;
    if (P->table_bytes > 0 && !P->d_table) return SPX_ERR_NOT_READY;
    return wcsr_run(P, M, K, nchunks, win_ptr, win_col, win_val, N, B, ldb, alpha, beta, C, ldc, scratch,
                    scratch_bytes, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
