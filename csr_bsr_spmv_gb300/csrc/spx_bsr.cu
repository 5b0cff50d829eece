// spx_bsr.cu -- BSR SpMM C = A*B on the sm_103a tensor cores (tcgen05 + TMEM,
// TMA-fed), bf16 inputs, fp32 accumulation.
//
// [SpMM-ops] §3.4: loop over the nonzero blocks of a block-row, each a small
// dense GEMM on the matrix units, with asynchronous copies into shared memory
// and a multi-stage pipeline.  [AsyncSparse] §3 gives a Hopper design
// (warp-specialised TMA producer, WGMMA consumers, full/empty mbarrier ring);
// this kernel keeps the ring and the producer/consumer split and maps them to
// Blackwell: one thread issues tcgen05.mma into a TMEM accumulator,
// tcgen05.commit frees each stage, and the accumulator lives in TMEM, so no
// warpgroup holds it in registers.
//
// The MMA computes a transposed tile  D[n, r] += B[J*64 + k, n0 + n] * Ablk[r, k]
// with M = 128 (n), N = 64 (r), K = 16: B's tile is the A operand in MN-major
// form (n contiguous, exactly as B is stored) and the A block is the B operand
// in K-major form (k contiguous, as BSR stores a row-major block).  Both
// arrive by 2-D TMA with the 128-byte swizzle.  L2->SM traffic, not the
// tensor pipe, bounds this product: every B tile is read once per block-row
// that uses its block column.
//
// Default kernel (bsr_spmm_tile_kernel, "tile3"): non-persistent, one CTA per
// (128-column tile, block-row), three CTAs per SM, each an independent 3-deep
// TMA -> MMA ring; many small independent pipelines per SM measured fastest.
// Variants kept for measurement (SPX_BSR_VARIANT): other ring depths, 256-
// column tiles ("wideS"), and the persistent kernel below (bsr_spmm_tc_kernel:
// one CTA per SM walking a static tile schedule, five producer warps each
// owning a ring stage, one MMA warp, four epilogue warps, a double-buffered
// TMEM accumulator so the epilogue of tile i overlaps tile i+1).
//
// Every mbarrier wait is bounded (clock64); on expiry the CTA records an error
// word (read by spx_last_device_error), stops issuing, waits (bounded) for
// its copies and MMAs in flight, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <type_traits>
#include <mutex>

#include "spx_internal.h"
#include "spx_tc.cuh"

using namespace spx_tc;

namespace {

constexpr int kBlk = 64;                                // BSR block edge (rows = cols)
constexpr int kTileN = 256;                             // output columns per tile
constexpr int kHalves = kTileN / 128;                   // M = 128 MMA halves per tile
constexpr int kBoxes = kTileN / 64;                     // 64-column TMA boxes of B per stage
constexpr int kStages = 5;                              // smem ring depth
constexpr int kProducers = kStages;                     // producer warps; warp p owns ring stage p
constexpr int kMmaWarp = kProducers;                    // the MMA-issuing warp
constexpr int kThreads = 32 * (kProducers + 1 + 4);
constexpr uint32_t kABytes = kBlk * kBlk * 2;           // one bf16 A block, 8 KB
constexpr uint32_t kBBox = kBlk * 64 * 2;               // 64 k-rows x 64 n, 8 KB
constexpr uint32_t kStageBytes = kABytes + kBoxes * kBBox;  // 40 KB
constexpr uint32_t kAccCols = kHalves * 64;             // TMEM columns of one accumulator
constexpr uint32_t kTmemCols = 2 * kAccCols;            // double-buffered: 256
constexpr size_t kSmemBytes = kStages * kStageBytes + 1024 + 256;
constexpr uint32_t kIdesc = idesc_bf16_mn_k(128, 64);  // M = 128 output columns, N = 64 block rows
constexpr long long kSpinLimit = 2000000000LL;  // cycles (~1 s): only a broken pipeline reaches it

enum : int { kErrFull = 1, kErrEmpty = 2, kErrAcc = 3, kErrDrain = 4, kErrTmemEmpty = 5, kErrProbe = 6 };

__device__ int g_bsr_error;


__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_bsr_error, 0, code); }

// Persistent variant: 256-column tiles (two M = 128 halves share each A block),
// a static tile schedule over one CTA per SM, warps 0..4 TMA producers each
// owning one ring stage (lanes issue the A block and the four B boxes at
// once), warp 5 the MMA issuer, warps 6..9 the epilogue; the TMEM accumulator
// is double-buffered (2 x 128 columns).
__global__ void __launch_bounds__(kThreads, 1)
    bsr_spmm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const int* __restrict__ brp, const int* __restrict__ bcol, float* __restrict__ C,
                       long long ldc, float alpha, float beta, int N, int ntiles, int ntq, long long spin_limit) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ uint32_t s_issued_by[kProducers], s_consumed;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 1 KB alignment for the 128-byte swizzle atoms
    const uint32_t bars = base + kStages * kStageBytes;
    auto full_bar = [&](uint32_t s) { return bars + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bars + 8u * (kStages + s); };
    auto tfull_bar = [&](int b) { return bars + 8u * (2 * kStages + b); };
    auto tempty_bar = [&](int b) { return bars + 8u * (2 * kStages + 2 + b); };
    const uint32_t fin_bar = bars + 8u * (2 * kStages + 4);
    auto stage_a = [&](uint32_t s) { return base + s * kStageBytes; };
    auto stage_b = [&](uint32_t s) { return base + s * kStageBytes + kABytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4);  // one arrive per epilogue warp
        }
        mbar_init(fin_bar, 1);
        s_abort = 0;
        for (int p = 0; p < kProducers; ++p) s_issued_by[p] = 0;
        s_consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp < kProducers) {
        // ---------------- producers: warp p fills ring stage p for the ring positions g = p (mod kStages)
        const uint32_t s = static_cast<uint32_t>(warp);
        uint32_t G0 = 0, mine = 0;  // G0: ring position of the current tile's first block
        for (int t = blockIdx.x; t < ntiles && !s_abort; t += gridDim.x) {
            const int I = t / ntq, n0 = (t % ntq) * kTileN;
            const int nbox = min(kBoxes, (N - n0) / 64);  // 4, or 2 for a 128-wide last tile
            const int b0 = __ldg(brp + I), nb = __ldg(brp + I + 1) - b0;
            bool stop = false;
            for (int b = static_cast<int>((s + kStages - G0 % kStages) % kStages); b < nb; b += kStages) {
                const uint32_t g = G0 + static_cast<uint32_t>(b);
                const uint32_t ph = (g / kStages) & 1u;
                int ok = 1;
                if (lane == 0) ok = (mbar_wait(empty_bar(s), ph ^ 1u, spin_limit) && !s_abort) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) record_error(kErrEmpty);
                    s_abort = 1;
                    stop = true;
                    break;
                }
                if (lane == 0) mbar_expect_tx(full_bar(s), kABytes + nbox * kBBox);
                __syncwarp();
                if (lane == 0) {
                    tma_load_2d(stage_a(s), &tmA, 0, (b0 + b) * kBlk, full_bar(s));
                } else if (lane <= nbox) {
                    const int J = __ldg(bcol + b0 + b);
                    tma_load_2d(stage_b(s) + (lane - 1) * kBBox, &tmB, n0 + 64 * (lane - 1), J * kBlk, full_bar(s));
                }
                __syncwarp();
                mine = g + 1;
            }
            if (stop) break;
            G0 += static_cast<uint32_t>(nb);
        }
        if (lane == 0) s_issued_by[warp] = mine;  // 1 + the last ring position this warp filled (0: none)
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ---------------- MMA issuer
            uint32_t g = 0;
            int i = 0;
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int buf = i & 1;
                const uint32_t use = static_cast<uint32_t>(i >> 1);
                const int I = t / ntq;
                const int nh = min(kHalves, (N - (t % ntq) * kTileN) / 128);
                const int nb = __ldg(brp + I + 1) - __ldg(brp + I);
                if (!mbar_wait(tempty_bar(buf), (use & 1u) ^ 1u, spin_limit)) {
                    record_error(kErrTmemEmpty);
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * kAccCols;
                bool ok = true;
                for (int b = 0; b < nb; ++b, ++g) {
                    const uint32_t s = g % kStages, ph = (g / kStages) & 1u;
                    if (!mbar_wait(full_bar(s), ph, spin_limit)) {
                        record_error(kErrFull);
                        s_abort = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int h = 0; h < nh; ++h)
#pragma unroll
                        for (int ks = 0; ks < kBlk / 16; ++ks) {
                            // A operand: B's tile, MN-major; half h = TMA boxes 2h, 2h+1 (LBO 8 KB);
                            // 16 k-rows = two 8-row swizzle atoms (SBO 1 KB).
                            const uint64_t adesc = sw128_desc(stage_b(s) + 2 * h * kBBox + ks * 2048u, kBBox, 1024u);
                            // B operand: the A block, K-major; 16 k = 32 bytes inside each 128-byte row.
                            const uint64_t bdesc = sw128_desc(stage_a(s) + ks * 32u, 16u, 1024u);
                            mma_bf16(d + h * 64, adesc, bdesc, kIdesc, (b > 0 || ks > 0) ? 1u : 0u);
                        }
                    mma_commit(empty_bar(s));
                }
                if (nb > 0) mma_commit(tfull_bar(buf));  // arrives when this tile's MMAs complete
                else mbar_arrive(tfull_bar(buf));
                if (!ok) break;
            }
            s_consumed = g;
        }
    } else {
        // ---------------- epilogue warps 6..9: TMEM lane quarter (warp % 4) -> 32 output columns per half
        const int quarter = warp & 3;
        int i = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int buf = i & 1;
            const uint32_t use = static_cast<uint32_t>(i >> 1);
            const int I = t / ntq, n0 = (t % ntq) * kTileN;
            const int nh = min(kHalves, (N - n0) / 128);
            const int nb = __ldg(brp + I + 1) - __ldg(brp + I);
            int ok = 1;
            if (lane == 0) ok = mbar_wait(tfull_bar(buf), use & 1u, spin_limit) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) record_error(kErrAcc);
                s_abort = 1;
                break;
            }
            tc_fence_after();
            for (int h = 0; h < nh; ++h) {
                float* cp = C + static_cast<long long>(I) * kBlk * ldc + n0 + h * 128 + 32 * quarter + lane;
                if (nb == 0) {
                    for (int r = 0; r < kBlk; ++r) __stcs(cp + r * ldc, beta != 0.f ? beta * cp[r * ldc] : 0.f);
                    continue;
                }
#pragma unroll
                for (int c0 = 0; c0 < kBlk; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + (static_cast<uint32_t>(32 * quarter) << 16) + buf * kAccCols + h * 64 + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        float* q = cp + static_cast<long long>(c0 + j) * ldc;
                        const float acc = alpha * __uint_as_float(v[j]);
                        __stcs(q, beta != 0.f ? acc + beta * *q : acc);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(buf));
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (s_abort) {
        if (warp < kProducers && lane == 0) {
            // this warp's copies issued but never consumed: wait (bounded) until they have landed
            const uint32_t last = s_issued_by[warp];
            if (last > s_consumed && !mbar_wait(full_bar(warp), ((last - 1) / kStages) & 1u, spin_limit))
                record_error(kErrDrain);
        } else if (warp == kMmaWarp && lane == 0) {
            // MMAs in flight: one more commit, then wait (bounded) for it
            mma_commit(fin_bar);
            if (!mbar_wait(fin_bar, 0, spin_limit)) record_error(kErrDrain);
        }
    }
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

constexpr int32_t kDefaultTaskBlocks = 64;  // blocks per task before a block-row is split

// Split block-rows of a planned call: C rows of block-row I = alpha * (sum of
// its pieces' partial tiles, in piece order) + beta * C; one thread per
// (row, column), grid (column blocks, 64 rows, split block-rows).
__global__ void __launch_bounds__(256) bsr_fixup_kernel(const int4* __restrict__ splits, int nsplit,
                                                       const float* __restrict__ partials, int M, int N, float alpha,
                                                       float beta, float* C, long long ldc) {
    const int n = blockIdx.x * 256 + threadIdx.x, r = blockIdx.y;
    if (n >= N) return;
    for (int i = blockIdx.z; i < nsplit; i += gridDim.z) {
        const int4 sp = splits[i];  // {block-row, first slot, pieces, 0}
        if (sp.x * kBlk + r >= M) continue;  // a ragged last block-row: rows beyond M are not stored
        float s = 0.f;
        for (int k = 0; k < sp.z; ++k) s += __ldcs(partials + (static_cast<long long>(sp.y + k) * kBlk + r) * N + n);
        float* q = C + (static_cast<long long>(sp.x) * kBlk + r) * ldc + n;
        *q = beta != 0.f ? alpha * s + beta * *q : alpha * s;
    }
}

// ---------------------------------------------------------------- tile variant
// Non-persistent: one CTA per (128*HALVES-column tile, block-row), one TMA
// warp, one MMA thread, four epilogue warps, a STAGES-deep ring of {A block
// 8 KB, B tile 16*HALVES KB}.  Several CTAs share an SM (smem-bound), each an
// independent load/MMA pipeline, so one pipeline's hand-off latency is covered
// by the others.  HALVES = 2 shares each A block between two M = 128 MMAs
// (fewer A bytes per flop, fewer and larger CTAs).
constexpr int kTThreads = 128;

template <int HALVES>
__host__ __device__ constexpr uint32_t tile_stage_bytes() { return kABytes + 2 * HALVES * kBBox; }

template <int STAGES, int HALVES>
constexpr size_t tile_smem_bytes() { return STAGES * tile_stage_bytes<HALVES>() + 1024 + 256; }

template <int STAGES, int HALVES, bool TASKS = false>
__global__ void __launch_bounds__(kTThreads)
    bsr_spmm_tile_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const int* __restrict__ brp, const int* __restrict__ bcol, float* __restrict__ C,
                         long long ldc, float alpha, float beta, long long spin_limit, int M, int N,
                         const int4* __restrict__ tasks = nullptr, float* __restrict__ partials = nullptr) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_issued, s_consumed;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    constexpr uint32_t kSB = tile_stage_bytes<HALVES>();
    constexpr uint32_t kTmemColsT = 64 * HALVES;
    const uint32_t bars = base + STAGES * kSB;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    const uint32_t acc_bar = bars + 16u * STAGES;
    auto stage_a = [&](int s) { return base + s * kSB; };
    auto stage_b = [&](int s) { return base + s * kSB + kABytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * 128 * HALVES;
    // one block-row per grid row, or (planned call) one task: a piece of a
    // block-row's blocks {block-row, first block, blocks, partial slot or -1}
    int I, b0, nblk, slot = -1;
    if (TASKS) {
        const int4 t = tasks[blockIdx.y];
        I = t.x;
        b0 = t.y;
        nblk = t.z;
        slot = t.w;
    } else {
        I = blockIdx.y;
        b0 = __ldg(brp + I);
        nblk = __ldg(brp + I + 1) - b0;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(acc_bar, 1);
        s_abort = 0;
        s_issued = 0;
        s_consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTmemColsT)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = s_tmem;

    if (warp == 0) {
        // Producer warp: lane 0 waits for the free slot and arms the barrier,
        // then lanes 0..2*HALVES issue the stage's boxes side by side (the A
        // block and the 64-column boxes of the B tile).  The block columns
        // of this block-row sit in registers, 32 at a time.
        int b = 0, jreg = 0;
        for (; b < nblk; ++b) {
            const int s = b % STAGES;
            const uint32_t ph = (b / STAGES) & 1u;
            if ((b & 31) == 0) jreg = b + lane < nblk ? __ldg(bcol + b0 + b + lane) : 0;
            const int J = __shfl_sync(0xffffffffu, jreg, b & 31);
            int ok = 1;
            if (lane == 0) ok = (mbar_wait(empty_bar(s), ph ^ 1u, spin_limit) && !s_abort) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    record_error(kErrEmpty);
                    s_abort = 1;
                }
                break;
            }
            if (lane == 0) mbar_expect_tx(full_bar(s), kSB);
            __syncwarp();
            if (lane == 0) tma_load_2d(stage_a(s), &tmA, 0, (b0 + b) * kBlk, full_bar(s));
            else if (lane <= 2 * HALVES)
                tma_load_2d(stage_b(s) + (lane - 1) * kBBox, &tmB, n0 + 64 * (lane - 1), J * kBlk, full_bar(s));
        }
        if (lane == 0) s_issued = b;
    } else if (warp == 1 && lane == 0) {
        int b = 0;
        for (; b < nblk; ++b) {
            const int s = b % STAGES;
            const uint32_t ph = (b / STAGES) & 1u;
            if (!mbar_wait(full_bar(s), ph, spin_limit)) {
                record_error(kErrFull);
                s_abort = 1;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < kBlk / 16; ++ks) {
                const uint64_t bdesc = sw128_desc(stage_a(s) + ks * 32u, 16u, 1024u);
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    const uint64_t adesc = sw128_desc(stage_b(s) + 2 * h * kBBox + ks * 2048u, kBBox, 1024u);
                    mma_bf16(tmem_d + 64 * h, adesc, bdesc, kIdesc, (b > 0 || ks > 0) ? 1u : 0u);
                }
            }
            mma_commit(empty_bar(s));
        }
        s_consumed = b;
        if (b > 0) mma_commit(acc_bar);
        else mbar_arrive(acc_bar);
    }
    __syncwarp();

    int ok = 1;
    if (lane == 0) ok = mbar_wait(acc_bar, 0, spin_limit) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) record_error(kErrAcc);
    tc_fence_after();
    // C rows of this block-row inside [0, M) (a ragged last block-row is zero-padded in A)
    const int mrows = min(kBlk, M - I * kBlk);
#pragma unroll
    for (int h = 0; h < HALVES; ++h) {
        const int cn = n0 + 128 * h + 32 * warp + lane;  // this thread's column; columns >= N are not stored
        const bool cok = cn < N;
        float* cp = C + static_cast<long long>(I) * kBlk * ldc + cn;
        // a piece of a split block-row writes its raw partial tile (1 * sum, exact; the fix-up applies alpha/beta)
        const bool raw = TASKS && slot >= 0;
        float* dst = raw ? partials + static_cast<long long>(slot) * kBlk * N + cn : cp;
        const long long dstride = raw ? N : ldc;
        const int rows = raw ? kBlk : mrows;
        const float ealpha = raw ? 1.f : alpha, ebeta = raw ? 0.f : beta;
        if (nblk == 0) {
            if (cok)
                for (int r = 0; r < mrows; ++r) __stcs(cp + r * ldc, beta != 0.f ? beta * cp[r * ldc] : 0.f);
        } else if (ok && !s_abort) {
            // GUARD: the tile reaches past row M or column N (a ragged edge), so each store is checked;
            // whole tiles (CTA-uniform test) take the unchecked copy of the loop
            auto drain = [&](auto guard) {
                constexpr bool GUARD = decltype(guard)::value;
#pragma unroll
                for (int c0 = 0; c0 < kBlk; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem_d + (static_cast<uint32_t>(32 * warp) << 16) + 64 * h + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (!GUARD || (cok && c0 + j < rows)) {
                            float* q = dst + static_cast<long long>(c0 + j) * dstride;
                            const float acc = ealpha * __uint_as_float(v[j]);
                            __stcs(q, ebeta != 0.f ? acc + ebeta * *q : acc);
                        }
                    }
                }
            };
            if (n0 + 128 * (h + 1) <= N && rows == kBlk) drain(std::false_type{});
            else drain(std::true_type{});
        }
    }
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0) {
        for (int b = s_consumed; b < s_issued; ++b)
            if (!mbar_wait(full_bar(b % STAGES), (b / STAGES) & 1u, spin_limit)) {
                record_error(kErrDrain);
                break;
            }
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_d), "r"(kTmemColsT) : "memory");
}

// Test aid for the bounded waits: one thread arms an mbarrier that nothing
// completes and waits on it with the pipelines' own bounded wait; when the
// limit runs out it records the timeout in the error word, as a stalled
// pipeline would, and the kernel returns.
__global__ void wait_probe_kernel(long long limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!mbar_wait(smem_u32(&bar), 0u, limit)) record_error(kErrProbe);
    }
}

// C = beta * C (a BSR matrix without stored blocks).
__global__ void bsr_scale_kernel(float* C, long long ldc, int M, int N, float beta) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= N) return;
    for (int r = blockIdx.y; r < M; r += gridDim.y) {
        float* q = C + static_cast<long long>(r) * ldc + c;
        *q = beta * *q;
    }
}

// ------------------------------------------------------------ host side

}  // namespace

extern "C" {

spx_status spx_spmm_bsr(int32_t M, int32_t K, int32_t br, int32_t bc, int64_t nnzb, const int32_t* bsr_row_ptr,
                        const int32_t* bsr_col, const uint16_t* bsr_val, int32_t N, const uint16_t* B, int64_t ldb,
                        float alpha, float beta, float* C, int64_t ldc, spx_stream_t stream) {
    if (M < 0 || K < 0 || N < 0 || nnzb < 0 || br <= 0 || bc <= 0) return SPX_ERR_ARG;
    if (nnzb > kI32Max || static_cast<int64_t>(nnzb) * kBlk > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (br != kBlk || bc != kBlk) return SPX_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return SPX_OK;
    if (!bsr_row_ptr || !C || (nnzb > 0 && (!bsr_col || !bsr_val || !B))) return SPX_ERR_ARG;
    if (ldb < N || ldc < N) return SPX_ERR_ARG;
    if (ldb % 8 || !spx_aligned(bsr_val, 16) || !spx_aligned(B, 16) || !spx_aligned(C, 4) ||
        !spx_aligned(bsr_row_ptr, 4) || !spx_aligned(bsr_col, 4))
        return SPX_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (nnzb == 0 && beta == 0.f) {
        // no stored block: C = 0
        return spx_cuda_status(cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 4, 0, static_cast<size_t>(N) * 4,
                                                 static_cast<size_t>(M), st));
    }
    if (nnzb == 0) {
        // no stored block: C = beta * C
        dim3 grid((N + 255) / 256, M < 65535 ? M : 65535);
        bsr_scale_kernel<<<grid, 256, 0, st>>>(C, ldc, M, N, beta);
        spx_note_launches(1);
        return spx_cuda_status(cudaGetLastError());
    }
    CUtensorMap tmA, tmB;
    if (!make_map(&tmA, bsr_val, kBlk, static_cast<uint64_t>(nnzb) * kBlk, kBlk * 2) ||
        !make_map(&tmB, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K), static_cast<uint64_t>(ldb) * 2))
        return SPX_ERR_CUDA;
    // Variant: "tileS" = non-persistent 128-column tiles with an S-deep ring
    // (S = 2..5; smaller rings fit more CTAs per SM), "wideS" = the same with
    // 256-column tiles (S = 2..4, N a multiple of 256), "persistent" = the
    // persistent 256-column kernel.  SPX_BSR_VARIANT overrides the default.
    static const int env_variant = [] {  // read once, thread-safe
        int v = 3;
        if (const char* e = std::getenv("SPX_BSR_VARIANT")) {
            if (!std::strcmp(e, "persistent")) v = 0;
            else if (!std::strncmp(e, "tile", 4) && e[4] >= '2' && e[4] <= '5' && e[5] == 0) v = e[4] - '0';
            else if (!std::strncmp(e, "wide", 4) && e[4] >= '2' && e[4] <= '4' && e[5] == 0) v = 10 + e[4] - '0';
        }
        return v;
    }();
    // per call: 256-column tiles need N % 256 == 0, and the persistent and 256-column kernels whole
    // 64-row block-rows, 64-row block columns and 128-column tiles; other shapes take the tile kernel
    const bool ragged = M % kBlk || K % kBlk || N % 128;
    int variant = env_variant;
    if ((variant >= 10 && (N % 256 || ragged)) || (variant == 0 && ragged)) variant = 3;
    if (variant == 0) {
        if (set_smem_limit(bsr_spmm_tc_kernel, kSmemBytes) != cudaSuccess) return SPX_ERR_CUDA;
        int dev = 0, nsm = 0;  // SM count of the current device (cheap attribute query)
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SPX_ERR_CUDA;
        const int ntq = (N + kTileN - 1) / kTileN;
        const long long tiles = static_cast<long long>(M / kBlk) * ntq;
        if (tiles > kI32Max) return SPX_ERR_INDEX_RANGE;
        const int grid = static_cast<int>(tiles < nsm ? tiles : nsm);
        bsr_spmm_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(tmA, tmB, bsr_row_ptr, bsr_col, C, ldc, alpha, beta, N,
                                                               static_cast<int>(tiles), ntq, kSpinLimit);
    } else {
        const int MB = (M + kBlk - 1) / kBlk;
        if (MB > 65535) return SPX_ERR_UNSUPPORTED;  // block-rows map to gridDim.y
        switch (variant) {
#define SPX_TILE(S, H, V)                                                                                      \
    case V: {                                                                                                     \
        if (set_smem_limit(bsr_spmm_tile_kernel<S, H>, tile_smem_bytes<S, H>()) != cudaSuccess)                   \
            return SPX_ERR_CUDA;                                                                                  \
        bsr_spmm_tile_kernel<S, H><<<dim3((N + 128 * H - 1) / (128 * H), MB), kTThreads, tile_smem_bytes<S, H>(), \
                                     st>>>(tmA, tmB, bsr_row_ptr, bsr_col, C, ldc, alpha, beta, kSpinLimit, M, N); \
        break;                                                                                                    \
    }
            SPX_TILE(2, 1, 2) SPX_TILE(3, 1, 3) SPX_TILE(4, 1, 4) SPX_TILE(5, 1, 5)
            SPX_TILE(2, 2, 12) SPX_TILE(3, 2, 13) SPX_TILE(4, 2, 14)
#undef SPX_TILE
        }
    }
    spx_note_launches(1);
    return spx_cuda_status(cudaGetLastError());
}

spx_status spx_bsr_plan_build(int32_t M, int64_t nnzb, const int32_t* bsr_row_ptr, spx_loc where, int32_t max_blocks,
                              spx_wcsr_plan** out) {
    return spx_wcsr_plan_build(M, nnzb, bsr_row_ptr, where, max_blocks > 0 ? max_blocks : kDefaultTaskBlocks, out);
}

size_t spx_spmm_bsr_planned_scratch_bytes(const spx_wcsr_plan* plan, int32_t N) {
    return spx_spmm_wcsr_planned_scratch_bytes(plan, N);
}

spx_status spx_spmm_bsr_planned(const spx_wcsr_plan* P, int32_t M, int32_t K, int32_t br, int32_t bc, int64_t nnzb,
                                const int32_t* bsr_row_ptr, const int32_t* bsr_col, const uint16_t* bsr_val,
                                int32_t N, const uint16_t* B, int64_t ldb, float alpha, float beta, float* C,
                                int64_t ldc, void* scratch, size_t scratch_bytes, spx_stream_t stream) {
    if (!P || P->magic != kWcsrPlanMagic) return SPX_ERR_ARG;
    if (P->M != M || P->nchunks != nnzb) return SPX_ERR_ARG;
    if (M < 0 || K < 0 || N < 0 || nnzb < 0 || br <= 0 || bc <= 0) return SPX_ERR_ARG;
    if (nnzb > kI32Max || static_cast<int64_t>(nnzb) * kBlk > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (br != kBlk || bc != kBlk) return SPX_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return SPX_OK;
    if (nnzb == 0)  // nothing to split
        return spx_spmm_bsr(M, K, br, bc, nnzb, bsr_row_ptr, bsr_col, bsr_val, N, B, ldb, alpha, beta, C, ldc, stream);
    if (P->table_bytes > 0 && !P->d_table) return SPX_ERR_NOT_READY;
    if (!bsr_row_ptr || !C || !bsr_col || !bsr_val || !B) return SPX_ERR_ARG;
    if (ldb < N || ldc < N) return SPX_ERR_ARG;
    if (ldb % 8 || !spx_aligned(bsr_val, 16) || !spx_aligned(B, 16) || !spx_aligned(C, 4) ||
        !spx_aligned(bsr_row_ptr, 4) || !spx_aligned(bsr_col, 4))
        return SPX_ERR_ALIGN;
    const int64_t ntasks = static_cast<int64_t>(P->tasks.size() / 4);
    const int nsplit = static_cast<int>(P->splits.size() / 4);
    if (ntasks > 65535) return SPX_ERR_UNSUPPORTED;  // tasks map to gridDim.y
    if (nsplit > 0) {
        const size_t need = sizeof(float) * static_cast<size_t>(P->slots) * kBlk * static_cast<size_t>(N);
        if (!scratch || scratch_bytes < need) return SPX_ERR_ARG;
        if (!spx_aligned(scratch, 16)) return SPX_ERR_ALIGN;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap tmA, tmB;
    if (!make_map(&tmA, bsr_val, kBlk, static_cast<uint64_t>(nnzb) * kBlk, kBlk * 2) ||
        !make_map(&tmB, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K), static_cast<uint64_t>(ldb) * 2))
        return SPX_ERR_CUDA;
    const int4* tasks = static_cast<const int4*>(P->d_table);
    float* partials = static_cast<float*>(scratch);
    if (set_smem_limit(bsr_spmm_tile_kernel<3, 1, true>, tile_smem_bytes<3, 1>()) != cudaSuccess) return SPX_ERR_CUDA;
    bsr_spmm_tile_kernel<3, 1, true><<<dim3((N + 127) / 128, static_cast<unsigned>(ntasks)), kTThreads,
                                       tile_smem_bytes<3, 1>(), st>>>(tmA, tmB, bsr_row_ptr, bsr_col, C, ldc, alpha,
                                                                      beta, kSpinLimit, M, N, tasks, partials);
    uint64_t launches = 1;
    if (nsplit > 0) {
        bsr_fixup_kernel<<<dim3((N + 255) / 256, kBlk, nsplit < 65535 ? nsplit : 65535), 256, 0, st>>>(
            tasks + ntasks, nsplit, partials, M, N, alpha, beta, C, ldc);
        ++launches;
    }
    spx_note_launches(launches);
    return spx_cuda_status(cudaGetLastError());
}

spx_status spx_wait_probe(int64_t limit_cycles, spx_stream_t stream) {
    if (limit_cycles < 0 || limit_cycles > kSpinLimit) return SPX_ERR_ARG;
    wait_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_cycles);
    spx_note_launches(1);
    return spx_cuda_status(cudaGetLastError());
}

spx_status spx_last_device_error(spx_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int h = 0;
    const int zero = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&h, g_bsr_error, sizeof(int));
    if (e == cudaSuccess && h != 0) e = cudaMemcpyToSymbol(g_bsr_error, &zero, sizeof(int));
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    const int coo = spx_coo_error_take();
    const int wcsr = spx_wcsr_error_take();
    if (h || wcsr == SPX_ERR_TIMEOUT) return SPX_ERR_TIMEOUT;
    if (wcsr == SPX_ERR_CUDA) return SPX_ERR_CUDA;
    return static_cast<spx_status>(coo);
}

}  // extern "C"
