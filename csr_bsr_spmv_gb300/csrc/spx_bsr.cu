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
// Two kernels share the tile (128 output columns x one 64-row block-row), the
// 3-deep ring of {A block 8 KB, B tile 16 KB} stages and three CTAs per SM:
//   bsr_spmm_persist_kernel (spx_spmm_bsr): persistent, a static schedule of
//     tiles per CTA, the ring running on across tiles, a double-buffered TMEM
//     accumulator so each tile's epilogue overlaps the next tile's MMAs
//     (86.7 -> 78.5 us on 256 block-rows of 26 blocks, N = 1024); when the
//     last round of tiles would leave half the CTAs idle, its tiles are cut
//     into a head piece (this launch) and a tail piece (a second launch of
//     the TAIL variant that adds into C once the first has finished);
//   bsr_spmm_tile_kernel (spx_spmm_bsr_planned): one CTA per (task, column
//     tile), where tasks are block-rows or pieces of unequal length and the
//     hardware's dynamic CTA scheduling balances them better.
// The persistent kernel also takes other block shapes (GEN = true, the
// shape in a TcShape argument): br rows as the MMA's N (a multiple of 16 up
// to 128), bc columns in 64-column chunks of one ring stage each, a narrower
// block read with its columns past bc zero-filled and only bc / 16 K-steps.
// Three CTAs of three stages per SM measured fastest: two CTAs of four
// stages, four of two and one of five were slower, as were 256-column tiles
// sharing each A block; many independent pipelines per SM beat deep ones.
//
// Every mbarrier wait is bounded (clock64); on expiry the CTA records an error
// word (read by spx_last_device_error), stops issuing, waits (bounded) for
// its copies and MMAs in flight, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <type_traits>

#include "spx_check.cuh"
#include "spx_internal.h"
#include "spx_tc.cuh"

using namespace spx_tc;

namespace {

constexpr int kBlk = 64;                                // BSR block edge (rows = cols)
constexpr uint32_t kABytes = kBlk * kBlk * 2;           // one bf16 A block, 8 KB
constexpr uint32_t kBBox = kBlk * 64 * 2;               // 64 k-rows x 64 n, 8 KB
constexpr uint32_t kIdesc = idesc_bf16_mn_k(128, 64);  // M = 128 output columns, N = 64 block rows
constexpr long long kSpinLimit = 2000000000LL;  // cycles (~1 s): only a broken pipeline reaches it

enum : int { kErrFull = 1, kErrEmpty = 2, kErrAcc = 3, kErrDrain = 4, kErrProbe = 6 };

__device__ int g_bsr_error;


__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_bsr_error, 0, code); }

SPX_CHECK_WORD(g_bsr_check)

// The checked build's tests (the TMA engine already turns an out-of-range box
// into zeros, so these guard the index reads and report the error): a block
// column in [0, KB) -- else it becomes KB, a box past the end, read as zeros --
// and a block-row's blocks inside [0, nnzb) -- else the block-row counts as
// empty, identically in every role of the kernel.
__device__ __forceinline__ int checked_bcol(int J, int KB) {
    if (SPX_CHECKED && (J < 0 || J >= KB)) {
        check_fail();
        return KB;
    }
    return J;
}
__device__ __forceinline__ int checked_nb(int b0, int nb, long long nnzb, bool report) {
    if (SPX_CHECKED && !(b0 >= 0 && nb >= 0 && b0 + static_cast<long long>(nb) <= nnzb)) {
        if (report) check_fail();
        return 0;
    }
    return nb;
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

// ---------------------------------------------------------------- the tile kernel
// Non-persistent: one CTA per (128-column tile, block-row), one TMA warp, one
// MMA thread, four epilogue warps, a STAGES-deep ring of {A block 8 KB, B tile
// 16 KB}.  Three CTAs share an SM (smem-bound), each an independent load/MMA
// pipeline, so one pipeline's hand-off latency is covered by the others.
constexpr int kTThreads = 128;
constexpr int STAGES = 3;
constexpr uint32_t kSB = kABytes + 2 * kBBox;                 // one ring stage: 24 KB
constexpr size_t kTileSmem = STAGES * kSB + 1024 + 256;      // the ring, 1 KB alignment slack, barriers
constexpr uint32_t kTmemColsT = 64;                           // the 128 x 64 fp32 accumulator

__global__ void __launch_bounds__(kTThreads)
    bsr_spmm_tile_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const int* __restrict__ bcol, float* __restrict__ C, long long ldc, float alpha, float beta,
                         long long spin_limit, int M, int N, const int4* __restrict__ tasks,
                         float* __restrict__ partials, int KB) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_issued, s_consumed;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + STAGES * kSB;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    const uint32_t acc_bar = bars + 16u * STAGES;
    auto stage_a = [&](int s) { return base + s * kSB; };
    auto stage_b = [&](int s) { return base + s * kSB + kABytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * 128;
    // one task per grid row: a block-row or a piece of one {block-row, first block, blocks, partial slot or -1}
    const int4 task = tasks[blockIdx.y];
    const int I = task.x, b0 = task.y, nblk = task.z, slot = task.w;

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
        // then lanes 0..2 issue the stage's boxes side by side (the A block
        // and the two 64-column boxes of the B tile).  The block columns
        // of this block-row sit in registers, 32 at a time.
        int b = 0, jreg = 0;
        for (; b < nblk; ++b) {
            const int s = b % STAGES;
            const uint32_t ph = (b / STAGES) & 1u;
            if ((b & 31) == 0) jreg = b + lane < nblk ? __ldg(bcol + b0 + b + lane) : 0;
            const int J = checked_bcol(__shfl_sync(0xffffffffu, jreg, b & 31), KB);
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
            else if (lane <= 2)
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
                const uint64_t adesc = sw128_desc(stage_b(s) + ks * 2048u, kBBox, 1024u);
                mma_bf16(tmem_d, adesc, bdesc, kIdesc, (b > 0 || ks > 0) ? 1u : 0u);
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
    {
        const int cn = n0 + 32 * warp + lane;  // this thread's column; columns >= N are not stored
        const bool cok = cn < N;
        float* cp = C + static_cast<long long>(I) * kBlk * ldc + cn;
        // a piece of a split block-row writes its raw partial tile (1 * sum, exact; the fix-up applies alpha/beta)
        const bool raw = slot >= 0;
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
                    tmem_ld32(tmem_d + (static_cast<uint32_t>(32 * warp) << 16) + c0, v);
                    float old[32];  // beta != 0: all 32 old values are loaded before any store (no load waits on one)
                    if (ebeta != 0.f) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            old[j] = (!GUARD || (cok && c0 + j < rows)) ? dst[static_cast<long long>(c0 + j) * dstride] : 0.f;
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (!GUARD || (cok && c0 + j < rows)) {
                            float* q = dst + static_cast<long long>(c0 + j) * dstride;
                            const float acc = ealpha * __uint_as_float(v[j]);
                            __stcs(q, ebeta != 0.f ? acc + ebeta * old[j] : acc);
                        }
                    }
                }
            };
            if (n0 + 128 <= N && rows == kBlk) drain(std::false_type{});
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

// ---------------------------------------------------------------- the persistent kernel
// The same tiles (128 output columns x one block-row: 64 rows, or br for
// the other shapes) and the same ring stages as the tile kernel, but a CTA
// stays resident and walks a static schedule of tiles (tile = block-row *
// column tiles + column tile; CTA b runs tiles b, b + G, b + 2G, ...), so the
// ring never drains between tiles:
//   warps 0-3 : epilogue (TMEM lane quarter = warp), one tile behind the MMAs;
//   warp 4    : TMA producer, one ring position per block (per 64-column chunk
//               of a block), across tiles;
//   warp 5    : lane 0 issues the MMAs into one of two TMEM accumulators
//               (64 columns each for 64-row blocks), so tile i+1 accumulates
//               while tile i is stored.
// On dense block-rows (256 blocks each) the tile kernel reaches its steady
// rate; on short ones (26 blocks) each CTA's start-up, pipeline fill and
// epilogue are paid per tile, and this kernel hides them.
constexpr int kPThreads = 192;
constexpr uint32_t kPTmemCols = 2 * kTmemColsT;
enum : int { kErrTmemFree = 7 };

// Block shapes other than 64 x 64 on the same kernel (GEN = true): br rows
// (the MMA's N, a multiple of 16 up to 128) and bc columns, taken in chunks
// of up to 64 (one ring stage each; bc <= 64 or a multiple of 64).  The
// A box is always 64 wide: a block narrower than 64 columns is read with the
// columns past bc zero-filled by the copy engine, and only bc / 16 K-steps
// are issued on its chunk.  The B box has min(bc, 64) rows, so no stage
// reads B rows of another block column.
struct TcShape {
    int br, bc, kc, ksl, brows;  // rows, columns, chunks per block, K-steps of the last chunk, B box rows
    uint32_t abytes, sb, tx;     // A region and stage bytes (the B region is 16 KB), bytes a stage's copies bring
    uint32_t pitch, cols;        // TMEM columns per accumulator (a power of two) and allocated (two of them)
};

__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t v) {
    uint32_t p = 32;
    while (p < v) p <<= 1;
    return p;
}

inline TcShape tc_shape(int br, int bc) {
    TcShape sh{};
    sh.br = br;
    sh.bc = bc;
    sh.kc = (bc + kBlk - 1) / kBlk;
    sh.ksl = (bc - (sh.kc - 1) * kBlk) / 16;
    sh.brows = bc < kBlk ? bc : kBlk;
    sh.abytes = static_cast<uint32_t>(kBlk * 2 * br);
    sh.sb = sh.abytes + 2 * kBBox;
    sh.tx = sh.abytes + 2u * static_cast<uint32_t>(64 * 2 * sh.brows);
    sh.pitch = pow2_at_least(static_cast<uint32_t>(br));
    sh.cols = 2 * sh.pitch;
    return sh;
}

// Shapes the tensor-core kernel takes besides 64 x 64.
inline bool tc_general_shape(int br, int bc) {
    return br % 16 == 0 && br >= 16 && br <= 128 && bc % 16 == 0 && bc >= 16 && (bc <= kBlk || bc % kBlk == 0);
}

// The work of one CTA of the persistent kernel, item by item.  First launch:
// the whole tiles c, c + G, c + 2G, ... below `full`, then -- when c < tail --
// the head piece of tile full + c (its first nb/2 blocks), stored as a whole
// tile would be.  Second launch (TAIL): one item, the tail piece of tile
// full + c (the other blocks), added into C once the first launch is done.
// tail == 0: no pieces, every tile below full (= all tiles) whole.
struct Item {
    int t, I, b0, blo, bhi;  // tile, block-row, its first block, block range [blo, bhi) of the block-row
};
template <bool TAIL>
__device__ __forceinline__ bool work_item(int i, int G, int full, int tail, int ntq, const int* __restrict__ brp,
                                          long long nnzb, bool report, Item& it) {
    const int c = static_cast<int>(blockIdx.x);
    int t, part;  // part: 0 whole tile, 1 head piece, 2 tail piece
    if (TAIL) {
        if (i > 0 || c >= tail) return false;
        t = full + c;
        part = 2;
    } else {
        const int whole = c < full ? (full - c + G - 1) / G : 0;  // whole tiles of this CTA
        if (i < whole) {
            t = c + i * G;
            part = 0;
        } else if (i == whole && c < tail) {
            t = full + c;
            part = 1;
        } else {
            return false;
        }
    }
    it.t = t;
    it.I = t / ntq;
    it.b0 = __ldg(brp + it.I);
    const int nb = checked_nb(it.b0, __ldg(brp + it.I + 1) - it.b0, nnzb, report);
    it.blo = part == 2 ? nb / 2 : 0;
    it.bhi = part == 1 ? nb / 2 : nb;
    return true;
}

template <bool TAIL = false, bool GEN = false>
__global__ void __launch_bounds__(kPThreads, 3)  // three resident per SM (the shared-memory limit)
    bsr_spmm_persist_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const int* __restrict__ brp, const int* __restrict__ bcol, float* __restrict__ C,
                            long long ldc, float alpha, float beta, long long spin_limit, int M, int N, int full,
                            int tail, int ntq, int KB, long long nnzb, TcShape sh) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ uint32_t s_issued, s_consumed;

    // the block shape: constants for 64 x 64, the launch's TcShape otherwise
    const int BR = GEN ? sh.br : kBlk, BC = GEN ? sh.bc : kBlk, KC = GEN ? sh.kc : 1, KSL = GEN ? sh.ksl : 4;
    const uint32_t SB = GEN ? sh.sb : kSB, AB = GEN ? sh.abytes : kABytes, TX = GEN ? sh.tx : kSB;
    const uint32_t PITCH = GEN ? sh.pitch : kTmemColsT, TCOLS = GEN ? sh.cols : kPTmemCols;
    const uint32_t IDESC = GEN ? idesc_bf16_mn_k(128, static_cast<uint32_t>(BR)) : kIdesc;

    // the second launch may start while the first runs: let it be scheduled as this grid's SMs free up
    if (!TAIL) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + STAGES * SB;
    auto full_bar = [&](uint32_t s) { return bars + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bars + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
    const uint32_t fin_bar = bars + 8u * (2 * STAGES + 4);
    auto stage_a = [&](uint32_t s) { return base + s * SB; };
    auto stage_b = [&](uint32_t s) { return base + s * SB + AB; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4);  // one arrive per epilogue warp
        }
        mbar_init(fin_bar, 1);
        s_abort = 0;
        s_issued = 0;
        s_consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(TCOLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    Item it;
    if (warp == 4) {
        // ---------------- producer: lane 0 waits for a free stage and arms it, lanes 0..2 issue its boxes
        uint32_t g = 0;
        bool stop = false;
        for (int i = 0; !stop && !s_abort && work_item<TAIL>(i, G, full, tail, ntq, brp, nnzb, lane == 0, it); ++i) {
            const int n0 = (it.t % ntq) * 128;
            int jreg = 0;
            for (int b = it.blo; !stop && b < it.bhi; ++b) {
                const int k = b - it.blo;
                if ((k & 31) == 0) jreg = b + lane < it.bhi ? __ldg(bcol + it.b0 + b + lane) : 0;
                const int J = checked_bcol(__shfl_sync(0xffffffffu, jreg, k & 31), KB);
                for (int kc = 0; kc < KC; ++kc, ++g) {  // the block's column chunks, one stage each
                    const uint32_t s = g % STAGES, ph = (g / STAGES) & 1u;
                    int ok = 1;
                    if (lane == 0) ok = (mbar_wait(empty_bar(s), ph ^ 1u, spin_limit) && !s_abort) ? 1 : 0;
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) {
                        if (lane == 0) {
                            record_error(kErrEmpty);
                            s_abort = 1;
                        }
                        stop = true;
                        break;
                    }
                    if (lane == 0) mbar_expect_tx(full_bar(s), TX);
                    __syncwarp();
                    if (lane == 0) tma_load_2d(stage_a(s), &tmA, kBlk * kc, (it.b0 + b) * BR, full_bar(s));
                    else if (lane <= 2)
                        tma_load_2d(stage_b(s) + (lane - 1) * kBBox, &tmB, n0 + 64 * (lane - 1), J * BC + kBlk * kc,
                                    full_bar(s));
                    __syncwarp();
                }
            }
        }
        if (lane == 0) s_issued = g;
    } else if (warp == 5) {
        if (lane == 0) {
            // ---------------- MMA issuer
            uint32_t g = 0;
            bool ok = true;
            for (int i = 0; ok && work_item<TAIL>(i, G, full, tail, ntq, brp, nnzb, false, it); ++i) {
                const int buf = i & 1;
                const uint32_t use = static_cast<uint32_t>(i >> 1);
                if (!mbar_wait(tempty_bar(buf), (use & 1u) ^ 1u, spin_limit) || s_abort) {
                    record_error(kErrTmemFree);
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * PITCH;
                for (int b = it.blo; ok && b < it.bhi; ++b) {
                    for (int kc = 0; kc < KC; ++kc, ++g) {
                        const uint32_t s = g % STAGES, ph = (g / STAGES) & 1u;
                        if (!mbar_wait(full_bar(s), ph, spin_limit)) {
                            record_error(kErrFull);
                            s_abort = 1;
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const int nks = kc == KC - 1 ? KSL : 4;  // K-steps of 16 columns in this chunk
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            if (ks >= nks) break;
                            const uint64_t bdesc = sw128_desc(stage_a(s) + ks * 32u, 16u, 1024u);
                            const uint64_t adesc = sw128_desc(stage_b(s) + ks * 2048u, kBBox, 1024u);
                            mma_bf16(d, adesc, bdesc, IDESC, (b > it.blo || kc > 0 || ks > 0) ? 1u : 0u);
                        }
                        mma_commit(empty_bar(s));
                    }
                }
                if (!ok) break;
                if (it.bhi > it.blo) mma_commit(tfull_bar(buf));  // arrives when this item's MMAs have completed
                else mbar_arrive(tfull_bar(buf));
            }
            s_consumed = g;
        }
    } else {
        // ---------------- epilogue warps 0..3: TMEM lane quarter = warp -> 32 output columns
        for (int i = 0; work_item<TAIL>(i, G, full, tail, ntq, brp, nnzb, false, it); ++i) {
            const int buf = i & 1;
            const uint32_t use = static_cast<uint32_t>(i >> 1);
            const int I = it.I, n0 = (it.t % ntq) * 128;
            const bool empty = it.bhi == it.blo;
            int ok = 1;
            if (lane == 0) ok = (mbar_wait(tfull_bar(buf), use & 1u, spin_limit) && !s_abort) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    record_error(kErrAcc);
                    s_abort = 1;
                }
                break;
            }
            tc_fence_after();
            // a tail piece adds into what the first launch stored: wait until that launch has finished
            if (TAIL) asm volatile("griddepcontrol.wait;" ::: "memory");
            const int cn = n0 + 32 * warp + lane;  // this thread's column; columns >= N are not stored
            const bool cok = cn < N;
            const int mrows = min(BR, M - I * BR);  // rows of this block-row inside [0, M)
            float* cp = C + static_cast<long long>(I) * BR * ldc + cn;
            if (empty) {
                // nothing to add (a tail piece), or C = 0 * A B + beta C (a whole tile or a head piece)
                if (!TAIL && cok)
                    for (int r = 0; r < mrows; ++r) __stcs(cp + r * ldc, beta != 0.f ? beta * cp[r * ldc] : 0.f);
            } else {
                // GUARD: a tile on a ragged edge (row M or column N inside it) checks each store
                auto drain = [&](auto guard) {
                    constexpr bool GUARD = decltype(guard)::value;
#pragma unroll 1
                    for (int c0 = 0; c0 < BR; c0 += 16) {  // 16 rows at a time: few live registers
                        uint32_t v[16];
                        tmem_ld16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + buf * PITCH + c0, v);
                        // old values (a tail piece, or beta != 0): all 16 loaded before any store, so no load
                        // waits on the store before it
                        float old[16];
                        if (TAIL || beta != 0.f) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                old[j] = (!GUARD || (cok && c0 + j < mrows)) ? cp[static_cast<long long>(c0 + j) * ldc] : 0.f;
                        }
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            if (!GUARD || (cok && c0 + j < mrows)) {
                                float* q = cp + static_cast<long long>(c0 + j) * ldc;
                                const float acc = alpha * __uint_as_float(v[j]);
                                // a tail piece: the head piece's alpha A B + beta C, plus this piece
                                __stcs(q, TAIL ? old[j] + acc : (beta != 0.f ? acc + beta * old[j] : acc));
                            }
                        }
                    }
                };
                if (n0 + 128 <= N && mrows == BR) drain(std::false_type{});
                else drain(std::true_type{});
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
        if (warp == 4 && lane == 0) {
            // copies issued but never consumed: wait (bounded) until each has landed
            for (uint32_t g = s_consumed; g < s_issued; ++g)
                if (!mbar_wait(full_bar(g % STAGES), (g / STAGES) & 1u, spin_limit)) {
                    record_error(kErrDrain);
                    break;
                }
        } else if (warp == 5 && lane == 0) {
            // MMAs in flight: one more commit, then wait (bounded) for it
            mma_commit(fin_bar);
            if (!mbar_wait(fin_bar, 0, spin_limit)) record_error(kErrDrain);
        }
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 5)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TCOLS) : "memory");
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

// Dynamic shared memory of the persistent kernel for a stage of `sb` bytes:
// the ring, 1 KB alignment slack, the barriers.
constexpr size_t persist_smem(uint32_t sb) { return STAGES * static_cast<size_t>(sb) + 1024 + 256; }
constexpr size_t kPersistSmemMax = persist_smem(kBlk * 2 * 128 + 2 * kBBox);  // 128-row blocks

// CTAs of the persistent kernel that the SMs of the current device hold at
// once, from the shared-memory, thread, register and tensor-memory limits
// with the whole L1/shared array as shared memory, for a stage of `sb` bytes
// and `cols` TMEM columns per CTA (64 x 64 blocks: three per SM).  The
// kernels' attributes are set and each count worked out once per device.
long long persist_resident(uint32_t sb, uint32_t cols) {
    static std::mutex mu;
    static std::map<std::pair<int, uint64_t>, long long> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    const auto key = std::make_pair(dev, (static_cast<uint64_t>(sb) << 32) | cols);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int nsm = 0, smem_sm = 0, reserved = 0, max_thr = 0, regs_sm = 0;
    int regs = 1;
    size_t static_smem = 0;
    for (auto* k : {bsr_spmm_persist_kernel<false, false>, bsr_spmm_persist_kernel<true, false>,
                    bsr_spmm_persist_kernel<false, true>, bsr_spmm_persist_kernel<true, true>}) {
        cudaFuncAttributes fa{};
        if (set_smem_limit(k, kPersistSmemMax) != cudaSuccess ||
            cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
                cudaSuccess ||
            cudaFuncGetAttributes(&fa, k) != cudaSuccess)
            return -1;
        regs = std::max(regs, fa.numRegs);
        static_smem = std::max(static_smem, fa.sharedSizeBytes);
    }
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_thr, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess)
        return -1;
    const long long per_block = static_cast<long long>(persist_smem(sb) + static_smem) + reserved;
    long long per_sm = smem_sm / per_block;
    per_sm = std::min<long long>(per_sm, max_thr / kPThreads);
    per_sm = std::min<long long>(per_sm, regs_sm / (static_cast<long long>(regs) * kPThreads));
    per_sm = std::min<long long>(per_sm, 512 / cols);  // the SM's 512 TMEM columns
    const long long G = std::max<long long>(per_sm, 1) * nsm;
    cache[key] = G;
    return G;
}

template <bool GEN>
spx_status launch_persist(const CUtensorMap& tmA, const CUtensorMap& tmB, const int* brp, const int* bcol, float* C,
                          long long ldc, float alpha, float beta, int M, int N, int K, long long nnzb, int ntiles,
                          int ntq, const TcShape& sh, cudaStream_t st, uint64_t* launches) {
    const long long G = persist_resident(GEN ? sh.sb : kSB, GEN ? sh.cols : kPTmemCols);  // CTAs held at once
    if (G <= 0) return SPX_ERR_CUDA;
    const size_t smem = persist_smem(GEN ? sh.sb : kSB);
    // The last round of tiles: with at most half the CTAs busy in it, its tiles are cut in two.  The first
    // launch stores each such tile's head piece (its first half of the blocks) beside the whole tiles; a
    // second launch of as many CTAs computes the tail pieces on the SMs the first launch frees and adds them
    // into C once the first has finished.  Every tile is then done after about ntiles / G rounds, not
    // ceil(ntiles / G).  A piece pays a CTA start-up and a pipeline fill of its own, so block-rows of fewer
    // than kSplitBlocks ring stages on average are not cut (64 x 64 blocks, 256 block-rows, N = 1024, the
    // whole tiles against the cut last round: 26 blocks 76.4 / 78.5 us, 52 blocks 133.8 / 130.7, 104 blocks
    // 250.5 / 237.2, 256 blocks 582.3 / 537.2).
    constexpr long long kSplitBlocks = 48;
    const int R = static_cast<int>(ntiles % G);
    const int br = GEN ? sh.br : kBlk, kc = GEN ? sh.kc : 1;
    const long long MB = (M + br - 1) / br;
    const bool split = R > 0 && 2LL * R <= G && nnzb * kc >= kSplitBlocks * MB;
    const int full = split ? ntiles - R : ntiles, tail = split ? R : 0;
    const int grid = static_cast<int>(split ? (full > 0 ? G : R) : std::min<long long>(ntiles, G));
    const int KB = (K + (GEN ? sh.bc : kBlk) - 1) / (GEN ? sh.bc : kBlk);
    bsr_spmm_persist_kernel<false, GEN><<<grid, kPThreads, smem, st>>>(tmA, tmB, brp, bcol, C, ldc, alpha, beta,
                                                                       kSpinLimit, M, N, full, tail, ntq, KB, nnzb,
                                                                       sh);
    *launches = 1;
    if (!split) return spx_cuda_status(cudaGetLastError());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(R));
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the first launch ends
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, bsr_spmm_persist_kernel<true, GEN>, tmA, tmB, brp, bcol, C, ldc,
                                             alpha, beta, kSpinLimit, M, N, full, tail, ntq, KB, nnzb, sh);
    *launches = 2;
    return spx_cuda_status(e != cudaSuccess ? e : cudaGetLastError());
}

// 2-D bf16 tensor map with a box of box_inner x box_outer elements, 128-byte swizzle.
bool make_map_box(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_bytes,
                  uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

spx_status spx_spmm_bsr(int32_t M, int32_t K, int32_t br, int32_t bc, int64_t nnzb, const int32_t* bsr_row_ptr,
                        const int32_t* bsr_col, const uint16_t* bsr_val, int32_t N, const uint16_t* B, int64_t ldb,
                        float alpha, float beta, float* C, int64_t ldc, spx_stream_t stream) {
    if (M < 0 || K < 0 || N < 0 || nnzb < 0 || br <= 0 || bc <= 0) return SPX_ERR_ARG;
    // 64 x 64 blocks: the tensor-core kernel, which needs its alignment; other shapes whose sides are
    // multiples of 16 (tc_general_shape): the same kernel when the arrays are aligned for it, else, and for
    // every other shape, bsr_spmm_simt_kernel
    const bool tc64 = br == kBlk && bc == kBlk;
    const bool tc_aligned = ldb % 8 == 0 && spx_aligned(bsr_val, 16) && spx_aligned(B, 16);
    const bool tcg = !tc64 && tc_general_shape(br, bc) && tc_aligned;
    if (nnzb > kI32Max || static_cast<int64_t>(nnzb) * std::max(br, bc) > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (M == 0 || N == 0) return SPX_OK;
    if (!bsr_row_ptr || !C || (nnzb > 0 && (!bsr_col || !bsr_val || !B))) return SPX_ERR_ARG;
    if (ldb < N || ldc < N) return SPX_ERR_ARG;
    if (tc64 && (!tc_aligned || !spx_aligned(C, 4) || !spx_aligned(bsr_row_ptr, 4) || !spx_aligned(bsr_col, 4)))
        return SPX_ERR_ALIGN;
    if (!tc64 && (ldb % 2 || !spx_aligned(bsr_val, 2) || !spx_aligned(B, 4) || !spx_aligned(C, 4) ||
                  !spx_aligned(bsr_row_ptr, 4) || !spx_aligned(bsr_col, 4)))
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
    // A as nnzb * br rows of bc columns, read in 64-column boxes (past bc: zero-filled); B in boxes of
    // min(bc, 64) rows
    const bool mapped =
        (tc64 || tcg) &&
        make_map_box(&tmA, bsr_val, static_cast<uint64_t>(bc), static_cast<uint64_t>(nnzb) * br,
                     static_cast<uint64_t>(bc) * 2, kBlk, static_cast<uint32_t>(br)) &&
        make_map_box(&tmB, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K), static_cast<uint64_t>(ldb) * 2,
                     64, static_cast<uint32_t>(std::min(bc, kBlk)));
    if (tc64 && !mapped) return SPX_ERR_CUDA;
    if (!mapped)
        return spx_bsr_simt_spmm(M, K, br, bc, nnzb, bsr_row_ptr, bsr_col, bsr_val, N, B, ldb, alpha, beta, C, ldc,
                                 st);
    const long long ntiles = static_cast<long long>((M + br - 1) / br) * ((N + 127) / 128);
    if (ntiles > kI32Max) return SPX_ERR_INDEX_RANGE;
    uint64_t launches = 0;
    const TcShape sh = tc_shape(br, bc);
    const spx_status s =
        tc64 ? launch_persist<false>(tmA, tmB, bsr_row_ptr, bsr_col, C, ldc, alpha, beta, M, N, K, nnzb,
                                     static_cast<int>(ntiles), (N + 127) / 128, sh, st, &launches)
             : launch_persist<true>(tmA, tmB, bsr_row_ptr, bsr_col, C, ldc, alpha, beta, M, N, K, nnzb,
                                    static_cast<int>(ntiles), (N + 127) / 128, sh, st, &launches);
    spx_note_launches(launches);
    return s;
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
    // Pieces of unequal length: one CTA per (task, column tile), so the hardware hands the next task to
    // whichever CTA slot frees first (the persistent kernel's static schedule balanced them worse:
    // 160 against 123 us on block-rows of 26 and of 208 blocks)
    if (set_smem_limit(bsr_spmm_tile_kernel, kTileSmem) != cudaSuccess) return SPX_ERR_CUDA;
    bsr_spmm_tile_kernel<<<dim3((N + 127) / 128, static_cast<unsigned>(ntasks)), kTThreads, kTileSmem, st>>>(
        tmA, tmB, bsr_col, C, ldc, alpha, beta, kSpinLimit, M, N, tasks, partials, (K + kBlk - 1) / kBlk);
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
    // the checked build's index errors (always 0 in the product build, which reads no word for them)
    const int checked[] = {spx_check_take(g_bsr_check), spx_spmv_check_take(), spx_spmm_check_take(),
                           spx_sell_check_take(), spx_wcsr_check_take(), spx_bsrg_check_take()};
    if (h || wcsr == SPX_ERR_TIMEOUT) return SPX_ERR_TIMEOUT;
    if (wcsr == SPX_ERR_CUDA) return SPX_ERR_CUDA;
    for (int c : checked)
        if (c == SPX_ERR_CUDA) return SPX_ERR_CUDA;
    if (coo) return static_cast<spx_status>(coo);
    for (int c : checked)
        if (c) return static_cast<spx_status>(c);
    return SPX_OK;
}

}  // extern "C"
