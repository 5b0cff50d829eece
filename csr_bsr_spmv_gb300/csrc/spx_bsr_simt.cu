// spx_bsr_simt.cu -- BSR SpMM C = alpha*A*B + beta*C for block shapes other
// than 64 x 64 (any br x bc), bf16 blocks and B, fp32 accumulation, on the
// CUDA cores.
//
// [Formats] (block sparse) and [AsyncSparse] §2.2.1 define BSR for any
// br x bc block; [SpMM-ops] §3.4 gives the product: for every stored block of
// a block-row, a small dense product of the block with the B rows of its
// block column.  The 64 x 64 shape runs on the tensor cores (spx_bsr.cu);
// this kernel takes every other shape, where the block is too small or too
// oddly sized for a 128 x N x 16 MMA to pay.
//
// A block-row's blocks, taken in order, form one long reduction axis of
// nb * bc terms: term g is column g % bc of block g / bc.  A CTA owns up to
// 64 rows of one block-row and a strip of output columns; it walks that axis
// in chunks of kQ terms:
//   - a table of the chunk's terms (offset of the term's column in its block,
//     the B row it multiplies, or -1 past K) is built by kQ threads;
//   - the A columns (rows x kQ, as fp32) and the B rows (kQ x strip, as bf16
//     pairs) are staged in shared memory, both with consecutive threads on
//     consecutive addresses;
//   - warp w of the CTA owns 8 rows and 64 columns (two per lane): each lane
//     reads its B pair (consecutive across the warp) and the 8 rows' A values
//     (one broadcast 16-byte read per row and 4 terms), and accumulates the
//     terms in order with fused multiply-adds.
// Small blocks leave rows idle in a 64-row CTA, so the CTA trades row warps
// for column warps: WR = ceil(rows / 8) warps over the rows and 8 / WR over
// the columns (a strip of 64 * 8 / WR columns).
//
// Every element's sum runs over the block-row's terms in their stored order,
// so the result is the same from run to run.  B rows at or past K read as
// zeros, C is written only inside M x N.
#include <cuda_runtime.h>

#include <cstdint>

#include "spx_check.cuh"
#include "spx_internal.h"

namespace {

constexpr int kQ = 32;         // terms per staged chunk
constexpr int kRowsCta = 64;   // rows of a block-row per CTA
constexpr int kWarps = 8;      // warps per CTA (row warps x column warps)

SPX_CHECK_WORD(g_bsrg_check)

__device__ __forceinline__ float bf16_bits(uint32_t h) { return __uint_as_float(h << 16); }

// Dynamic shared memory: As[WR*8][kQ] fp32, Bs[kQ][32*WN] bf16 pairs, then the term table.
__global__ void __launch_bounds__(kWarps * 32) bsr_spmm_simt_kernel(
    const int* __restrict__ brp, const int* __restrict__ bcol, const uint16_t* __restrict__ bval,
    const uint16_t* __restrict__ B, long long ldb, float* C, long long ldc, float alpha, float beta, int M, int K,
    int N, int br, int bc, int nnzb, int rch, int ntn, int WR) {
    extern __shared__ __align__(16) float smem[];
    const int WN = kWarps / WR;
    float* As = smem;                                                     // [WR*8][kQ]
    uint32_t* Bs = reinterpret_cast<uint32_t*>(As + WR * 8 * kQ);         // [kQ][32*WN]
    long long* s_aoff = reinterpret_cast<long long*>(Bs + kQ * 32 * WN);  // [kQ]
    int* s_brow = reinterpret_cast<int*>(s_aoff + kQ);                    // [kQ]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wr = warp % WR, wn = warp / WR;
    const long long unit = blockIdx.x / ntn;
    const int tile = static_cast<int>(blockIdx.x - unit * ntn);
    const int I = static_cast<int>(unit / rch);
    const int rbase = static_cast<int>(unit - static_cast<long long>(I) * rch) * kRowsCta;
    const int rows = min(kRowsCta, br - rbase);  // rows of this CTA inside the block
    const int n0 = tile * 64 * WN;
    const int KB = (K + bc - 1) / bc;

    int b0 = brp[I], b1 = brp[I + 1];
    if (SPX_CHECKED && (b0 < 0 || b1 < b0 || b1 > nnzb)) {
        if (tid == 0) check_fail();
        b0 = b1 = 0;  // the block-row counts as empty
    }
    const int total = (b1 - b0) * bc;
    const long long blk_elems = static_cast<long long>(br) * bc;

    float acc[8][2];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = 0.f;

    for (int q0 = 0; q0 < total; q0 += kQ) {
        const int qn = min(kQ, total - q0);
        __syncthreads();  // the previous chunk's reads are done
        for (int q = tid; q < kQ; q += kWarps * 32) {
            long long aoff = -1;
            int brow = -1;
            if (q < qn) {
                const int g = q0 + q, j = g / bc, c = g - j * bc, blk = b0 + j;
                int J = bcol[blk];
                if (SPX_CHECKED && (J < 0 || J >= KB)) {
                    check_fail();
                    J = -1;
                }
                aoff = static_cast<long long>(blk) * blk_elems + c;
                const long long r = static_cast<long long>(J) * bc + c;
                brow = (J >= 0 && r < K) ? static_cast<int>(r) : -1;
            }
            s_aoff[q] = aoff;
            s_brow[q] = brow;
        }
        __syncthreads();
        for (int e = tid; e < WR * 8 * kQ; e += kWarps * 32) {
            const int r = e / kQ, q = e - r * kQ;
            const long long aoff = s_aoff[q];
            As[e] = (r < rows && aoff >= 0)
                        ? bf16_bits(bval[aoff + static_cast<long long>(rbase + r) * bc])
                        : 0.f;
        }
        for (int e = tid; e < kQ * 32 * WN; e += kWarps * 32) {
            const int q = e / (32 * WN), t = e - q * (32 * WN);
            const int brow = s_brow[q];
            const int n = n0 + 2 * t;
            uint32_t v = 0;
            if (brow >= 0 && n < N) {
                const uint16_t* p = B + static_cast<long long>(brow) * ldb + n;
                v = (n + 1 < N) ? __ldg(reinterpret_cast<const unsigned int*>(p)) : static_cast<uint32_t>(__ldg(p));
            }
            Bs[e] = v;
        }
        __syncthreads();
        const float* a_row = As + (wr * 8) * kQ;
        const uint32_t* b_col = Bs + wn * 32 + lane;
#pragma unroll 2
        for (int q = 0; q < kQ; q += 4) {
            float bx[4], by[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t w = b_col[(q + j) * 32 * WN];
                bx[j] = bf16_bits(w & 0xffffu);
                by[j] = bf16_bits(w >> 16);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 a = *reinterpret_cast<const float4*>(a_row + i * kQ + q);
                acc[i][0] = fmaf(a.x, bx[0], acc[i][0]);
                acc[i][1] = fmaf(a.x, by[0], acc[i][1]);
                acc[i][0] = fmaf(a.y, bx[1], acc[i][0]);
                acc[i][1] = fmaf(a.y, by[1], acc[i][1]);
                acc[i][0] = fmaf(a.z, bx[2], acc[i][0]);
                acc[i][1] = fmaf(a.z, by[2], acc[i][1]);
                acc[i][0] = fmaf(a.w, bx[3], acc[i][0]);
                acc[i][1] = fmaf(a.w, by[3], acc[i][1]);
            }
        }
    }

    const int n = n0 + wn * 64 + 2 * lane;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = wr * 8 + i;
        const long long row = static_cast<long long>(I) * br + rbase + r;
        if (r >= rows || row >= M) continue;
        float* q = C + row * ldc;
#pragma unroll
        for (int j = 0; j < 2; ++j)
            if (n + j < N) q[n + j] = beta != 0.f ? alpha * acc[i][j] + beta * q[n + j] : alpha * acc[i][j];
    }
}

}  // namespace

int spx_bsrg_check_take() { return spx_check_take(g_bsrg_check); }

spx_status spx_bsr_simt_spmm(int32_t M, int32_t K, int32_t br, int32_t bc, int64_t nnzb, const int32_t* bsr_row_ptr,
                             const int32_t* bsr_col, const uint16_t* bsr_val, int32_t N, const uint16_t* B,
                             int64_t ldb, float alpha, float beta, float* C, int64_t ldc, cudaStream_t st) {
    const int rows_cta = br < kRowsCta ? br : kRowsCta;
    const int WR = rows_cta <= 8 ? 1 : rows_cta <= 16 ? 2 : rows_cta <= 32 ? 4 : 8;
    const int WN = kWarps / WR;
    const long long MB = (static_cast<long long>(M) + br - 1) / br;
    const int rch = (br + kRowsCta - 1) / kRowsCta;
    const int ntn = (N + 64 * WN - 1) / (64 * WN);
    const long long grid = MB * rch * ntn;
    if (grid > kI32Max) return SPX_ERR_INDEX_RANGE;
    const size_t smem = sizeof(float) * WR * 8 * kQ + sizeof(uint32_t) * kQ * 32 * WN +
                        (sizeof(long long) + sizeof(int)) * kQ;
    bsr_spmm_simt_kernel<<<static_cast<unsigned>(grid), kWarps * 32, smem, st>>>(
        bsr_row_ptr, bsr_col, bsr_val, B, ldb, C, ldc, alpha, beta, M, K, N, br, bc, static_cast<int>(nnzb), rch,
        ntn, WR);
    spx_note_launches(1);
    return spx_cuda_status(cudaGetLastError());
}
