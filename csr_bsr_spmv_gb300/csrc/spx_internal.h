// Internal declarations shared by the host and device translation units of libspx.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "spx.h"

#ifdef __CUDACC__
#define SPX_HD __host__ __device__
#else
#define SPX_HD
#endif

// One term of a row_ptr's structure fingerprint: SplitMix64's output function
// (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
// OOPSLA 2014) of the state 2^32 * i + (uint32) row_ptr[i].  The fingerprint
// is the sum of the terms mod 2^64, so any summation order gives the same value.
inline SPX_HD uint64_t spx_fp_term(uint64_t i, int32_t v) {
    uint64_t z = ((i << 32) | static_cast<uint32_t>(v)) + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Fingerprint of a device row_ptr[0..M] (one launch; synchronises st).
spx_status spx_dev_rp_fingerprint(int32_t M, const int32_t* row_ptr, uint64_t* out, cudaStream_t st);

// Counts kernel launches (reported by spx_launch_count).
void spx_note_launches(uint64_t n);

// Status of the last CUDA runtime error, or SPX_OK.
spx_status spx_cuda_status(int cuda_error);

// Reads and clears the error word of the COO kernel: 0 or a negative spx_status.
int spx_coo_error_take();

// Reads and clears the error word of the WCSR kernel: 0 or SPX_ERR_TIMEOUT.
int spx_wcsr_error_take();

// The checked build (-DSPX_CHECK): read and clear the index-error word of each
// translation unit's kernels, 0 or SPX_ERR_INDEX_RANGE (0 without reading
// anything in the product build).
int spx_spmv_check_take();
int spx_spmm_check_take();
int spx_sell_check_take();
int spx_wcsr_check_take();
int spx_bsrg_check_take();

// BSR SpMM for block shapes other than 64 x 64 (spx_bsr_simt.cu): the
// arguments of spx_spmm_bsr, validated by it (ldb even; bsr_val 2-, B and C
// 4-byte aligned); nnzb > 0, M > 0, N > 0.
spx_status spx_bsr_simt_spmm(int32_t M, int32_t K, int32_t br, int32_t bc, int64_t nnzb, const int32_t* bsr_row_ptr,
                             const int32_t* bsr_col, const uint16_t* bsr_val, int32_t N, const uint16_t* B,
                             int64_t ldb, float alpha, float beta, float* C, int64_t ldc, cudaStream_t st);

// Device-side builders (spx_build.cu): stable radix sorts on the GPU, results
// identical to the host builders.  Stream-ordered; temporary memory from the
// stream-ordered allocator.
spx_status spx_dev_build_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* coo_row, const int32_t* coo_col,
                             const void* coo_val, int32_t val_bytes, int32_t* row_ptr, int32_t* col, void* val,
                             spx_stream_t stream);
spx_status spx_dev_transpose_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                                 const void* val, int32_t val_bytes, int32_t* t_row_ptr, int32_t* t_col, void* t_val,
                                 spx_stream_t stream);
// CSR -> BSR on the device (same two-call protocol and results as the host builder).
spx_status spx_dev_build_bsr(int32_t M, int32_t K, const int32_t* row_ptr, const int32_t* col, const void* val,
                             int32_t vb, int32_t br, int32_t bc, int32_t* bsr_row_ptr, int32_t* bsr_col,
                             void* bsr_val, int64_t* nnzb_out, double* fill_out, cudaStream_t st);
// CSR -> WCSR on the device (same two-call protocol and results as the host builder).
spx_status spx_dev_build_wcsr(int32_t M, int32_t K, const int32_t* row_ptr, const int32_t* col, const void* val,
                              int32_t vb, int32_t* win_ptr, int32_t* win_col, void* win_val, int64_t* nchunks_out,
                              double* fill_out, cudaStream_t st);
// SELL-C-sigma image built on the GPU (layout of spx_sell.cu): `image` is
// device memory from cudaMalloc that the caller of spx_dev_build_sell owns.
struct spx_sell_dev_image {
    void* image = nullptr;
    size_t bytes = 0, off_prow = 0, off_long = 0, off_col = 0, off_val = 0;
    int64_t nslices = 0, pseudo_rows = 0, padded = 0, nlong = 0, slots = 0;
};
spx_status spx_dev_build_sell(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                              const float* val, int32_t sigma, int32_t piece, spx_sell_dev_image* out,
                              cudaStream_t st);
// Row statistics of a device row_ptr (lengths, sums and extremes in one
// kernel, percentiles from a radix sort of the lengths); synchronous.
spx_status spx_dev_row_stats(int32_t M, const int32_t* row_ptr, spx_row_stats_t* out, cudaStream_t st);
// mean, variance and cv from out->nnz and out->sumsq (shared by both paths).
void spx_row_stats_finish(int32_t M, spx_row_stats_t* out);

struct spx_plan {
    int32_t M = 0, K = 0;
    int64_t nnz = 0;
    spx_plan_opts_t opts{};
    std::vector<int32_t> tasks;     // 4 per task, the documented (host) form
    std::vector<int32_t> dtasks;    // 4 per task, the device form (see spx_spmv.cu)
    std::vector<int32_t> longrows;  // 4 per split row
    std::vector<uint16_t> first;    // segmented groups: spx_group_threads entries per group (see below)
    int64_t counts[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    spx_row_stats_t stats{};
    const void* d_table = nullptr;  // caller-owned copy of dtasks, longrows, first
    size_t table_bytes = 0;
    size_t scratch_bytes = 0;
    uint64_t fingerprint = 0;       // of the row_ptr the plan was built from
    uint64_t magic = 0;
};

// Plan on the GPU from a device row_ptr: spx_dev_check_rp validates it (the
// host checks' codes), spx_dev_make_plan fills P's tasks, device tasks, split
// rows and counts exactly as the host builder does (P->opts set).  Synchronous.
spx_status spx_dev_check_rp(int32_t M, int64_t nnz, const int32_t* row_ptr, cudaStream_t st);
spx_status spx_dev_make_plan(spx_plan* P, const int32_t* row_ptr, cudaStream_t st);

// Task split of 64-row units (WCSR windows, BSR block-rows): units with more
// than max_chunks chunks (blocks) are cut into pieces with partial-tile slots.
struct spx_wcsr_plan {
    int32_t M = 0;
    int64_t nchunks = 0;  // chunks (WCSR) or blocks (BSR) in all
    int32_t max_chunks = 0;
    std::vector<int32_t> tasks;   // 4 per task: unit, first chunk, chunks, partial slot (-1: the whole unit)
    std::vector<int32_t> splits;  // 4 per split unit: unit, first slot, pieces, 0
    int64_t slots = 0;
    size_t table_bytes = 0;
    const void* d_table = nullptr;  // caller-owned copy: tasks, then splits
    uint64_t magic = 0;
};
constexpr uint64_t kWcsrPlanMagic = 0x5350585f57504c4eull;  // "SPX_WPLN"

constexpr uint64_t kPlanMagic = 0x5350585f504c414eull;  // "SPX_PLAN"

enum : int32_t { kTaskGroup = 0, kTaskCta = 1, kTaskSeg = 2 };
constexpr int32_t kReduceSegmented = 6;  // group reduction code of the segmented reduction

// A packed group runs on spx_group_threads(B) threads, thread t owning the
// products [t * P, t * P + P) of the group (P = spx_group_per(B)) in the
// segmented reduction.  B = 512 / 1024 / 2048 / 4096 run B / 8 threads with
// eight products each; other sizes run 256 threads.
inline SPX_HD int32_t spx_group_threads(int32_t B) {
    return (B == 512 || B == 1024 || B == 2048 || B == 4096) ? B / 8 : 256;
}
inline SPX_HD int32_t spx_group_per(int32_t B) {
    const int32_t nt = spx_group_threads(B);
    return (B + nt - 1) / nt;
}
// Entry `first` of a segmented group's thread t (relative rows r of the
// group, products counted from the group's first): the row holding product
// a = t * P -- the last r with start(r) <= a -- shifted left once, plus 1 when
// that row starts before a (its first products belong to earlier threads);
// 0 for a thread past the group's products.  The plan stores the entries of
// all groups (in task order) after the split-row table when lanes_div == 0.
inline SPX_HD uint16_t spx_first_entry(int32_t r, bool starts_before) {
    return static_cast<uint16_t>((r << 1) | (starts_before ? 1 : 0));
}

// Device task (int4): x = kind | code << 2 | aux << 8 where aux = #rows for a
// group and the partial-sum slot for a segment; y = first row; z, w = the
// nonzero range [p0, p1) the task covers.
inline void spx_dev_task(int32_t* d, int32_t kind, int32_t code, int32_t aux, int32_t row, int32_t p0, int32_t p1) {
    d[0] = kind | (code << 2) | (aux << 8);
    d[1] = row;
    d[2] = p0;
    d[3] = p1;
}

inline bool spx_plan_ok(const spx_plan* p) { return p && p->magic == kPlanMagic; }

inline bool spx_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t kI32Max = 2147483647LL;
