/*
 * spx.h -- C ABI of libspx: sparse x dense products on one GB300 (sm_103a).
 *
 * Operations (page titles as cited throughout this library):
 *   [SpMM-ops]    "通用稀疏矩阵乘法CUDA算子实现" (chengzipai.xyz)
 *   [BCSR-SpMV]   "GPU加速实战用BCSR格式优化稀疏矩阵乘法附CUDA代码" (xxqk.cn)
 *   [AsyncSparse] AsyncSparse summary, "异步GPU架构下的稀疏矩阵乘法加速" (capital-peak.com)
 *   [LSMR-dual]   "CUDA LSMR 专栏（二）：用 CSR/CSC 双存储压榨双向 SpMV" (chengzipai.xyz)
 *   [Formats]     "稀疏矩阵存储格式:COO、CSR、ELL、Hybrid 与块稀疏" (geek-doc.cn)
 *
 * Conventions for every call:
 *   - The caller owns every array.  The library allocates no device memory on
 *     the compute calls; sizes of the extra device buffers a call needs (the
 *     plan table, the scratch for long-row partial sums) are reported by the
 *     plan so the caller can allocate them once.
 *   - Indices are 0-based int32.  Any size or index that does not fit int32
 *     (M, K, nnz, nnz of a block pattern) is rejected with
 *     SPX_ERR_INDEX_RANGE, never truncated ([LSMR-dual] §8).
 *   - Device work is enqueued on `stream` (NULL = the legacy default stream)
 *     and the call returns after enqueueing; results are ready when the
 *     stream reaches that point.  Host-side builders finish before return.
 *   - beta == 0 means the output is write-only: it is not read, so NaN/Inf
 *     already in it do not propagate.
 *   - No call aborts; every failure is a negative spx_status and, for a
 *     rejected argument, nothing is launched.
 *   - Calls may come from several host threads at once.  Plans, SELL forms
 *     and task splits are read-only once built and uploaded, so calls on any
 *     stream may share them.  A scratch buffer is written by the call that
 *     gets it: calls that can overlap on the GPU (different streams with no
 *     ordering between them) each need their own, while calls ordered on one
 *     stream may share one.
 */
#ifndef SPX_H_
#define SPX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* spx_stream_t; /* same type as cudaStream_t */

typedef enum spx_status {
    SPX_OK = 0,
    SPX_ERR_ARG = -1,          /* null pointer, negative size, bad option, plan mismatch */
    SPX_ERR_INDEX_RANGE = -2,  /* size/index beyond int32, or an index outside [0, dim) */
    SPX_ERR_NOT_SORTED = -3,   /* row_ptr not monotone / columns not ascending where required */
    SPX_ERR_DUPLICATE = -4,    /* a repeated (row, col) where one value slot exists */
    SPX_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed */
    SPX_ERR_TIMEOUT = -6,      /* a bounded device wait gave up (see spx_last_device_error) */
    SPX_ERR_UNSUPPORTED = -7,  /* shape/type combination this build has no kernel for */
    SPX_ERR_ALIGN = -8,        /* pointer or leading dimension not aligned as documented */
    SPX_ERR_NOMEM = -9,        /* host allocation failed */
    SPX_ERR_NOT_READY = -10,   /* plan used before spx_plan_upload (or see spx_spmv_csr_noalloc) */
    SPX_ERR_SCRATCH_LIMIT = -11 /* needs more scratch than the library's fixed buffer holds */
} spx_status;

typedef enum spx_loc {
    SPX_HOST = 0,   /* all array arguments of the call are host pointers   */
    SPX_DEVICE = 1  /* all array arguments of the call are device pointers */
} spx_loc;

/* Human-readable name of a status code (static string). */
const char* spx_status_string(spx_status s);

/* Number of kernel launches this library has issued since load. */
spx_status spx_launch_count(uint64_t* count);

/* ------------------------------------------------------------ format builders */

/*
 * COO -> CSR.  [Formats] §3: count entries per row (histogram), exclusive
 * prefix sum -> row_ptr[M+1], then move col/val into each row's range;
 * [SpMM-ops] §1.2: entries end sorted by (row, col).  Entries with equal
 * (row, col) are kept (not summed), in input order.
 *   coo_row, coo_col, coo_val: nnz entries in any order; coo_val holds
 *     val_bytes bytes per entry (2, 4 or 8; values are moved, not read).
 *   row_ptr[M+1], col[nnz], val[nnz*val_bytes]: outputs.
 * Errors: SPX_ERR_INDEX_RANGE for a row outside [0, M) or col outside [0, K).
 * where == SPX_HOST: a counting sort on the host.  where == SPX_DEVICE: the
 * arrays are device memory and the build runs on the GPU (a stable LSD radix
 * sort by column, then by row, with 8-bit digits; exact per-row counts and a
 * scan give row_ptr): same result, bit for bit.  The device build validates
 * the indices first (one synchronisation of `stream`), then enqueues the rest
 * on `stream`; its temporary memory (about 16 bytes per entry) comes from the
 * stream-ordered allocator and is released on `stream`.
 */
spx_status spx_build_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* coo_row, const int32_t* coo_col,
                         const void* coo_val, int32_t val_bytes, int32_t* row_ptr, int32_t* col, void* val,
                         spx_loc where, spx_stream_t stream);

/*
 * CSR(A) (M x K) -> CSR(A^T) (K x M), which is CSC(A): [LSMR-dual] §2 (CSC(A)
 * has exactly the memory layout of CSR(A^T)) and §4 (build it once, at
 * construction).  Output row j holds the entries of column j in increasing
 * source row order (a stable counting sort by column).
 *   t_row_ptr[K+1], t_col[nnz], t_val[nnz*val_bytes]: outputs.
 * Errors: SPX_ERR_ARG if row_ptr[0] != 0 or row_ptr[M] != nnz;
 * SPX_ERR_INDEX_RANGE for a column outside [0, K); SPX_ERR_NOT_SORTED when
 * row_ptr decreases.  where == SPX_DEVICE: built on the GPU by a stable radix
 * sort of the entries by column (validation synchronises `stream` once; the
 * rest is stream-ordered, temporary memory from the stream-ordered allocator).
 */
spx_status spx_transpose_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                             const void* val, int32_t val_bytes, int32_t* t_row_ptr, int32_t* t_col, void* t_val,
                             spx_loc where, spx_stream_t stream);

/*
 * CSR -> BSR with br x bc blocks.  [AsyncSparse] §2.2.1 (store each block
 * holding at least one entry, dense and contiguous; block_row_ptr,
 * block_col_idx; fill_ratio = nnz / (nnz_blocks * br * bc)); [BCSR-SpMV] §1
 * (one block-column index per block).  Blocks are row-major inside; block
 * columns ascend within a block-row; a last partial block-row/column is
 * zero-padded (logical M, K unchanged).
 * Two calls: with bsr_col == NULL and bsr_val == NULL the call only fills
 * *nnzb_out, *fill_out and (if non-NULL) bsr_row_ptr[ceil(M/br)+1]; then the
 * caller allocates bsr_col[nnzb] and bsr_val[nnzb*br*bc*val_bytes].
 * Errors: SPX_ERR_ARG (row_ptr[0] != 0), SPX_ERR_NOT_SORTED (row_ptr
 * decreasing), SPX_ERR_INDEX_RANGE (a column outside [0, K), more than
 * 2^31-1 blocks), SPX_ERR_DUPLICATE for a repeated (row, col).
 * where == SPX_DEVICE builds on the GPU (device arrays in and out; stable
 * radix sort of the entries by block row, block column and place in the
 * block; temporary memory from the stream-ordered allocator) with the same
 * results as the host build; it synchronises the stream before returning and
 * returns SPX_ERR_UNSUPPORTED when br * bc exceeds 2^31-1.  With several
 * errors at once the device path reports the structural ones first.
 */
spx_status spx_build_bsr(int32_t M, int32_t K, const int32_t* row_ptr, const int32_t* col, const void* val,
                         int32_t val_bytes, int32_t br, int32_t bc, int32_t* bsr_row_ptr, int32_t* bsr_col,
                         void* bsr_val, int64_t* nnzb_out, double* fill_out, spx_loc where, spx_stream_t stream);

/*
 * Structural check of a CSR: row_ptr[0] == 0, non-decreasing, row_ptr[M] ==
 * nnz, every column in [0, K); with strict != 0 also strictly ascending
 * columns inside each row.  Returns SPX_OK, SPX_ERR_ARG, SPX_ERR_NOT_SORTED,
 * SPX_ERR_INDEX_RANGE or SPX_ERR_DUPLICATE.  The compute calls trust their
 * inputs; run this once on untrusted matrices.
 */
spx_status spx_check_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                         int32_t strict, spx_loc where, spx_stream_t stream);

/* ------------------------------------------------------------ row statistics */

typedef struct spx_row_stats_t {
    int64_t rows;    /* M */
    int64_t nnz;     /* S1 = sum of row lengths l_i */
    int64_t sumsq;   /* S2 = sum of l_i^2 */
    int32_t min, max;
    int32_t p50, p95, p99; /* nearest rank: the ceil(q*M/100)-th smallest l_i */
    int32_t empty;         /* rows with l_i == 0 */
    double mean;     /* (double)S1 / (double)M */
    double var;      /* (double)(M*S2 - S1^2) / ((double)M*(double)M), population */
    double cv;       /* sqrt(var) / mean, 0 when mean == 0 */
} spx_row_stats_t;

/*
 * Row-length statistics of a CSR.  [LSMR-dual] §5.3 (l_i = row_ptr[i+1] -
 * row_ptr[i]; mean, variance and long tail) and [SpMM-ops] §4 (avg/p95/max
 * and coefficient of variation in the dispatch key).
 * where == SPX_DEVICE computes them on the GPU: one kernel forms the lengths
 * and folds S1, S2, min, max and the empty rows with integer atomics (exact),
 * and a radix sort of the lengths gives the percentiles.  It runs on the
 * default stream, returns when done, and gives the same numbers as the host
 * path bit for bit (the doubles come from the same integer sums).
 */
spx_status spx_row_stats(int32_t M, const int32_t* row_ptr, spx_loc where, spx_row_stats_t* out);

/* ------------------------------------------------------------ dispatch plan */

typedef struct spx_plan_opts_t {
    int32_t block_nnz;  /* B: most nonzeros in a packed group (one CTA)             */
    int32_t block_rows; /* R: most rows in a packed group                           */
    int32_t pack_max;   /* P: rows with l <= P are packed into groups (P <= B)      */
    int32_t cta_max;    /* C: rows with P < l <= C get one CTA each                 */
    int32_t seg_nnz;    /* S: rows with l > C are cut into segments of S nonzeros   */
    int32_t lanes_div;  /* D >= 1: a group reduces each row with w lanes,
                           w = pow2ceil(ceil(nnz_g / (rows_g * D))) clamped to [1, 32];
                           D == 0: segmented reduction -- each thread sums an
                           equal run of consecutive products, rows crossing
                           threads are joined by a block scan */
} spx_plan_opts_t;

/* Fills the fixed defaults: B 2048, R 256, P 512, C 8192, S 4096, D 16. */
spx_status spx_plan_opts_default(spx_plan_opts_t* out);

/*
 * Options chosen from a matrix's row statistics (the "dispatch key" of
 * [SpMM-ops] §4: mean, spread and tail of the row lengths pick the mapping):
 * cv >= 2 (skewed, power-law-like lengths): B 1024 (128-thread CTAs) and the
 * segmented reduction (D 0), whose work per thread ignores row length;
 * otherwise the defaults above (256-thread CTAs, D 16 lanes-per-row rule).
 */
spx_status spx_plan_opts_auto(const spx_row_stats_t* stats, spx_plan_opts_t* out);

typedef struct spx_plan_info_t {
    int64_t M, K, nnz;
    int64_t tasks;         /* CTAs of the main launch                         */
    int64_t long_rows;     /* rows split into segments                        */
    int64_t slots;         /* partial sums (one per segment)                  */
    int64_t packed_rows, cta_rows, split_rows;
    int64_t thread_groups; /* groups reduced thread-per-row (w == 1)          */
    int64_t lane_groups;   /* groups reduced with 2..32 lanes per row         */
    int64_t segmented_groups; /* groups with the segmented reduction          */
    size_t table_bytes;    /* device bytes for spx_plan_upload (16-B aligned) */
    size_t scratch_bytes;  /* device scratch bytes each SpMV call needs       */
    spx_row_stats_t stats;
    spx_plan_opts_t opts;  /* the options the plan was built with             */
} spx_plan_info_t;

typedef struct spx_plan spx_plan; /* opaque, host-side */

/*
 * Build the dispatch plan of a CSR matrix (rows binned by length onto
 * thread/lane-group, CTA-per-row and split-row kernels).  [SpMM-ops] §2.1-§2.4
 * (thread-, warp-, CTA-per-row and segmented long rows with a second-pass
 * reduction), §4 (profile once, cache it on the descriptor) and [Formats] §6
 * (pack rows into bundles of similar work).  The rule:
 *   l <= P: packed; consecutive packed rows form groups of <= R rows and <= B
 *           nonzeros (a CTA or split row closes a group);
 *   P < l <= C: one CTA;  l > C: ceil(l/S) segments, then a fix-up pass.
 * Task table (4 int32 per task): first all CTA rows {1,row,0,0} and segments
 * {2,row,seg,slot} in row order, then groups {256*c, r0, r1, 0} where the
 * reduction code c is log2(w) (lanes per row) or 6 (segmented, D == 0).
 * Long-row table (4 int32 per split row): {row, first slot, #segments, 0}.
 * opts == NULL uses spx_plan_opts_auto of the matrix's statistics.
 * block_nnz 512 / 1024 / 2048 / 4096 runs 64 / 128 / 256 / 512-thread CTAs
 * (eight products per thread); other sizes run 256 threads.  row_ptr is read once (on the
 * GPU when where == SPX_DEVICE: validation, statistics and the plan are built
 * there).  *plan_out must be released with spx_plan_destroy.
 */
spx_status spx_plan_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, spx_loc where,
                        const spx_plan_opts_t* opts, spx_plan** plan_out);

spx_status spx_plan_get_info(const spx_plan* plan, spx_plan_info_t* out);

/* Host copies of the task table (4*tasks int32) and long-row table
   (4*long_rows int32); either pointer may be NULL. */
spx_status spx_plan_get_tasks(const spx_plan* plan, int32_t* tasks, int32_t* long_rows);

/*
 * The device table (info.table_bytes bytes), in this order:
 *   - the tasks in the device form, 4 int32 each: {kind | code << 2 |
 *     aux << 8, first row, p0, p1} with aux = #rows of a group or the slot of
 *     a segment, [p0, p1) the nonzeros the task covers;
 *   - the long-row table as spx_plan_get_tasks gives it;
 *   - when lanes_div == 0 (every group segmented): T uint16 per group, in task
 *     order, T = the group's threads (block_nnz / 8 for block_nnz 512, 1024,
 *     2048 or 4096, else 256).  Thread t sums the group's products [t*Q,
 *     t*Q + Q), Q = ceil(block_nnz / T); its entry is 2*r + s, r the group's
 *     row (counted from its first) holding product t*Q (the last row starting
 *     at or before it), s = 1 when that row starts before t*Q; 0 for a thread
 *     past the group's products.  The SpMV kernel takes each thread's first
 *     row from here instead of searching the row offsets.
 * The table depends only on row_ptr (the structure), like the plan.
 */
/* Host copy of the device table: writes info.table_bytes bytes to `table`. */
spx_status spx_plan_get_table(const spx_plan* plan, void* table);

/*
 * Copy the plan's device table into caller-owned device memory `table` (at
 * least info.table_bytes, 16-byte aligned) on `stream`, and remember that
 * address.  Must precede the first compute call with this plan; `table` must
 * stay valid while the plan is used.
 */
spx_status spx_plan_upload(spx_plan* plan, void* table, size_t table_bytes, spx_stream_t stream);

spx_status spx_plan_destroy(spx_plan* plan);

/*
 * Structure fingerprint of a plan, for callers that rewrite a matrix's row
 * offsets in place and keep its plan.  [SpMM-ops] §4 (the profile cached on
 * the matrix descriptor is invalidated when the matrix changes).  A plan is
 * built from one row_ptr, and the compute calls check only M, K and nnz, so a
 * changed row_ptr with the same sizes would use a stale plan.  The fingerprint
 * of row_ptr[0..M] is
 *   F = sum over i = 0..M of mix(2^32 * i + (uint32) row_ptr[i])   (mod 2^64),
 * where mix is SplitMix64's output function (add 0x9E3779B97F4A7C15, then
 * xor-shift-multiply by 0xBF58476D1CE4E5B9 and 0x94D049BB133111EB with shifts
 * 30, 27, 31).  Being a sum, it is the same on the host and on the GPU.
 *   spx_plan_fingerprint: F of the row_ptr the plan was built from.
 *   spx_plan_validate: recomputes F from `row_ptr` (host, or device memory:
 *     one launch and temporary memory from the stream-ordered allocator, then
 *     `stream` is synchronised) and returns SPX_OK when M, K, nnz and F all
 *     match the plan, SPX_ERR_ARG otherwise (a stale plan: build a new one).
 *     One O(M) read of row_ptr; not needed on the compute path.
 */
spx_status spx_plan_fingerprint(const spx_plan* plan, uint64_t* fingerprint_out);
spx_status spx_plan_validate(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr,
                             spx_loc where, spx_stream_t stream);

/*
 * Measured choice of plan options, cached per matrix profile.  [SpMM-ops] §4
 * (profile the matrix once -- row-length statistics as the dispatch key --
 * pick the mapping, keep the choice with the matrix).  Times each candidate
 * option set with spx_spmv_csr on `stream` (one warm-up, then `reps` timed
 * calls, CUDA events) on the caller's matrix and x, and returns the fastest
 * in *best.
 *   row_ptr_host: the row offsets in host memory (for the plans and the key);
 *   row_ptr, col, val, x: the matrix and a representative x in device memory;
 *   y_scratch: device fp32[M], overwritten (alpha 1, beta 0).
 *   candidates: ncand (1..16) option sets, or NULL for the built-in four:
 *     the defaults (B 2048, D 16); D 4; the segmented reduction (D 0) with
 *     B 1024; and with B 2048.
 *   times_ms: optional, ncand (or 4) floats: mean time per call of each
 *     candidate; -1 when the answer came from the cache.
 *   cached: optional; 1 when the answer came from the cache, else 0.
 * The cache is process-wide, keyed by the device, M, K, nnz, the row-length
 * sum of squares, maximum and 99th percentile, and the candidate list: a
 * matrix with the same profile reuses the choice without timing.  Unlike
 * the compute calls, this one allocates and frees device memory for the
 * candidate plans (cudaMalloc / cudaFree) and synchronises `stream`.
 */
spx_status spx_plan_autotune(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr_host, const int32_t* row_ptr,
                             const int32_t* col, const float* val, const float* x, float* y_scratch,
                             const spx_plan_opts_t* candidates, int32_t ncand, int32_t reps, spx_stream_t stream,
                             spx_plan_opts_t* best, float* times_ms, int32_t* cached);

/* Empties the spx_plan_autotune cache. */
spx_status spx_plan_autotune_forget(void);

/* ------------------------------------------------------------ SpMV */

/*
 * y = alpha * A x + beta * y, A in CSR (M x K, fp32 values, int32 indices),
 * fp32 arithmetic.  [SpMM-ops] §2 (y_i = sum over row i of values[p] *
 * x[col_indices[p]]; thread/warp/CTA/segment mappings), [LSMR-dual] §2 and
 * §5.2 (alpha/beta with beta scaling the old output).
 *   plan: built from this row_ptr with the same M, K, nnz, and uploaded.
 *   x[K], y[M] device fp32 (4-byte aligned); x and y must not overlap.
 *   scratch: device memory of at least info.scratch_bytes (may be NULL when
 *     that is 0); two calls that share a scratch buffer must not overlap in
 *     time.
 * Each row is reduced in a fixed order, so the result is bitwise
 * reproducible run to run (no floating-point atomics).
 * Launches: 1, plus 1 fix-up launch when the plan has split rows.
 */
spx_status spx_spmv_csr(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr,
                        const int32_t* col, const float* val, float alpha, const float* x, float beta, float* y,
                        void* scratch, size_t scratch_bytes, spx_stream_t stream);

/*
 * spx_spmv_csr over nbatch (x, y) pairs in HOST memory (pinned for full
 * speed): for batch b, x_host[b*x_stride .. +K) is copied up (x_stride 0:
 * the same x for every batch; else x_stride >= K), y = alpha*A x +
 * beta*y is computed (y_host[b*y_stride .. +M) copied up first when beta != 0)
 * and y is copied back into y_host.  The copies run on two streams of their
 * own, so batch b's upload and batch b-2's download overlap batch b-1's
 * product (two device slots for x and y in `work`).  A serving pipeline over
 * one stored matrix; the pages' SpMV ([SpMM-ops] §2) per batch.
 *   work: device memory of at least spx_spmv_csr_hostio_work_bytes(M, K)
 *         bytes, 256-byte aligned, owned by the caller;
 *   scratch: as for spx_spmv_csr.
 * All work is ordered after earlier work on `stream`, and `stream` resumes
 * only when every result is back in y_host: synchronise `stream` before
 * reading y_host.  Launches: those of spx_spmv_csr, per batch.
 */
size_t spx_spmv_csr_hostio_work_bytes(int32_t M, int32_t K);
spx_status spx_spmv_csr_hostio(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr,
                               const int32_t* col, const float* val, float alpha, const float* x_host,
                               int64_t x_stride, float beta, float* y_host, int64_t y_stride, int32_t nbatch,
                               void* work, size_t work_bytes, void* scratch, size_t scratch_bytes,
                               spx_stream_t stream);

/*
 * The two-direction operator pair of a least-squares solver, with CSC(A)
 * stored as CSR(A^T) so both directions are row sweeps ([LSMR-dual] §1, §4,
 * §5.2):
 *   u = alpha_u * A v   + beta_u * u     (A: m x n,  CSR(A))
 *   v = alpha_v * A^T u + beta_v * v     (A^T: n x m, CSR(A^T)), reading the new u
 * enqueued in that order on one stream.  The solver's step is alpha_u = 1,
 * beta_u = -alpha_k and alpha_v = 1, beta_v = -beta_k.
 *   plan_A / plan_At: uploaded plans of CSR(A) and CSR(A^T).
 *   scratch: at least max(scratch_bytes of both plans).
 * The second product is launched with programmatic dependent launch: its
 * CTAs start loading CSR(A^T) while the first product's last CTAs run, and
 * read u only after the first product has finished.
 */
spx_status spx_spmv_csr_dual(const spx_plan* plan_A, const spx_plan* plan_At, int32_t m, int32_t n, int64_t nnz,
                             const int32_t* A_row_ptr, const int32_t* A_col, const float* A_val,
                             const int32_t* At_row_ptr, const int32_t* At_col, const float* At_val, float* v,
                             float alpha_u, float beta_u, float* u, float alpha_v, float beta_v, void* scratch,
                             size_t scratch_bytes, spx_stream_t stream);

/*
 * spx_spmv_csr for callers that cannot allocate device memory -- code that
 * runs where cudaMalloc is not available or not allowed (an allocator-free
 * host runtime, a plugin handed only fixed buffers, a context that forbids
 * allocation after start-up), and so cannot provide the scratch buffer
 * spx_spmv_csr takes.  The pages have no counterpart; it is a deployment aid.
 *
 * Same operation, kernels and result as spx_spmv_csr (bitwise); the partial
 * sums of split rows go to one fixed device array inside this library
 * instead: SPX_NOALLOC_MAX_SLOTS floats (256 KiB), held by every GPU that
 * loads the library until the process exits.  The caller still provides the
 * plan (uploaded), the matrix, x and y.  No call allocates: no cudaMalloc,
 * no cudaFree, no allocating library routine.
 *   - A plan needing more than SPX_NOALLOC_MAX_SLOTS partial sums (split-row
 *     segments; spx_plan_info_t.slots) is rejected with
 *     SPX_ERR_SCRATCH_LIMIT before anything is launched.
 *   - Each call made outside stream capture looks up the array's device
 *     address (cudaGetSymbolAddress, with the calling device current), so a
 *     cudaDeviceReset between calls is picked up by the next such call.  A
 *     call on a capturing stream reuses the address the last call outside
 *     capture found on that device: make the first call on each device before
 *     any stream capture there (SPX_ERR_NOT_READY otherwise), and do not
 *     reset the device between that call and the end of the capture.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents; each slot is written before it is read within a call,
 *     so nothing needs clearing.  Calls that overlap in time on the GPU
 *     (different streams, no ordering between them) race on the array and
 *     give wrong results; order them on one stream or with events.
 */
#define SPX_NOALLOC_MAX_SLOTS 65536
spx_status spx_spmv_csr_noalloc(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr,
                                const int32_t* col, const float* val, float alpha, const float* x, float beta,
                                float* y, spx_stream_t stream);

/* ------------------------------------------------------------ SpMM */

/*
 * C = alpha * A B + beta * C, A in CSR (M x K, fp32), B dense K x N
 * row-major (leading dimension ldb >= N), C dense M x N row-major (ldc >= N),
 * fp32 arithmetic.  [SpMM-ops] §3 (C_{i,n} = sum_{k in N(i)} A_{ik} B_{k,n};
 * B's contiguous columns accumulated in registers) and §3.1-§3.3 (variant
 * chosen by N):
 *   N <= 8           lanes split the row's nonzeros, N accumulators each;
 *   N % 4 == 0       column tiles of T = pow2ceil(N) capped at 128, one
 *                    sub-warp of T/4 lanes per (row, tile), float4 B loads,
 *                    tiles outermost;
 *   otherwise        a warp per row, lanes over columns (scalar).
 * The float4 variants need B, C 16-byte aligned and ldb, ldc multiples of 4;
 * otherwise the scalar variant runs.  Launches: 1.
 */
spx_status spx_spmm_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                        const float* val, int32_t N, const float* B, int64_t ldb, float alpha, float beta, float* C,
                        int64_t ldc, spx_stream_t stream);

/* spx_spmm_csr with the column tile T of the float4 variants given by the
   caller (0 = automatic as above; else a power of two in [8, 128]). */
spx_status spx_spmm_csr_tiled(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                              const float* val, int32_t N, const float* B, int64_t ldb, float alpha, float beta,
                              float* C, int64_t ldc, int32_t col_tile, spx_stream_t stream);

/*
 * spx_spmm_csr with A's values and B stored as bf16 (bit patterns), products
 * and sums in fp32, C fp32.  [SpMM-ops] §5: storage and accumulation
 * precision are separate; for SpMM the narrower B halves the gathered bytes.
 * bf16 -> fp32 widening is exact and bf16 x bf16 products are exact in fp32,
 * so the result carries fp32 summation error only.
 * Needs N, ldb, ldc multiples of 4; B 8-byte and C 16-byte aligned
 * (SPX_ERR_UNSUPPORTED / SPX_ERR_ALIGN otherwise).  Launches: 1.
 */
spx_status spx_spmm_csr_bf16(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                             const uint16_t* val, int32_t N, const uint16_t* B, int64_t ldb, float alpha, float beta,
                             float* C, int64_t ldc, spx_stream_t stream);

/*
 * spx_spmm_csr_bf16 with IEEE binary16 (fp16) bit patterns instead of bf16
 * ([SpMM-ops] §5 names both 16-bit formats).  fp16 -> fp32 widening is exact
 * (subnormals included) and an fp16 x fp16 product (11-bit significands) is
 * exact in fp32, so the result again carries fp32 summation error only.  Same
 * shape and alignment rules as spx_spmm_csr_bf16.  Launches: 1.
 */
spx_status spx_spmm_csr_f16(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                            const uint16_t* val, int32_t N, const uint16_t* B, int64_t ldb, float alpha, float beta,
                            float* C, int64_t ldc, spx_stream_t stream);

/*
 * Planned SpMM for skewed rows.  [SpMM-ops] §2.4 (a long row is split, its
 * partial sums combined in a second pass) applied to C = alpha*A*B + beta*C:
 * the rows the SpMV plan `plan` (spx_plan_csr of the same matrix, uploaded)
 * classes as long -- longer than its pack_max -- are not walked by one
 * sub-warp.  A CTA row (length <= cta_max) is reduced by a whole CTA; a split
 * row's segments of seg_nnz nonzeros each write a partial row to scratch, and
 * a fix-up launch adds them in segment order and applies alpha/beta.  All
 * other rows run as in spx_spmm_csr.  Every sum is in a fixed order, so the
 * result is reproducible run to run (it may differ in rounding from
 * spx_spmm_csr, which sums a long row in one sequence).
 * scratch: spx_spmm_csr_planned_scratch_bytes(plan, N) bytes (slots x N
 * floats, 4-byte aligned; none without split rows).  Needs N, ldb, ldc
 * multiples of 4, B 16-byte (fp32) or 8-byte (16-bit) and C 16-byte aligned
 * (SPX_ERR_UNSUPPORTED / SPX_ERR_ALIGN otherwise); SPX_ERR_ARG for a plan of
 * another matrix or too little scratch, SPX_ERR_NOT_READY before the upload.
 * Launches: 1 to 3.  The _bf16 and _f16 forms take 16-bit A values and B as
 * spx_spmm_csr_bf16 / spx_spmm_csr_f16 do.  A row costs an SpMM sub-warp far
 * more than an SpMV group, so plans for SpMM want a lower pack_max than the
 * SpMV defaults: on a 4.2M-row power-law matrix at N = 32, block_nnz 1024,
 * pack_max 64, cta_max 2048, seg_nnz 2048 measured 1.9 ms against 2.9 ms
 * with spx_plan_opts_auto's choice (and 32.7 ms for spx_spmm_csr).
 */
size_t spx_spmm_csr_planned_scratch_bytes(const spx_plan* plan, int32_t N);
spx_status spx_spmm_csr_planned(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr,
                                const int32_t* col, const float* val, int32_t N, const float* B, int64_t ldb,
                                float alpha, float beta, float* C, int64_t ldc, void* scratch, size_t scratch_bytes,
                                spx_stream_t stream);
spx_status spx_spmm_csr_bf16_planned(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz,
                                     const int32_t* row_ptr, const int32_t* col, const uint16_t* val, int32_t N,
                                     const uint16_t* B, int64_t ldb, float alpha, float beta, float* C, int64_t ldc,
                                     void* scratch, size_t scratch_bytes, spx_stream_t stream);
spx_status spx_spmm_csr_f16_planned(const spx_plan* plan, int32_t M, int32_t K, int64_t nnz,
                                    const int32_t* row_ptr, const int32_t* col, const uint16_t* val, int32_t N,
                                    const uint16_t* B, int64_t ldb, float alpha, float beta, float* C, int64_t ldc,
                                    void* scratch, size_t scratch_bytes, spx_stream_t stream);

/* Which SpMM variant spx_spmm_csr would launch for these arguments:
   0 = small-N, 1 = float4 with N <= 128, 2 = float4 with N > 128, 3 = scalar. */
int32_t spx_spmm_csr_variant(int32_t N, const float* B, int64_t ldb, const float* C, int64_t ldc);

/* ------------------------------------------------------------ SELL-C-sigma */

/*
 * Sliced ELLPACK, C = 32 ([SpMM-ops] §1.4 and [Formats] §6: rows sorted by
 * length inside windows of sigma rows, slices of C rows padded to their
 * longest row and stored column-major, so the C threads of a slice read
 * consecutive words).  Rows longer than `piece` entries are first cut into
 * pieces of `piece` entries, each sorted and sliced like a row; a second
 * launch adds each long row's pieces in piece order.
 *   sigma: window of pseudo-rows sorted together, a multiple of 32 in
 *          [32, 2^20]; piece: in [1, 2^24].  Defaults: sigma 1024, piece 64
 *          (fastest of a sweep on a power-law matrix, mean row length 16).
 */
typedef struct spx_sell_opts_t {
    int32_t sigma;
    int32_t piece;
} spx_sell_opts_t;

typedef struct spx_sell_info_t {
    int64_t M, K, nnz;
    int64_t slices;       /* ceil(pseudo_rows / 32)                          */
    int64_t pseudo_rows;  /* rows of length <= piece, plus the pieces        */
    int64_t padded;       /* stored entries including padding (32 per slice
                             per position up to the slice's longest row)     */
    int64_t long_rows;    /* rows cut into pieces                            */
    int64_t slots;        /* partial sums (one per piece)                    */
    size_t image_bytes;   /* device bytes for spx_sell_upload                */
    size_t scratch_bytes; /* device scratch bytes of each spx_spmv_sell call */
    spx_sell_opts_t opts;
} spx_sell_info_t;

typedef struct spx_sell spx_sell; /* opaque, host-side */

spx_status spx_sell_opts_default(spx_sell_opts_t* out);

/*
 * Build the SELL-C-sigma form of a CSR matrix from host or device arrays.
 * Device arrays are converted on the GPU (the default stream, synchronous):
 * pieces and slots from per-row counts and scans, the window-local order by two
 * stable radix passes (length descending, then window), slice widths from
 * each slice's first pseudo-row, and a scatter into the column-major image.
 * The image then lives in library-owned device memory until the first
 * spx_sell_upload, which copies it device to device and frees it.  Both paths
 * give the same image.  Pseudo-rows are listed in row order (a
 * long row's pieces in piece order), stably sorted by length, longest first,
 * inside each window of sigma pseudo-rows, then cut into slices of 32.
 * Within a slice, entry j of lane r sits at slice_ptr[s] + 32 j + r; padding
 * has column -1 and value 0.  prow holds the row of each pseudo-row, -1-slot
 * for a piece, INT32_MIN for the unused lanes of the last slice.  opts NULL:
 * the defaults.  Errors: SPX_ERR_ARG (row_ptr[0] != 0 or row_ptr[M] != nnz),
 * SPX_ERR_NOT_SORTED (row_ptr decreasing),
 * SPX_ERR_INDEX_RANGE (a column outside [0, K) or more than 2^31-1 padded
 * entries).  Release with spx_sell_destroy.
 */
spx_status spx_sell_build(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                          const float* val, spx_loc where, const spx_sell_opts_t* opts, spx_sell** out);
spx_status spx_sell_get_info(const spx_sell* sell, spx_sell_info_t* out);
/* Host copies of slice_ptr[slices+1], prow[32 slices], longrows[4 long_rows]
   ({row, first slot, #pieces, 0}), scol[padded], sval[padded]; any may be NULL.
   A GPU-built form is read back from device memory (its own copy before the
   first upload, the uploaded image after it). */
spx_status spx_sell_get_arrays(const spx_sell* sell, int32_t* slice_ptr, int32_t* prow, int32_t* longrows,
                               int32_t* scol, float* sval);
/* Copy the format into caller-owned device memory (info.image_bytes, 16-byte
   aligned) and remember the address; required before spx_spmv_sell. */
spx_status spx_sell_upload(spx_sell* sell, void* image, size_t image_bytes, spx_stream_t stream);
spx_status spx_sell_destroy(spx_sell* sell);

/*
 * y = alpha * A x + beta * y with A in uploaded SELL-C-sigma form: one warp
 * per slice, one thread per pseudo-row, coalesced column-major loads, x
 * gathered through the read-only path; pieces write partial sums to
 * `scratch` (info.scratch_bytes) and a second launch (one warp per long
 * row) adds them in piece order and applies alpha/beta.  Deterministic
 * (fixed summation order).  x[K], y[M] device fp32, not overlapping.
 * Launches: 1, plus 1 when the matrix has long rows.
 */
spx_status spx_spmv_sell(const spx_sell* sell, int32_t M, int32_t K, float alpha, const float* x, float beta,
                         float* y, void* scratch, size_t scratch_bytes, spx_stream_t stream);

/*
 * COO SpMV y = alpha * A x + beta * y over triplets sorted by row (columns in
 * any order within a row; duplicates allowed and summed as separate terms).
 * [Formats] §1 (the COO format: one row index, column index and value per
 * stored entry) and the COO row of the dispatch rule table in [SpMM-ops] §4
 * (work split by nonzeros with a segmented reduction, so row lengths never
 * unbalance the launch).
 *   coo_row, coo_col int32[nnz], coo_val fp32[nnz], x fp32[K], y fp32[M]:
 *   device memory, owned by the caller; x and y must not overlap.
 *   Each row's sum is taken in a fixed order (bitwise reproducible); rows
 *   without entries get beta * y (0 when beta == 0: y is then write-only).
 *   scratch: device memory of at least spx_spmv_coo_scratch_bytes(nnz)
 *   bytes (two floats per 2048 entries), owned by the caller.
 * Launches: 1 for nnz <= 2048 or nnz == 0, else 2.  Entries whose row is out
 * of [0, M) or smaller than the row before it, or whose column is out of
 * [0, K), are skipped without any out-of-bounds access; the kernel records
 * SPX_ERR_INDEX_RANGE or SPX_ERR_NOT_SORTED, which spx_last_device_error
 * returns (y is then unspecified).
 */
size_t spx_spmv_coo_scratch_bytes(int64_t nnz);
spx_status spx_spmv_coo(int32_t M, int32_t K, int64_t nnz, const int32_t* coo_row, const int32_t* coo_col,
                        const float* coo_val, float alpha, const float* x, float beta, float* y, void* scratch,
                        size_t scratch_bytes, spx_stream_t stream);

typedef struct spx_wcsr_plan spx_wcsr_plan; /* opaque, host-side: the task split of WCSR windows / BSR block-rows */

/*
 * C = alpha * A B + beta * C with A in BSR (br x bc blocks, row-major inside,
 * bf16), B dense K x N bf16 row-major (ldb), C dense M x N fp32 row-major
 * (ldc); products accumulated in fp32 (on the tensor cores for the shapes
 * below), the epilogue in fp32 (beta == 0: C is write-only).  [SpMM-ops]
 * §3.4 (loop over the nonzero blocks, each a small dense GEMM on the tensor
 * cores) and
 * [AsyncSparse] §2.2.1, §3 (BCSR SpMM: asynchronous copies of A blocks and
 * B tiles into shared memory feeding the matrix units).
 * Shapes: any br x bc block, any M, K and N.  A ragged last block-row or
 * block column is zero-padded in the BSR arrays (as spx_build_bsr writes
 * them).  B rows at or beyond K are read as zeros, and C is stored only
 * inside its M x N part, so a ragged last column tile does a whole tile's
 * work but writes nothing past column N.  ldb >= N, ldc >= N; nnzb * br
 * and nnzb * bc must fit int32 (SPX_ERR_INDEX_RANGE otherwise).
 * 64 x 64 blocks run on the tensor cores: ldb a multiple of 8, bsr_val and
 * B 16-byte aligned, C 4-byte aligned (SPX_ERR_ALIGN otherwise).  Blocks
 * whose br is a multiple of 16 up to 128 and whose bc is 16, 32, 48, 64 or a
 * multiple of 64 run on the same tensor-core kernel when ldb is a multiple
 * of 8 and bsr_val and B are 16-byte aligned.  Every other shape, or those
 * shapes with other alignments, runs on the CUDA cores (one launch; each CTA
 * owns up to 64 rows of a block-row and a strip of columns and sums every
 * element's terms in their stored order with fp32 fused multiply-adds): ldb
 * even, bsr_val 2-byte, B and C 4-byte aligned (SPX_ERR_ALIGN otherwise).
 * The tensor-core launches are 1 persistent kernel (as many CTAs as the SMs
 * hold at once, each walking a static list of output tiles of 128 columns x
 * one block-row; a tile's epilogue overlaps the next tile's MMAs), or 2 when
 * the last round of tiles would leave at least half the CTAs idle and the
 * block-rows average 48 ring stages (64-column chunks of blocks) or more:
 * that round's tiles are then cut in
 * two, the first launch storing their head pieces and a second one (allowed
 * to start early, programmatic dependent launch) adding the tail pieces into
 * C after the first has finished.  Results are then rounded in a different
 * order than with one launch (fp32 rounding level), but are the same from
 * run to run.  Pipeline waits are bounded: on expiry the kernel records an
 * error that spx_last_device_error reports as SPX_ERR_TIMEOUT.
 */
spx_status spx_spmm_bsr(int32_t M, int32_t K, int32_t br, int32_t bc, int64_t nnzb, const int32_t* bsr_row_ptr,
                        const int32_t* bsr_col, const uint16_t* bsr_val, int32_t N, const uint16_t* B, int64_t ldb,
                        float alpha, float beta, float* C, int64_t ldc, spx_stream_t stream);

/*
 * BSR task split, the counterpart of the WCSR one for block-rows (the same
 * plan type): spx_bsr_plan_build(M, nnzb, bsr_row_ptr, where, max_blocks,
 * &plan) cuts every block-row of more than max_blocks blocks (max_blocks <= 0:
 * 64) into balanced pieces of consecutive blocks; upload, inspect and
 * destroy it with the spx_wcsr_plan_* calls.  spx_spmm_bsr_planned runs one
 * CTA per task and column tile; whole block-rows write C as spx_spmm_bsr
 * does, pieces write raw 64 x N partial tiles to scratch
 * (spx_spmm_bsr_planned_scratch_bytes) and a fix-up adds them in piece order
 * and applies alpha/beta.  Same shape, alignment and error rules as
 * spx_spmm_bsr, plus those of spx_spmm_wcsr_planned for the plan and scratch;
 * the planned call takes 64 x 64 blocks only (SPX_ERR_UNSUPPORTED otherwise).
 * Launches: 1, or 2 with split block-rows.
 */
spx_status spx_bsr_plan_build(int32_t M, int64_t nnzb, const int32_t* bsr_row_ptr, spx_loc where, int32_t max_blocks,
                              spx_wcsr_plan** out);
size_t spx_spmm_bsr_planned_scratch_bytes(const spx_wcsr_plan* plan, int32_t N);
spx_status spx_spmm_bsr_planned(const spx_wcsr_plan* plan, int32_t M, int32_t K, int32_t br, int32_t bc, int64_t nnzb,
                                const int32_t* bsr_row_ptr, const int32_t* bsr_col, const uint16_t* bsr_val,
                                int32_t N, const uint16_t* B, int64_t ldb, float alpha, float beta, float* C,
                                int64_t ldc, void* scratch, size_t scratch_bytes, spx_stream_t stream);

/* ------------------------------------------------------------ WCSR */

/*
 * CSR -> WCSR (window CSR) with windows of 64 rows.  [AsyncSparse] §2.2.2:
 * each window keeps the union of the columns its rows use (window_col_idx,
 * -1 = padding) and a dense block of values for those compressed columns.
 * Here the union of window w (ascending) is padded with -1 to a multiple of
 * 64 and cut into chunks of 64 compressed columns:
 *   win_ptr int32[ceil(M/64)+1]: first chunk of each window (chunk count);
 *   win_col int32[64 * nchunks]: original column of each compressed position;
 *   win_val [nchunks][64 rows][64 positions] of val_bytes each, row-major,
 *           zero where the row has no entry in that column (and for rows
 *           beyond M in the last window).
 * fill = nnz / (nchunks * 4096).  Two calls: with win_col == win_val == NULL
 * only *nchunks_out (and win_ptr, when given) is produced.  Arrays are all
 * host or all device per `where`.  where == SPX_DEVICE builds on the GPU
 * (stable radix sort of the entries by window, column and row in the window;
 * temporary memory from the stream-ordered allocator) with the same results
 * as the host build, and synchronises the stream before returning.
 * Errors: SPX_ERR_ARG (row_ptr[0] != 0), SPX_ERR_DUPLICATE (a repeated
 * (row, col)), SPX_ERR_INDEX_RANGE, SPX_ERR_NOT_SORTED (row_ptr decreasing).
 */
spx_status spx_build_wcsr(int32_t M, int32_t K, const int32_t* row_ptr, const int32_t* col, const void* val,
                          int32_t val_bytes, int32_t* win_ptr, int32_t* win_col, void* win_val, int64_t* nchunks_out,
                          double* fill_out, spx_loc where, spx_stream_t stream);

/*
 * C = alpha * A B + beta * C with A in WCSR (bf16 values), B dense K x N bf16
 * row-major (ldb), C dense M x N fp32 (ldc); fp32 accumulation on the tensor
 * cores.  [AsyncSparse] §4.1 (TMA for the window's values, a cooperative
 * gather of the B rows named by window_col_idx into a swizzled shared tile,
 * tensor-core MMA).  One CTA per (window, 128 output columns); no atomics,
 * so the result is deterministic.  Supported: N a multiple of 8 (B rows are
 * gathered in 16-byte pieces; a ragged last 128-column tile gathers zeros
 * past column N and stores nothing there), ldb a multiple of 8, win_val and
 * B 16-byte aligned, at most 65535 windows (M <= 4,194,240); any K.
 * Launches: 1.
 * Bounded pipeline waits report SPX_ERR_TIMEOUT through
 * spx_last_device_error.
 */
spx_status spx_spmm_wcsr(int32_t M, int32_t K, int64_t nchunks, const int32_t* win_ptr, const int32_t* win_col,
                         const uint16_t* win_val, int32_t N, const uint16_t* B, int64_t ldb, float alpha, float beta,
                         float* C, int64_t ldc, spx_stream_t stream);

/*
 * WCSR task split.  [AsyncSparse] §4.1 (the WCSR kernel splits windows with
 * many chunks over several thread blocks so that no block carries a whole
 * wide window).  spx_wcsr_plan_build reads win_ptr (host or device, once) and
 * cuts every window with more than max_chunks chunks (max_chunks <= 0: 16)
 * into balanced pieces of consecutive chunks; the other windows stay whole.
 * tasks: {window, first chunk, chunks, partial slot or -1 for a whole
 * window}, longest first (ties in window and piece order: CTAs start in task
 * order, so the long tasks run early and the last wave holds short ones);
 * splits: {window, first slot, pieces, 0}.  The table (tasks then
 * splits, table_bytes, 16-byte aligned caller memory) goes to the device with
 * spx_wcsr_plan_upload.  spx_spmm_wcsr_planned runs one CTA per task and
 * column tile; a whole window writes C as spx_spmm_wcsr does, a piece writes
 * its raw 64 x N partial tile to scratch (spx_spmm_wcsr_planned_scratch_bytes:
 * slots x 64 x N floats, 16-byte aligned), and a fix-up launch adds a split
 * window's pieces in piece order and applies alpha/beta -- no atomics, so the
 * result is reproducible.  Errors: SPX_ERR_ARG (win_ptr[0] != 0 or
 * win_ptr[W] != nchunks, a plan of another matrix, too little scratch),
 * SPX_ERR_NOT_SORTED (win_ptr decreasing), SPX_ERR_NOT_READY (not uploaded),
 * SPX_ERR_UNSUPPORTED (more than 65535 tasks), and those of spx_spmm_wcsr.
 * Launches: 1, or 2 with split windows.
 */
typedef struct spx_wcsr_plan_info_t {
    int64_t windows, tasks, split_windows, slots;
    size_t table_bytes;
    int32_t max_chunks;
} spx_wcsr_plan_info_t;
spx_status spx_wcsr_plan_build(int32_t M, int64_t nchunks, const int32_t* win_ptr, spx_loc where, int32_t max_chunks,
                               spx_wcsr_plan** out);
spx_status spx_wcsr_plan_info(const spx_wcsr_plan* plan, spx_wcsr_plan_info_t* out);
/* Host copies of tasks[4 tasks] and splits[4 split_windows]; either may be NULL. */
spx_status spx_wcsr_plan_get_tasks(const spx_wcsr_plan* plan, int32_t* tasks, int32_t* splits);
spx_status spx_wcsr_plan_upload(spx_wcsr_plan* plan, void* table, size_t table_bytes, spx_stream_t stream);
spx_status spx_wcsr_plan_destroy(spx_wcsr_plan* plan);
size_t spx_spmm_wcsr_planned_scratch_bytes(const spx_wcsr_plan* plan, int32_t N);
spx_status spx_spmm_wcsr_planned(const spx_wcsr_plan* plan, int32_t M, int32_t K, int64_t nchunks,
                                 const int32_t* win_ptr, const int32_t* win_col, const uint16_t* win_val, int32_t N,
                                 const uint16_t* B, int64_t ldb, float alpha, float beta, float* C, int64_t ldc,
                                 void* scratch, size_t scratch_bytes, spx_stream_t stream);

/* ------------------------------------------------------------ measurement */

/*
 * The stream + gather floor of a CSR SpMV over a matrix: partials[b] = the
 * sum, over a grid-stride share of the nonzeros, of val[p] * x[col[p]] -- each
 * value and column read once, x gathered once per nonzero, no rows, no
 * reduction order (a probe, not a product).  Its time is the floor for any
 * SpMV kernel over the same col/val/x, since the random x gathers, not HBM
 * bandwidth, bound a product whose columns are spread over a vector larger
 * than the L1 caches (the request rate of the gathers, [SpMM-ops] §2.5).
 * Columns must lie in [0, K) (not checked: use matrices built by this
 * library).  nblocks: CTAs of 256 threads (spx_gather_probe_blocks() = 8 per
 * SM).  Launches: 1.
 */
int32_t spx_gather_probe_blocks(void);
spx_status spx_gather_probe(int64_t nnz, const int32_t* col, const float* val, const float* x, int32_t K,
                            float* partials, int32_t nblocks, spx_stream_t stream);

/*
 * Test aid for the bounded device waits: failure detection without a GPU fault
 * or hang.  One CTA arms an mbarrier that nothing completes and waits on it
 * with the same bounded wait the BSR and WCSR pipelines use.  After
 * limit_cycles SM clock cycles (0 .. 2e9; about 1 ms per 2e6 at 2 GHz) the
 * wait gives up, the timeout is recorded in the device error word and the
 * kernel returns: spx_last_device_error then reports SPX_ERR_TIMEOUT once,
 * and the context stays usable.  SPX_ERR_ARG (nothing launched) for a limit
 * outside that range.  Launches: 1.
 */
spx_status spx_wait_probe(int64_t limit_cycles, spx_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device-side error words:
 * SPX_ERR_TIMEOUT if a bounded wait of spx_spmm_bsr or spx_spmm_wcsr gave up, else the index
 * or ordering error spx_spmv_coo recorded, else SPX_OK.  The words are one
 * per device, shared by every stream: with calls still running on other
 * streams, the status read may come from any of them.
 */
spx_status spx_last_device_error(spx_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPX_H_ */
