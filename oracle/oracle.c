/*
 * oracle.c -- the test oracle for the sparse x dense products.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this code.  It shares no source, header,
 * table or helper with the CUDA library, and the library never calls it.
 *
 * Every function is the plain definition written out: single-threaded,
 * index order, fp64 accumulation for floating point, comparison sorts where
 * the library uses counting sorts.  No blocking, fusion or reordering.  The
 * same source built a second time with -fopenmp (liboracle_omp.so) runs the
 * independent row loops of the products on all host cores, for the CPU
 * baseline only; each row is still summed alone in index order, so no
 * result changes.
 *
 * Pages cited (by title and section):
 *   [SpMM-ops]  "通用稀疏矩阵乘法CUDA算子实现" (chengzipai.xyz)
 *   [BCSR-SpMV] "GPU加速实战用BCSR格式优化稀疏矩阵乘法附CUDA代码" (xxqk.cn)
 *   [AsyncSparse] AsyncSparse summary, "异步GPU架构下的稀疏矩阵乘法加速" (capital-peak.com)
 *   [LSMR-dual] "CUDA LSMR 专栏（二）：用 CSR/CSC 双存储压榨双向 SpMV" (chengzipai.xyz)
 *   [Formats]   "稀疏矩阵存储格式:COO、CSR、ELL、Hybrid 与块稀疏" (geek-doc.cn)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_ARG (-1)
#define OR_ERR_INDEX (-2)
#define OR_ERR_DUP (-4)
#define OR_ERR_NOMEM (-9)

#define I32MAX 2147483647LL

/* ------------------------------------------------------------ COO -> CSR */

typedef struct { int64_t a, b, pos; } key3_t;

static int cmp_key3(const void* x, const void* y) {
    const key3_t* p = (const key3_t*)x;
    const key3_t* q = (const key3_t*)y;
    if (p->a != q->a) return p->a < q->a ? -1 : 1;
    if (p->b != q->b) return p->b < q->b ? -1 : 1;
    if (p->pos != q->pos) return p->pos < q->pos ? -1 : 1;
    return 0;
}

/*
 * COO -> CSR.  [Formats] §3 (row_ptr from per-row counts and their prefix sum;
 * row i occupies [row_ptr[i], row_ptr[i+1])) and [SpMM-ops] §1.2 (sort the
 * triplets by (row, col)).  Written here as a comparison sort of
 * (row, col, input position): entries with equal (row, col) keep input order
 * and are not summed.  row_ptr[i] = number of entries whose row is < i.
 */
int or_build_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row, const int32_t* col,
                 const void* val, int32_t vbytes, int32_t* rp, int32_t* col_out, void* val_out) {
    if (M < 0 || K < 0 || nnz < 0 || nnz > I32MAX || vbytes <= 0) return OR_ERR_ARG;
    for (int64_t p = 0; p < nnz; ++p)
        if (row[p] < 0 || row[p] >= M || col[p] < 0 || col[p] >= K) return OR_ERR_INDEX;
    key3_t* t = (key3_t*)malloc(sizeof(key3_t) * (size_t)(nnz ? nnz : 1));
    if (!t) return OR_ERR_NOMEM;
    for (int64_t p = 0; p < nnz; ++p) { t[p].a = row[p]; t[p].b = col[p]; t[p].pos = p; }
    qsort(t, (size_t)nnz, sizeof(key3_t), cmp_key3);
    const char* vin = (const char*)val;
    char* vout = (char*)val_out;
    for (int64_t p = 0; p < nnz; ++p) {
        col_out[p] = (int32_t)t[p].b;
        memcpy(vout + p * vbytes, vin + t[p].pos * vbytes, (size_t)vbytes);
    }
    int64_t k = 0;
    for (int64_t i = 0; i <= M; ++i) {
        while (k < nnz && t[k].a < i) ++k;
        rp[i] = (int32_t)k;
    }
    free(t);
    return OR_OK;
}

/*
 * CSR(A) -> CSR(A^T), i.e. CSC(A).  [LSMR-dual] §2 (CSC(A) has exactly the
 * memory layout of CSR(A^T)) and §4 (build the other format once).  Output
 * row j lists the entries of column j in increasing source row (then source
 * position): a comparison sort of (col, row, position).
 */
int or_transpose(int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col, const void* val,
                 int32_t vbytes, int32_t* t_rp, int32_t* t_col, void* t_val) {
    if (M < 0 || K < 0 || nnz < 0 || nnz > I32MAX || vbytes <= 0) return OR_ERR_ARG;
    if (rp[0] != 0 || rp[M] != nnz) return OR_ERR_ARG;
    key3_t* t = (key3_t*)malloc(sizeof(key3_t) * (size_t)(nnz ? nnz : 1));
    if (!t) return OR_ERR_NOMEM;
    for (int32_t i = 0; i < M; ++i)
        for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
            if (col[p] < 0 || col[p] >= K) { free(t); return OR_ERR_INDEX; }
            t[p].a = col[p]; t[p].b = i; t[p].pos = p;
        }
    qsort(t, (size_t)nnz, sizeof(key3_t), cmp_key3);
    const char* vin = (const char*)val;
    char* vout = (char*)t_val;
    for (int64_t q = 0; q < nnz; ++q) {
        t_col[q] = (int32_t)t[q].b;
        memcpy(vout + q * vbytes, vin + t[q].pos * vbytes, (size_t)vbytes);
    }
    int64_t k = 0;
    for (int64_t j = 0; j <= K; ++j) {
        while (k < nnz && t[k].a < j) ++k;
        t_rp[j] = (int32_t)k;
    }
    free(t);
    return OR_OK;
}

/*
 * CSR -> BSR with br x bc blocks.  [AsyncSparse] §2.2.1 (store every block
 * that holds at least one nonzero, dense and contiguous; block_row_ptr over
 * block-rows, block_col_idx per block; fill_ratio = nnz / (nnz_blocks*br*bc))
 * and [BCSR-SpMV] §1 (one block-column index per block; values row-major or
 * column-major -- row-major here).  The last block-row/column is zero-padded
 * when br (bc) does not divide M (K).  A repeated (row, col) cannot live in
 * one dense slot: OR_ERR_DUP.  Two calls: with bcol_out == NULL only the
 * block count (and bsr_rp, when given) is produced.
 */
int or_build_bsr(int32_t M, int32_t K, const int32_t* rp, const int32_t* col, const void* val, int32_t vbytes,
                 int32_t br, int32_t bc, int32_t* bsr_rp, int32_t* bcol_out, void* bval_out,
                 int64_t* nnzb_out, double* fill_out) {
    if (M < 0 || K < 0 || br <= 0 || bc <= 0 || vbytes <= 0) return OR_ERR_ARG;
    int64_t nnz = rp[M];
    int64_t MB = ((int64_t)M + br - 1) / br;
    int64_t nb = 0;
    const char* vin = (const char*)val;
    char* vout = (char*)bval_out;
    int64_t blk_bytes = (int64_t)br * bc * vbytes;
    if (bsr_rp) bsr_rp[0] = 0;
    for (int64_t I = 0; I < MB; ++I) {
        int64_t r0 = I * br, r1 = r0 + br < M ? r0 + br : M;
        int64_t cnt = rp[r1] - rp[r0];
        key3_t* t = (key3_t*)malloc(sizeof(key3_t) * (size_t)(cnt ? cnt : 1));
        if (!t) return OR_ERR_NOMEM;
        int64_t n = 0;
        for (int64_t i = r0; i < r1; ++i)
            for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
                if (col[p] < 0 || col[p] >= K) { free(t); return OR_ERR_INDEX; }
                /* key: block column, then position inside the block, then p */
                t[n].a = col[p] / bc;
                t[n].b = (i - r0) * bc + col[p] % bc;
                t[n].pos = p;
                ++n;
            }
        qsort(t, (size_t)n, sizeof(key3_t), cmp_key3);
        for (int64_t q = 1; q < n; ++q)
            if (t[q].a == t[q - 1].a && t[q].b == t[q - 1].b) { free(t); return OR_ERR_DUP; }
        for (int64_t q = 0; q < n; ++q) {
            int first = (q == 0) || (t[q].a != t[q - 1].a);
            if (first) {
                if (bcol_out) {
                    bcol_out[nb] = (int32_t)t[q].a;
                    if (vout) memset(vout + nb * blk_bytes, 0, (size_t)blk_bytes);
                }
                ++nb;
            }
            if (bcol_out && vout)
                memcpy(vout + (nb - 1) * blk_bytes + t[q].b * vbytes, vin + t[q].pos * vbytes, (size_t)vbytes);
        }
        free(t);
        if (nb > I32MAX) return OR_ERR_INDEX;
        if (bsr_rp) bsr_rp[I + 1] = (int32_t)nb;
    }
    if (nnzb_out) *nnzb_out = nb;
    if (fill_out) *fill_out = nb ? (double)nnz / ((double)nb * (double)br * (double)bc) : 0.0;
    return OR_OK;
}

/* ---------------------------------------------------------- row statistics */

typedef struct {
    int64_t rows, nnz, sumsq;      /* M, S1 = sum l_i, S2 = sum l_i^2 */
    int32_t min, max, p50, p95, p99, empty;
    double mean, var, cv;
} or_row_stats_t;

static int cmp_i32(const void* x, const void* y) {
    int32_t a = *(const int32_t*)x, b = *(const int32_t*)y;
    return (a > b) - (a < b);
}

/*
 * Row-length statistics.  [LSMR-dual] §5.3 (l_i = row_ptr[i+1] - row_ptr[i];
 * its mean, variance and long tail) and [SpMM-ops] §4 (avg/p95/max nnz and the
 * coefficient of variation in the dispatch key).  Definitions fixed here:
 *   mean = (double)S1 / (double)M
 *   var  = (double)(M*S2 - S1^2) / ((double)M * (double)M)   (population; the
 *          numerator is exact in 128-bit integers and rounded once)
 *   cv   = sqrt(var) / mean  (0 when mean == 0)
 *   Pq   = nearest rank: the ceil(q*M/100)-th smallest length.
 */
int or_row_stats(int32_t M, const int32_t* rp, or_row_stats_t* out) {
    if (M < 0 || !out) return OR_ERR_ARG;
    memset(out, 0, sizeof(*out));
    out->rows = M;
    if (M == 0) return OR_OK;
    int32_t* l = (int32_t*)malloc(sizeof(int32_t) * (size_t)M);
    if (!l) return OR_ERR_NOMEM;
    int64_t s1 = 0, s2 = 0;
    int32_t empty = 0;
    for (int32_t i = 0; i < M; ++i) {
        l[i] = rp[i + 1] - rp[i];
        s1 += l[i];
        s2 += (int64_t)l[i] * l[i];
        empty += (l[i] == 0);
    }
    qsort(l, (size_t)M, sizeof(int32_t), cmp_i32);
    out->nnz = s1;
    out->sumsq = s2;
    out->min = l[0];
    out->max = l[M - 1];
    out->p50 = l[((int64_t)50 * M + 99) / 100 - 1];
    out->p95 = l[((int64_t)95 * M + 99) / 100 - 1];
    out->p99 = l[((int64_t)99 * M + 99) / 100 - 1];
    out->empty = empty;
    out->mean = (double)s1 / (double)M;
    __int128 num = (__int128)M * (__int128)s2 - (__int128)s1 * (__int128)s1;
    out->var = (double)num / ((double)M * (double)M);
    out->cv = out->mean > 0.0 ? sqrt(out->var) / out->mean : 0.0;
    free(l);
    return OR_OK;
}

/* ------------------------------------------------------------ SpMV plan */

typedef struct {
    int32_t block_nnz;   /* B: most nonzeros packed into one group            */
    int32_t block_rows;  /* R: most rows packed into one group                */
    int32_t pack_max;    /* P: rows with l <= P are packed into groups        */
    int32_t cta_max;     /* C: rows with P < l <= C get one CTA each          */
    int32_t seg_nnz;     /* S: rows with l > C are cut into segments of S     */
    int32_t lanes_div;   /* D: lanes per row in a group = pow2ceil(ceil(avg/D));
                            D == 0: every group uses the segmented reduction */
} or_plan_opts_t;

enum { OR_TASK_GROUP = 0, OR_TASK_CTA = 1, OR_TASK_SEG = 2 };

/*
 * Plan options from the row statistics ([SpMM-ops] §4: the dispatch key's
 * row-length spread picks the mapping): with cv >= 2 the groups hold 1024
 * nonzeros and use the segmented reduction (D = 0); otherwise 2048 nonzeros
 * and the lanes rule with D = 16.  R 256, P 512, C 8192, S 4096 either way.
 */
int or_plan_opts_auto(const or_row_stats_t* st, or_plan_opts_t* o) {
    if (!st || !o) return OR_ERR_ARG;
    int skewed = st->cv >= 2.0;
    o->block_nnz = skewed ? 1024 : 2048;
    o->block_rows = 256;
    o->pack_max = 512;
    o->cta_max = 8192;
    o->seg_nnz = 4096;
    o->lanes_div = skewed ? 0 : 16;
    return OR_OK;
}

static int32_t pow2ceil_clamp32(int64_t v) {
    int32_t w = 1;
    while (w < v && w < 32) w <<= 1;
    return w;
}

/*
 * The dispatch plan: which kernel mapping serves which rows.
 * [SpMM-ops] §2.1-§2.4 (thread-per-row, warp-per-row for rows up to a few
 * dozen nonzeros, a CTA per row for hundreds to thousands, segments of
 * SEGMENT_NNZ with a second-pass reduction for the longest rows), §4 (rule
 * table) and [Formats] §6 (pack rows into work bundles of similar nnz).
 *
 * Per row, by l_i:  l <= P        -> packed into a group
 *                   P < l <= C    -> one CTA for the row
 *                   l > C         -> split into ceil(l/S) segments
 * Groups: scanning rows upward, consecutive packed rows join the current
 * group while it has fewer than R rows and its nonzeros stay <= B; any
 * CTA/split row closes it.  Reduction code c of a group:
 *   D >= 1: each row is reduced by w lanes, w = the smallest power of two >=
 *           ceil(nnz_g / (rows_g * D)), clamped to [1, 32]; c = log2(w)
 *           (w == 1 is thread-per-row, w == 32 warp-per-row);
 *   D == 0: c = 6, the segmented reduction -- every thread sums an equal run
 *           of consecutive products and rows crossing threads are joined by a
 *           scan, so work per thread no longer follows row length
 *           ([Formats] §6, the merge-based remedy: equal nonzeros per thread).
 * Task list (4 ints per task): first every CTA row and split segment in row
 * order -- {1, row, 0, 0} or {2, row, segment, slot}, slots numbered
 * 0,1,2,... in that order -- then every group in row order:
 * {0 + 256*c, first row, end row (exclusive), 0}.
 * Long-row table (4 ints per split row, row order): {row, first slot, #segments, 0}.
 * counts_out = {#tasks, #long rows, #slots, #rows packed, #CTA rows, #split rows,
 *               #groups with c == 0, #groups with 1 <= c <= 5, #groups with c == 6}.
 * Pass tasks/longrows == NULL to only count.
 */
int or_plan_spmv(int32_t M, const int32_t* rp, const or_plan_opts_t* o, int32_t* tasks, int32_t* longrows,
                 int64_t* counts_out) {
    if (M < 0 || !o || !counts_out) return OR_ERR_ARG;
    if (o->block_nnz < 1 || o->block_rows < 1 || o->pack_max < 0 || o->pack_max > o->block_nnz ||
        o->cta_max < o->pack_max || o->seg_nnz < 1 || o->lanes_div < 0)
        return OR_ERR_ARG;
    int64_t nt = 0, nl = 0, slot = 0, npacked = 0, ncta = 0, nsplit = 0, g1 = 0, gw = 0, gs = 0;
    /* pass 1: CTA rows and segments */
    for (int32_t i = 0; i < M; ++i) {
        int64_t l = (int64_t)rp[i + 1] - rp[i];
        if (l <= o->pack_max) continue;
        if (l <= o->cta_max) {
            if (tasks) { int32_t* t = tasks + 4 * nt; t[0] = OR_TASK_CTA; t[1] = i; t[2] = 0; t[3] = 0; }
            ++nt; ++ncta;
        } else {
            int64_t ns = (l + o->seg_nnz - 1) / o->seg_nnz;
            if (longrows) { int32_t* t = longrows + 4 * nl; t[0] = i; t[1] = (int32_t)slot; t[2] = (int32_t)ns; t[3] = 0; }
            for (int64_t s = 0; s < ns; ++s) {
                if (tasks) { int32_t* t = tasks + 4 * nt; t[0] = OR_TASK_SEG; t[1] = i; t[2] = (int32_t)s; t[3] = (int32_t)(slot + s); }
                ++nt;
            }
            slot += ns; ++nl; ++nsplit;
        }
    }
    /* pass 2: groups of packed rows */
    int32_t i = 0;
    while (i < M) {
        int64_t l = (int64_t)rp[i + 1] - rp[i];
        if (l > o->pack_max) { ++i; continue; }
        int32_t r0 = i;
        int64_t gnnz = 0;
        while (i < M) {
            int64_t li = (int64_t)rp[i + 1] - rp[i];
            if (li > o->pack_max) break;
            if (i - r0 >= o->block_rows) break;
            if (gnnz + li > o->block_nnz) break;
            gnnz += li;
            ++i;
        }
        int64_t rows = i - r0;
        int32_t c = 6;
        if (o->lanes_div > 0) {
            int64_t per = (gnnz + rows * o->lanes_div - 1) / (rows * o->lanes_div);
            int32_t w = pow2ceil_clamp32(per);
            c = 0;
            while ((1 << c) < w) ++c;
        }
        if (tasks) { int32_t* t = tasks + 4 * nt; t[0] = OR_TASK_GROUP + 256 * c; t[1] = r0; t[2] = i; t[3] = 0; }
        ++nt;
        npacked += rows;
        if (c == 0) ++g1; else if (c == 6) ++gs; else ++gw;
    }
    counts_out[0] = nt; counts_out[1] = nl; counts_out[2] = slot; counts_out[3] = npacked;
    counts_out[4] = ncta; counts_out[5] = nsplit; counts_out[6] = g1; counts_out[7] = gw; counts_out[8] = gs;
    return OR_OK;
}

/* ------------------------------------------------------------------ SpMV */

/*
 * y_i = alpha * sum_p val_p * x[col_p] + beta * y_i over the stored entries of
 * row i, in fp64 and in p order.  [SpMM-ops] §2.1 (the per-row loop over
 * [row_offsets[i], row_offsets[i+1])), [LSMR-dual] §2 ((Av)_i as that sum) and
 * §5.2 (alpha/beta as in the library call: beta scales the old output; with
 * beta == 0 the old output is not read).  bound_i = |alpha| * sum |val_p x_col|
 * + |beta * y_i| is the scale the tolerance is measured against.
 * rows == NULL: all M rows; otherwise only rows[0..nrows) (output index k).
 */
int or_spmv(int32_t M, const int32_t* rp, const int32_t* col, const float* val, const float* x, double alpha,
            double beta, const float* y_in, const int32_t* rows, int64_t nrows, double* ref, double* bound) {
    if (M < 0) return OR_ERR_ARG;
    int64_t n = rows ? nrows : M;
    for (int64_t k = 0; rows && k < n; ++k)
        if (rows[k] < 0 || rows[k] >= M) return OR_ERR_INDEX;
    /* rows are independent: the all-core build (-fopenmp) hands them out to
       threads; every row is still summed alone, in p order */
#pragma omp parallel for schedule(dynamic, 256)
    for (int64_t k = 0; k < n; ++k) {
        int32_t i = rows ? rows[k] : (int32_t)k;
        double acc = 0.0, mag = 0.0;
        for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
            double t = (double)val[p] * (double)x[col[p]];
            acc += t;
            mag += fabs(t);
        }
        double r = alpha * acc, b = fabs(alpha) * mag;
        if (beta != 0.0) {
            r += beta * (double)y_in[i];
            b += fabs(beta * (double)y_in[i]);
        }
        ref[k] = r;
        if (bound) bound[k] = b;
    }
    return OR_OK;
}

/*
 * The same product summed the way a plain fp32 loop would: each product
 * val_p * x[col_p] rounded to fp32, added in p order to an fp32 running sum
 * (no fused multiply-add), then y_i = alpha * sum + beta * y_i in fp32.
 * [SpMM-ops] §5 (check a lower-precision result against a higher-precision
 * reference and report the error): this is the low-precision side.  Its
 * distance to or_spmv obeys the textbook bound for a recursively summed dot
 * product of length l, |fl(s) - s| <= gamma_l * sum |val_p x_col_p| with
 * gamma_l = l u / (1 - l u), u = 2^-24, which the tests check.
 */
int or_spmv_f32(int32_t M, const int32_t* rp, const int32_t* col, const float* val, const float* x, float alpha,
                float beta, const float* y_in, const int32_t* rows, int64_t nrows, float* out) {
    if (M < 0) return OR_ERR_ARG;
    int64_t n = rows ? nrows : M;
    for (int64_t k = 0; rows && k < n; ++k)
        if (rows[k] < 0 || rows[k] >= M) return OR_ERR_INDEX;
    for (int64_t k = 0; k < n; ++k) {
        int32_t i = rows ? rows[k] : (int32_t)k;
        float acc = 0.0f;
        for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
            float t = val[p] * x[col[p]];
            acc = acc + t;
        }
        float r = alpha * acc;
        if (beta != 0.0f) r = r + beta * y_in[i];
        out[k] = r;
    }
    return OR_OK;
}

/*
 * COO SpMV: y_i = alpha * sum over the triplets p with row_p == i of
 * val_p * x[col_p] + beta * y_i, fp64, triplets taken in index order.
 * [Formats] §1 (COO stores one (row, col, val) triplet per entry; the product
 * visits each triplet once and adds it to its row).  Rows without triplets
 * give beta * y_i (0 when beta == 0; y_in is then not read).  The triplets
 * need not be sorted here.  bound as in or_spmv.
 */
int or_spmv_coo(int32_t M, int32_t K, int64_t nnz, const int32_t* row, const int32_t* col, const float* val,
                const float* x, double alpha, double beta, const float* y_in, double* ref, double* bound) {
    if (M < 0 || K < 0 || nnz < 0) return OR_ERR_ARG;
    double* mag = (double*)calloc((size_t)(M ? M : 1), sizeof(double));
    if (!mag) return OR_ERR_NOMEM;
    for (int32_t i = 0; i < M; ++i) ref[i] = 0.0;
    for (int64_t p = 0; p < nnz; ++p) {
        if (row[p] < 0 || row[p] >= M || col[p] < 0 || col[p] >= K) {
            free(mag);
            return OR_ERR_INDEX;
        }
        double t = (double)val[p] * (double)x[col[p]];
        ref[row[p]] += t;
        mag[row[p]] += fabs(t);
    }
    for (int32_t i = 0; i < M; ++i) {
        double r = alpha * ref[i], b = fabs(alpha) * mag[i];
        if (beta != 0.0) {
            r += beta * (double)y_in[i];
            b += fabs(beta * (double)y_in[i]);
        }
        ref[i] = r;
        if (bound) bound[i] = b;
    }
    free(mag);
    return OR_OK;
}

/*
 * SELL-C-sigma with C = 32.  [SpMM-ops] §1.4 and [Formats] §6 (sliced
 * ELLPACK: sort rows by length inside windows of sigma rows, cut slices of C
 * rows, pad each slice to its longest row, store the slice column-major).
 * Rows longer than `piece` are first cut into pieces of `piece` entries (the
 * last one shorter); every row or piece is a "pseudo-row", listed in row
 * order (pieces in piece order).  Inside each window of sigma pseudo-rows the
 * pseudo-rows are emitted longest first, equal lengths in their listed order:
 * here by sweeping the lengths from the window's maximum down to 0 and
 * emitting each match in list order (no sort routine).  Layout: entry j of
 * lane r of slice s at slice_ptr[s] + 32 j + r; padding col -1, val 0.
 * prow: the row, or -1 - slot for a piece (slots numbered in listing order),
 * INT32_MIN for unused lanes of the last slice.  longrows: {row, first slot,
 * #pieces, 0} per cut row.  Two calls: with scol == NULL only the sizes
 * (npseudo, nslices, padded, nlong) are produced.
 */
int or_build_sell(int32_t M, const int32_t* rp, const int32_t* col, const float* val, int32_t sigma, int32_t piece,
                  int64_t* npseudo, int64_t* nslices, int64_t* padded, int64_t* nlong, int32_t* slice_ptr,
                  int32_t* prow, int32_t* longrows, int32_t* scol, float* sval) {
    if (M < 0 || sigma < 32 || sigma % 32 || piece < 1) return OR_ERR_ARG;
    int64_t np = 0, nl = 0;
    for (int32_t i = 0; i < M; ++i) {
        int32_t l = rp[i + 1] - rp[i];
        if (l > piece) {
            np += (l + piece - 1) / piece;
            ++nl;
        } else {
            ++np;
        }
    }
    /* the listing: (len, row, start, slot) */
    int32_t* L = (int32_t*)malloc(sizeof(int32_t) * (size_t)(4 * (np ? np : 1)));
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(np ? np : 1));
    if (!L || !order) {
        free(L);
        free(order);
        return OR_ERR_NOMEM;
    }
    int64_t q = 0, slot = 0, li = 0;
    for (int32_t i = 0; i < M; ++i) {
        int32_t l = rp[i + 1] - rp[i];
        if (l <= piece) {
            L[4 * q] = l; L[4 * q + 1] = i; L[4 * q + 2] = rp[i]; L[4 * q + 3] = -1;
            ++q;
            continue;
        }
        int32_t n = (l + piece - 1) / piece;
        if (longrows) {
            longrows[4 * li] = i; longrows[4 * li + 1] = (int32_t)slot; longrows[4 * li + 2] = n;
            longrows[4 * li + 3] = 0;
        }
        ++li;
        for (int32_t k = 0; k < n; ++k) {
            int32_t len = l - k * piece < piece ? l - k * piece : piece;
            L[4 * q] = len; L[4 * q + 1] = i; L[4 * q + 2] = rp[i] + k * piece; L[4 * q + 3] = (int32_t)(slot + k);
            ++q;
        }
        slot += n;
    }
    /* window order: lengths swept from the maximum down, list order within a length */
    int64_t o = 0;
    for (int64_t w0 = 0; w0 < np; w0 += sigma) {
        int64_t w1 = w0 + sigma < np ? w0 + sigma : np;
        int32_t mx = 0;
        for (int64_t p = w0; p < w1; ++p) if (L[4 * p] > mx) mx = L[4 * p];
        for (int32_t len = mx; len >= 0; --len)
            for (int64_t p = w0; p < w1; ++p)
                if (L[4 * p] == len) order[o++] = p;
    }
    int64_t ns = (np + 31) / 32, pad = 0;
    for (int64_t s = 0; s < ns; ++s) {
        int32_t mx = 0;
        for (int64_t r = 0; r < 32 && s * 32 + r < np; ++r) {
            int32_t len = L[4 * order[s * 32 + r]];
            if (len > mx) mx = len;
        }
        if (slice_ptr) slice_ptr[s] = (int32_t)pad;
        pad += 32 * (int64_t)mx;
    }
    if (slice_ptr) slice_ptr[ns] = (int32_t)pad;
    *npseudo = np; *nslices = ns; *padded = pad; *nlong = nl;
    if (scol && sval && prow && slice_ptr) {
        for (int64_t e = 0; e < pad; ++e) { scol[e] = -1; sval[e] = 0.0f; }
        for (int64_t t = 0; t < 32 * ns; ++t) {
            if (t >= np) { prow[t] = INT32_MIN; continue; }
            const int32_t* d = L + 4 * order[t];
            prow[t] = d[3] < 0 ? d[1] : -1 - d[3];
            int64_t s = t / 32, r = t % 32;
            for (int32_t j = 0; j < d[0]; ++j) {
                scol[slice_ptr[s] + 32 * (int64_t)j + r] = col[d[2] + j];
                sval[slice_ptr[s] + 32 * (int64_t)j + r] = val[d[2] + j];
            }
        }
    }
    free(L);
    free(order);
    return OR_OK;
}

/*
 * CSR -> WCSR with windows of 64 rows.  [AsyncSparse] §2.2.2 (rows grouped
 * into fixed-height windows; a window keeps the union of the columns its rows
 * use, window_col_idx with -1 for padding, and the values of those columns
 * as a dense block).  Here: the union of window w is found by marking the
 * columns its entries use and scanning the columns upward (so it comes out
 * ascending), padded with -1 to a multiple of 64, and cut into chunks of 64
 * positions; chunk values are a 64 x 64 row-major block (row r of the window,
 * position k), zero where the row has no entry there.  A repeated (row, col)
 * would need two values in one slot: OR_ERR_DUP.  Two calls: with
 * win_col == NULL only the chunk count (and win_ptr) is produced.
 */
int or_build_wcsr(int32_t M, int32_t K, const int32_t* rp, const int32_t* col, const void* val, int32_t vbytes,
                  int32_t* win_ptr, int32_t* win_col, void* win_val, int64_t* nchunks, double* fill) {
    if (M < 0 || K < 0 || vbytes <= 0) return OR_ERR_ARG;
    int64_t W = ((int64_t)M + 63) / 64;
    unsigned char* mark = (unsigned char*)calloc((size_t)(K ? K : 1), 1);
    int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K ? K : 1));
    unsigned char* used = (unsigned char*)malloc(64 * 64);
    if (!mark || !pos || !used) {
        free(mark); free(pos); free(used);
        return OR_ERR_NOMEM;
    }
    int64_t g = 0;
    int rc = OR_OK;
    if (win_ptr) win_ptr[0] = 0;
    for (int64_t w = 0; w < W && rc == OR_OK; ++w) {
        int64_t r0 = w * 64, r1 = r0 + 64 < M ? r0 + 64 : M;
        for (int64_t p = rp[r0]; p < rp[r1]; ++p) {
            if (col[p] < 0 || col[p] >= K) { rc = OR_ERR_INDEX; break; }
            mark[col[p]] = 1;
        }
        if (rc != OR_OK) break;
        int64_t n = 0;
        for (int32_t c = 0; c < K; ++c)
            if (mark[c]) pos[c] = (int32_t)(n++);
        int64_t nch = (n + 63) / 64;
        if (win_col) {
            int64_t k = 0;
            for (int32_t c = 0; c < K; ++c)
                if (mark[c]) win_col[g * 64 + k++] = c;
            for (; k < nch * 64; ++k) win_col[g * 64 + k] = -1;
            memset((char*)win_val + g * 4096 * vbytes, 0, (size_t)(nch * 4096 * vbytes));
        }
        for (int64_t ch = 0; ch < nch && rc == OR_OK; ++ch) {
            memset(used, 0, 64 * 64);
            for (int64_t i = r0; i < r1 && rc == OR_OK; ++i)
                for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
                    int64_t k = pos[col[p]];
                    if (k / 64 != ch) continue;
                    int64_t slot = (i - r0) * 64 + k % 64;
                    if (used[slot]) { rc = OR_ERR_DUP; break; }
                    used[slot] = 1;
                    if (win_val)
                        memcpy((char*)win_val + ((g + ch) * 4096 + slot) * vbytes, (const char*)val + p * vbytes,
                               (size_t)vbytes);
                }
        }
        for (int64_t p = rp[r0]; p < rp[r1]; ++p) mark[col[p]] = 0;
        g += nch;
        if (win_ptr) win_ptr[w + 1] = (int32_t)g;
    }
    free(mark); free(pos); free(used);
    if (rc != OR_OK) return rc;
    *nchunks = g;
    if (fill) *fill = g ? (double)rp[M] / ((double)g * 4096.0) : 0.0;
    return OR_OK;
}

/* ------------------------------------------------------------------ SpMM */

/*
 * C_{i,n} = alpha * sum_{k in N(i)} A_{ik} B_{k,n} + beta * C_{i,n}, fp64, p
 * order.  [SpMM-ops] §3 (the SpMM sum over the stored columns of row i).
 * B is K x N row-major with leading dimension ldb, C likewise with ldc; ref
 * and bound are (#rows x N) dense with leading dimension N.
 */
int or_spmm(int32_t M, int32_t N, const int32_t* rp, const int32_t* col, const float* val, const float* B,
            int64_t ldb, double alpha, double beta, const float* C_in, int64_t ldc, const int32_t* rows,
            int64_t nrows, double* ref, double* bound) {
    if (M < 0 || N < 0) return OR_ERR_ARG;
    int64_t n = rows ? nrows : M;
    for (int64_t k = 0; rows && k < n; ++k)
        if (rows[k] < 0 || rows[k] >= M) return OR_ERR_INDEX;
    int err = OR_OK;
    /* rows are independent: the all-core build (-fopenmp) hands them out to
       threads, each with its own accumulators */
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)(2 * (N ? N : 1)));
        double* mag = acc ? acc + N : NULL;
#pragma omp for schedule(dynamic, 16)
        for (int64_t k = 0; k < n; ++k) {
            if (!acc) { err = OR_ERR_NOMEM; continue; }
            int32_t i = rows ? rows[k] : (int32_t)k;
            for (int32_t c = 0; c < N; ++c) { acc[c] = 0.0; mag[c] = 0.0; }
            for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
                double a = (double)val[p];
                const float* brow = B + (int64_t)col[p] * ldb;
                for (int32_t c = 0; c < N; ++c) {
                    double t = a * (double)brow[c];
                    acc[c] += t;
                    mag[c] += fabs(t);
                }
            }
            for (int32_t c = 0; c < N; ++c) {
                double r = alpha * acc[c], b = fabs(alpha) * mag[c];
                if (beta != 0.0) {
                    double y = (double)C_in[(int64_t)i * ldc + c];
                    r += beta * y;
                    b += fabs(beta * y);
                }
                ref[k * N + c] = r;
                if (bound) bound[k * N + c] = b;
            }
        }
        free(acc);
    }
    return err;
}

/* -------------------------------------------------------------- BSR SpMM */

static double bf16_to_double(uint16_t h) {
    uint32_t b = (uint32_t)h << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
}

/*
 * C = A * B with A in BSR (br x bc row-major blocks, bf16) and B a K x N bf16
 * row-major matrix; fp64 sums in block order, then column order inside the
 * block.  [SpMM-ops] §3.4 (outer loop over the nonzero blocks, a small dense
 * product inside) and [AsyncSparse] §3 (BCSR SpMM, each block a dense
 * micro-GEMM against the B rows of its block column).  Padded block columns
 * beyond K contribute nothing.  ref = alpha * sum + beta * C_in (C_in read only
 * when beta != 0, fp32, leading dimension ldc); bound = |alpha| * sum |a b| +
 * |beta * C_in|.  ref/bound: (#rows x N), leading dimension N.
 */
int or_bsr_spmm(int32_t M, int32_t K, int32_t br, int32_t bc, const int32_t* bsr_rp, const int32_t* bcol,
                const uint16_t* bval, int32_t N, const uint16_t* B, int64_t ldb, double alpha, double beta,
                const float* C_in, int64_t ldc, const int32_t* rows, int64_t nrows, double* ref, double* bound) {
    if (M < 0 || K < 0 || N < 0 || br <= 0 || bc <= 0) return OR_ERR_ARG;
    int64_t n = rows ? nrows : M;
    for (int64_t k = 0; rows && k < n; ++k)
        if (rows[k] < 0 || rows[k] >= M) return OR_ERR_INDEX;
    int err = OR_OK;
    /* rows are independent: the all-core build (-fopenmp) hands them out to
       threads, each with its own accumulators */
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)(2 * (N ? N : 1)));
        double* mag = acc ? acc + N : NULL;
#pragma omp for schedule(dynamic, 4)
        for (int64_t k = 0; k < n; ++k) {
            if (!acc) { err = OR_ERR_NOMEM; continue; }
            int32_t i = rows ? rows[k] : (int32_t)k;
            int32_t I = i / br, r = i % br;
            for (int32_t c = 0; c < N; ++c) { acc[c] = 0.0; mag[c] = 0.0; }
            for (int64_t blk = bsr_rp[I]; blk < bsr_rp[I + 1]; ++blk) {
                const uint16_t* arow = bval + blk * (int64_t)br * bc + (int64_t)r * bc;
                for (int32_t cc = 0; cc < bc; ++cc) {
                    int64_t kk = (int64_t)bcol[blk] * bc + cc;
                    if (kk >= K) break;
                    double a = bf16_to_double(arow[cc]);
                    const uint16_t* brow = B + kk * ldb;
                    for (int32_t c = 0; c < N; ++c) {
                        double t = a * bf16_to_double(brow[c]);
                        acc[c] += t;
                        mag[c] += fabs(t);
                    }
                }
            }
            for (int32_t c = 0; c < N; ++c) {
                double rr = alpha * acc[c], b = fabs(alpha) * mag[c];
                if (beta != 0.0) {
                    double y = (double)C_in[(int64_t)i * ldc + c];
                    rr += beta * y;
                    b += fabs(beta * y);
                }
                ref[k * N + c] = rr;
                if (bound) bound[k * N + c] = b;
            }
        }
        free(acc);
    }
    return err;
}

/*
 * Threads of the all-core build: the same source compiled with -fopenmp runs
 * the row loops above on `threads` host threads (rows are independent, so no
 * result changes).  The single-thread build ignores the request and reports 1.
 */
int or_threads(int32_t threads) {
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
    return omp_get_max_threads();
#else
    (void)threads;
    return 1;
#endif
}
