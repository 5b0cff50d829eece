// spx_host.cpp -- host side of libspx: status strings, the format builders,
// row statistics, the dispatch plan and argument validation.
//
// Builders are O(nnz) counting sorts ([Formats] §3: histogram, prefix sum,
// scatter); the plan follows [SpMM-ops] §2.1-§2.4 and §4.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <new>

#include <cuda_runtime.h>

#include "spx_internal.h"

// mean, population variance and cv from the exact sums (one definition for
// the host and the device statistics, so both give the same doubles)
void spx_row_stats_finish(int32_t M, spx_row_stats_t* out) {
    const int64_t s1 = out->nnz, s2 = out->sumsq;
    out->mean = static_cast<double>(s1) / static_cast<double>(M);
    __int128 num = static_cast<__int128>(M) * s2 - static_cast<__int128>(s1) * s1;
    out->var = static_cast<double>(num) / (static_cast<double>(M) * static_cast<double>(M));
    out->cv = out->mean > 0.0 ? std::sqrt(out->var) / out->mean : 0.0;
}

namespace {

std::atomic<uint64_t> g_launches{0};

// Copies `bytes` from device memory to a host vector (synchronises `stream`).
template <class T>
spx_status to_host(std::vector<T>& dst, const T* src, int64_t n, cudaStream_t stream) {
    try {
        dst.resize(static_cast<size_t>(n));
    } catch (const std::bad_alloc&) {
        return SPX_ERR_NOMEM;
    }
    if (n == 0) return SPX_OK;
    cudaError_t e = cudaMemcpyAsync(dst.data(), src, sizeof(T) * static_cast<size_t>(n), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return e == cudaSuccess ? SPX_OK : SPX_ERR_CUDA;
}

spx_status to_device(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
    if (bytes == 0) return SPX_OK;
    cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return e == cudaSuccess ? SPX_OK : SPX_ERR_CUDA;
}

bool bad_vbytes(int32_t vb) { return !(vb == 1 || vb == 2 || vb == 4 || vb == 8); }

// ---------------------------------------------------------------- COO -> CSR
spx_status build_csr_host(int32_t M, int32_t K, int64_t nnz, const int32_t* row, const int32_t* col,
                          const char* val, int32_t vb, int32_t* rp, int32_t* col_out, char* val_out) {
    for (int64_t p = 0; p < nnz; ++p)
        if (row[p] < 0 || row[p] >= M || col[p] < 0 || col[p] >= K) return SPX_ERR_INDEX_RANGE;
    std::vector<int64_t> cnt(static_cast<size_t>(M) + 1, 0);
    for (int64_t p = 0; p < nnz; ++p) cnt[static_cast<size_t>(row[p]) + 1]++;   // histogram
    for (int32_t i = 0; i < M; ++i) cnt[i + 1] += cnt[i];                         // prefix sum
    for (int32_t i = 0; i <= M; ++i) rp[i] = static_cast<int32_t>(cnt[i]);
    std::vector<int32_t> src(static_cast<size_t>(nnz));
    std::vector<int64_t> cur(cnt.begin(), cnt.end() - 1);
    for (int64_t p = 0; p < nnz; ++p) src[static_cast<size_t>(cur[row[p]]++)] = static_cast<int32_t>(p);  // stable scatter
    // inside each row, order by column; stable, so equal columns keep input order
    for (int32_t i = 0; i < M; ++i) {
        auto b = src.begin() + rp[i], e = src.begin() + rp[i + 1];
        bool sorted = true;
        for (auto it = b; it + 1 < e; ++it)
            if (col[*(it + 1)] < col[*it]) { sorted = false; break; }
        if (!sorted) std::stable_sort(b, e, [&](int32_t a, int32_t c) { return col[a] < col[c]; });
    }
    for (int64_t q = 0; q < nnz; ++q) {
        int64_t p = src[static_cast<size_t>(q)];
        col_out[q] = col[p];
        std::memcpy(val_out + q * vb, val + p * vb, static_cast<size_t>(vb));
    }
    return SPX_OK;
}

spx_status check_rp(int32_t M, int64_t nnz, const int32_t* rp) {
    if (rp[0] != 0 || rp[M] != nnz) return SPX_ERR_ARG;
    for (int32_t i = 0; i < M; ++i)
        if (rp[i + 1] < rp[i]) return SPX_ERR_NOT_SORTED;
    return SPX_OK;
}

// ------------------------------------------------------------ CSR -> CSR(A^T)
spx_status transpose_host(int32_t M, int32_t K, int64_t nnz, const int32_t* rp, const int32_t* col, const char* val,
                          int32_t vb, int32_t* trp, int32_t* tcol, char* tval) {
    spx_status s = check_rp(M, nnz, rp);
    if (s != SPX_OK) return s;
    for (int64_t p = 0; p < nnz; ++p)
        if (col[p] < 0 || col[p] >= K) return SPX_ERR_INDEX_RANGE;
    std::vector<int64_t> cnt(static_cast<size_t>(K) + 1, 0);
    for (int64_t p = 0; p < nnz; ++p) cnt[static_cast<size_t>(col[p]) + 1]++;
    for (int32_t j = 0; j < K; ++j) cnt[j + 1] += cnt[j];
    for (int32_t j = 0; j <= K; ++j) trp[j] = static_cast<int32_t>(cnt[j]);
    // rows visited upward: each output row receives its entries in source-row order
    for (int32_t i = 0; i < M; ++i)
        for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
            int64_t q = cnt[col[p]]++;
            tcol[q] = i;
            std::memcpy(tval + q * vb, val + p * vb, static_cast<size_t>(vb));
        }
    return SPX_OK;
}

// ------------------------------------------------------------ CSR -> BSR
spx_status build_bsr_host(int32_t M, int32_t K, const int32_t* rp, const int32_t* col, const char* val, int32_t vb,
                          int32_t br, int32_t bc, int32_t* brp, int32_t* bcol, char* bval, int64_t* nnzb_out,
                          double* fill_out) {
    spx_status s = check_rp(M, rp[M], rp);
    if (s != SPX_OK) return s;
    const int64_t MB = (static_cast<int64_t>(M) + br - 1) / br;
    const int64_t KB = (static_cast<int64_t>(K) + bc - 1) / bc;
    const int64_t blk = static_cast<int64_t>(br) * bc;
    std::vector<int32_t> slot_of(static_cast<size_t>(KB), -1);  // block column -> slot in this block-row
    std::vector<int32_t> cols;
    std::vector<uint8_t> seen;
    int64_t nb = 0;
    if (brp) brp[0] = 0;
    for (int64_t I = 0; I < MB; ++I) {
        const int64_t r0 = I * br, r1 = std::min<int64_t>(r0 + br, M);
        cols.clear();
        for (int64_t p = rp[r0]; p < rp[r1]; ++p) {
            if (col[p] < 0 || col[p] >= K) return SPX_ERR_INDEX_RANGE;
            int32_t J = col[p] / bc;
            if (slot_of[J] < 0) { slot_of[J] = 0; cols.push_back(J); }
        }
        std::sort(cols.begin(), cols.end());
        for (size_t t = 0; t < cols.size(); ++t) slot_of[cols[t]] = static_cast<int32_t>(t);
        seen.assign(cols.size() * static_cast<size_t>(blk), 0);
        for (int64_t i = r0; i < r1; ++i)
            for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
                int64_t off = static_cast<int64_t>(slot_of[col[p] / bc]) * blk + (i - r0) * bc + col[p] % bc;
                if (seen[off]) {
                    for (int32_t J : cols) slot_of[J] = -1;
                    return SPX_ERR_DUPLICATE;
                }
                seen[off] = 1;
            }
        if (bcol && bval) {
            for (size_t t = 0; t < cols.size(); ++t) {
                bcol[nb + static_cast<int64_t>(t)] = cols[t];
                std::memset(bval + (nb + static_cast<int64_t>(t)) * blk * vb, 0, static_cast<size_t>(blk * vb));
            }
            for (int64_t i = r0; i < r1; ++i)
                for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
                    int64_t b = nb + slot_of[col[p] / bc];
                    std::memcpy(bval + (b * blk + (i - r0) * bc + col[p] % bc) * vb, val + p * vb,
                                static_cast<size_t>(vb));
                }
        }
        for (int32_t J : cols) slot_of[J] = -1;
        nb += static_cast<int64_t>(cols.size());
        if (nb > kI32Max) return SPX_ERR_INDEX_RANGE;
        if (brp) brp[I + 1] = static_cast<int32_t>(nb);
    }
    if (nnzb_out) *nnzb_out = nb;
    if (fill_out) *fill_out = nb ? static_cast<double>(rp[M]) / (static_cast<double>(nb) * br * bc) : 0.0;
    return SPX_OK;
}

// ------------------------------------------------------------ statistics
void row_stats_host(int32_t M, const int32_t* rp, spx_row_stats_t* out) {
    std::memset(out, 0, sizeof(*out));
    out->rows = M;
    if (M == 0) return;
    std::vector<int32_t> len(static_cast<size_t>(M));
    int64_t s1 = 0, s2 = 0;
    int32_t empty = 0;
    for (int32_t i = 0; i < M; ++i) {
        int32_t l = rp[i + 1] - rp[i];
        len[i] = l;
        s1 += l;
        s2 += static_cast<int64_t>(l) * l;
        empty += (l == 0);
    }
    auto kth = [&](int64_t rank) {  // rank-th smallest, 1-based
        std::nth_element(len.begin(), len.begin() + (rank - 1), len.end());
        return len[static_cast<size_t>(rank - 1)];
    };
    out->nnz = s1;
    out->sumsq = s2;
    out->empty = empty;
    out->p50 = kth((50LL * M + 99) / 100);
    out->p95 = kth((95LL * M + 99) / 100);
    out->p99 = kth((99LL * M + 99) / 100);
    out->min = *std::min_element(len.begin(), len.end());
    out->max = *std::max_element(len.begin(), len.end());
    spx_row_stats_finish(M, out);
}

// ------------------------------------------------------------ the plan
int32_t reduce_code(int64_t nnz_g, int64_t rows_g, int32_t div) {
    if (div == 0) return kReduceSegmented;
    int64_t per = (nnz_g + rows_g * div - 1) / (rows_g * div);
    int32_t lg = 0;
    while (lg < 5 && (int64_t{1} << lg) < per) ++lg;
    return lg;  // log2 of the lanes per row
}

spx_status make_plan(spx_plan* P, const int32_t* rp) {
    const spx_plan_opts_t& o = P->opts;
    const int32_t M = P->M;
    std::vector<int32_t> groups, dgroups;
    int64_t slot = 0, ncta = 0, nsplit = 0, npacked = 0, g1 = 0, gw = 0, gs = 0;
    int32_t d[4];
    auto push = [](std::vector<int32_t>& v, const int32_t* q) { v.insert(v.end(), q, q + 4); };
    int32_t i = 0;
    while (i < M) {
        int64_t l = static_cast<int64_t>(rp[i + 1]) - rp[i];
        if (l > o.pack_max) {
            if (l <= o.cta_max) {
                P->tasks.insert(P->tasks.end(), {kTaskCta, i, 0, 0});
                spx_dev_task(d, kTaskCta, 0, 0, i, rp[i], rp[i + 1]);
                push(P->dtasks, d);
                ++ncta;
            } else {
                int64_t ns = (l + o.seg_nnz - 1) / o.seg_nnz;
                if (slot + ns > (int64_t{1} << 23)) return SPX_ERR_INDEX_RANGE;  // slot must fit the task word
                P->longrows.insert(P->longrows.end(), {i, static_cast<int32_t>(slot), static_cast<int32_t>(ns), 0});
                for (int64_t sg = 0; sg < ns; ++sg) {
                    P->tasks.insert(P->tasks.end(), {kTaskSeg, i, static_cast<int32_t>(sg), static_cast<int32_t>(slot + sg)});
                    int64_t lo = rp[i] + sg * o.seg_nnz, hi = std::min<int64_t>(rp[i + 1], lo + o.seg_nnz);
                    spx_dev_task(d, kTaskSeg, 0, static_cast<int32_t>(slot + sg), i, static_cast<int32_t>(lo),
                                 static_cast<int32_t>(hi));
                    push(P->dtasks, d);
                }
                slot += ns;
                ++nsplit;
            }
            ++i;
            continue;
        }
        // grow a group of packed rows
        const int32_t r0 = i;
        int64_t g = 0;
        while (i < M && i - r0 < o.block_rows) {
            int64_t li = static_cast<int64_t>(rp[i + 1]) - rp[i];
            if (li > o.pack_max || g + li > o.block_nnz) break;
            g += li;
            ++i;
        }
        const int32_t c = reduce_code(g, i - r0, o.lanes_div);
        groups.insert(groups.end(), {kTaskGroup + 256 * c, r0, i, 0});
        spx_dev_task(d, kTaskGroup, c, i - r0, r0, rp[r0], rp[i]);
        push(dgroups, d);
        npacked += i - r0;
        (c == 0 ? g1 : c == kReduceSegmented ? gs : gw) += 1;
    }
    if (o.lanes_div == 0) {
        // segmented groups: each thread's first row, one walk over the group's rows
        const int32_t nth = spx_group_threads(o.block_nnz), per = spx_group_per(o.block_nnz);
        P->first.assign(groups.size() / 4 * static_cast<size_t>(nth), 0);
        uint16_t* f = P->first.data();
        for (size_t k = 0; k < groups.size(); k += 4, f += nth) {
            const int32_t r0 = groups[k + 1], r1 = groups[k + 2], p0 = rp[r0], n = rp[r1] - p0;
            int32_t r = 0;
            for (int32_t t = 0; t < nth && static_cast<int64_t>(t) * per < n; ++t) {  // past the products: 0
                const int32_t a = t * per;
                while (rp[r0 + r + 1] - p0 <= a) ++r;
                f[t] = spx_first_entry(r, rp[r0 + r] - p0 < a);
            }
        }
    }
    P->tasks.insert(P->tasks.end(), groups.begin(), groups.end());
    P->dtasks.insert(P->dtasks.end(), dgroups.begin(), dgroups.end());
    const int64_t nt = static_cast<int64_t>(P->tasks.size() / 4);
    if (nt > kI32Max) return SPX_ERR_INDEX_RANGE;
    int64_t c[9] = {nt, static_cast<int64_t>(P->longrows.size() / 4), slot, npacked, ncta, nsplit, g1, gw, gs};
    std::memcpy(P->counts, c, sizeof(c));
    P->table_bytes = (P->dtasks.size() + P->longrows.size()) * sizeof(int32_t) + P->first.size() * sizeof(uint16_t);
    P->scratch_bytes = static_cast<size_t>(slot) * sizeof(float);
    return SPX_OK;
}

}  // namespace

// =================================================================== C ABI
extern "C" {

const char* spx_status_string(spx_status s) {
    switch (s) {
        case SPX_OK: return "SPX_OK";
        case SPX_ERR_ARG: return "SPX_ERR_ARG: invalid argument";
        case SPX_ERR_INDEX_RANGE: return "SPX_ERR_INDEX_RANGE: size or index out of range (int32 or matrix bounds)";
        case SPX_ERR_NOT_SORTED: return "SPX_ERR_NOT_SORTED: row_ptr not monotone or columns not ascending";
        case SPX_ERR_DUPLICATE: return "SPX_ERR_DUPLICATE: repeated (row, col)";
        case SPX_ERR_CUDA: return "SPX_ERR_CUDA: CUDA runtime error";
        case SPX_ERR_TIMEOUT: return "SPX_ERR_TIMEOUT: a bounded device wait expired";
        case SPX_ERR_UNSUPPORTED: return "SPX_ERR_UNSUPPORTED: no kernel for this shape/type";
        case SPX_ERR_ALIGN: return "SPX_ERR_ALIGN: misaligned pointer or leading dimension";
        case SPX_ERR_NOMEM: return "SPX_ERR_NOMEM: host allocation failed";
        case SPX_ERR_NOT_READY: return "SPX_ERR_NOT_READY: plan not uploaded";
        case SPX_ERR_SCRATCH_LIMIT:
            return "SPX_ERR_SCRATCH_LIMIT: the plan needs more partial-sum slots than the fixed no-alloc buffer holds";
    }
    return "unknown spx_status";
}

spx_status spx_launch_count(uint64_t* count) {
    if (!count) return SPX_ERR_ARG;
    *count = g_launches.load();
    return SPX_OK;
}

spx_status spx_build_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* coo_row, const int32_t* coo_col,
                         const void* coo_val, int32_t val_bytes, int32_t* row_ptr, int32_t* col, void* val,
                         spx_loc where, spx_stream_t stream) {
    if (M < 0 || K < 0 || nnz < 0 || bad_vbytes(val_bytes) || !row_ptr) return SPX_ERR_ARG;
    if (nnz > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (nnz > 0 && (!coo_row || !coo_col || !coo_val || !col || !val)) return SPX_ERR_ARG;
    if (where == SPX_HOST)
        return build_csr_host(M, K, nnz, coo_row, coo_col, static_cast<const char*>(coo_val), val_bytes, row_ptr, col,
                              static_cast<char*>(val));
    if (where != SPX_DEVICE) return SPX_ERR_ARG;
    return spx_dev_build_csr(M, K, nnz, coo_row, coo_col, coo_val, val_bytes, row_ptr, col, val, stream);
}

spx_status spx_transpose_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                             const void* val, int32_t val_bytes, int32_t* t_row_ptr, int32_t* t_col, void* t_val,
                             spx_loc where, spx_stream_t stream) {
    if (M < 0 || K < 0 || nnz < 0 || bad_vbytes(val_bytes) || !row_ptr || !t_row_ptr) return SPX_ERR_ARG;
    if (nnz > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (nnz > 0 && (!col || !val || !t_col || !t_val)) return SPX_ERR_ARG;
    if (where == SPX_HOST)
        return transpose_host(M, K, nnz, row_ptr, col, static_cast<const char*>(val), val_bytes, t_row_ptr, t_col,
                              static_cast<char*>(t_val));
    if (where != SPX_DEVICE) return SPX_ERR_ARG;
    return spx_dev_transpose_csr(M, K, nnz, row_ptr, col, val, val_bytes, t_row_ptr, t_col, t_val, stream);
}

spx_status spx_build_bsr(int32_t M, int32_t K, const int32_t* row_ptr, const int32_t* col, const void* val,
                         int32_t val_bytes, int32_t br, int32_t bc, int32_t* bsr_row_ptr, int32_t* bsr_col,
                         void* bsr_val, int64_t* nnzb_out, double* fill_out, spx_loc where, spx_stream_t stream) {
    if (M < 0 || K < 0 || br <= 0 || bc <= 0 || bad_vbytes(val_bytes) || !row_ptr) return SPX_ERR_ARG;
    if ((bsr_col == nullptr) != (bsr_val == nullptr)) return SPX_ERR_ARG;
    if (where == SPX_HOST) {
        if (row_ptr[M] > 0 && (!col || !val)) return SPX_ERR_ARG;
        return build_bsr_host(M, K, row_ptr, col, static_cast<const char*>(val), val_bytes, br, bc, bsr_row_ptr,
                              bsr_col, static_cast<char*>(bsr_val), nnzb_out, fill_out);
    }
    if (where != SPX_DEVICE) return SPX_ERR_ARG;
    return spx_dev_build_bsr(M, K, row_ptr, col, val, val_bytes, br, bc, bsr_row_ptr, bsr_col, bsr_val, nnzb_out,
                             fill_out, reinterpret_cast<cudaStream_t>(stream));
}

spx_status spx_check_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                         int32_t strict, spx_loc where, spx_stream_t stream) {
    if (M < 0 || K < 0 || nnz < 0 || !row_ptr || (nnz > 0 && !col)) return SPX_ERR_ARG;
    if (nnz > kI32Max) return SPX_ERR_INDEX_RANGE;
    std::vector<int32_t> rp_h, c_h;
    const int32_t* rp = row_ptr;
    const int32_t* c = col;
    if (where == SPX_DEVICE) {
        cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
        spx_status s = to_host(rp_h, row_ptr, static_cast<int64_t>(M) + 1, st);
        if (s == SPX_OK) s = to_host(c_h, col, nnz, st);
        if (s != SPX_OK) return s;
        rp = rp_h.data();
        c = c_h.data();
    } else if (where != SPX_HOST) {
        return SPX_ERR_ARG;
    }
    spx_status s = check_rp(M, nnz, rp);
    if (s != SPX_OK) return s;
    for (int32_t i = 0; i < M; ++i)
        for (int64_t p = rp[i]; p < rp[i + 1]; ++p) {
            if (c[p] < 0 || c[p] >= K) return SPX_ERR_INDEX_RANGE;
            if (strict && p > rp[i]) {
                if (c[p] == c[p - 1]) return SPX_ERR_DUPLICATE;
                if (c[p] < c[p - 1]) return SPX_ERR_NOT_SORTED;
            }
        }
    return SPX_OK;
}

spx_status spx_row_stats(int32_t M, const int32_t* row_ptr, spx_loc where, spx_row_stats_t* out) {
    if (M < 0 || !row_ptr || !out) return SPX_ERR_ARG;
    if (where == SPX_HOST) {
        row_stats_host(M, row_ptr, out);
        return SPX_OK;
    }
    if (where != SPX_DEVICE) return SPX_ERR_ARG;
    return spx_dev_row_stats(M, row_ptr, out, nullptr);
}

spx_status spx_plan_opts_default(spx_plan_opts_t* o) {
    if (!o) return SPX_ERR_ARG;
    o->block_nnz = 2048;
    o->block_rows = 256;
    o->pack_max = 512;
    o->cta_max = 8192;
    o->seg_nnz = 4096;
    o->lanes_div = 16;
    return SPX_OK;
}

spx_status spx_plan_opts_auto(const spx_row_stats_t* st, spx_plan_opts_t* o) {
    if (!st || !o) return SPX_ERR_ARG;
    spx_plan_opts_default(o);
    if (st->cv >= 2.0) {
        o->block_nnz = 1024;
        o->lanes_div = 0;
    }
    return SPX_OK;
}

static uint64_t rp_fingerprint_host(int32_t M, const int32_t* rp) {
    uint64_t f = 0;
    for (int64_t i = 0; i <= M; ++i) f += spx_fp_term(static_cast<uint64_t>(i), rp[i]);
    return f;
}

spx_status spx_plan_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, spx_loc where,
                        const spx_plan_opts_t* opts, spx_plan** plan_out) {
    if (!plan_out) return SPX_ERR_ARG;
    *plan_out = nullptr;
    if (M < 0 || K < 0 || nnz < 0 || !row_ptr) return SPX_ERR_ARG;
    if (nnz > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (where != SPX_HOST && where != SPX_DEVICE) return SPX_ERR_ARG;
    const int32_t* rp = row_ptr;
    const bool dev = where == SPX_DEVICE;  // device row_ptr: validation, statistics and plan on the GPU
    {
        spx_status s = dev ? spx_dev_check_rp(M, nnz, rp, nullptr) : check_rp(M, nnz, rp);
        if (s != SPX_OK) return s;
    }
    spx_row_stats_t stats;
    try {
        if (dev) {
            spx_status s = spx_dev_row_stats(M, rp, &stats, nullptr);
            if (s != SPX_OK) return s;
        } else {
            row_stats_host(M, rp, &stats);
        }
    } catch (const std::bad_alloc&) {
        return SPX_ERR_NOMEM;
    }
    spx_plan_opts_t o;
    if (opts) o = *opts; else spx_plan_opts_auto(&stats, &o);
    if (o.block_nnz < 1 || o.block_rows < 1 || o.pack_max < 0 || o.pack_max > o.block_nnz || o.cta_max < o.pack_max ||
        o.seg_nnz < 1 || o.lanes_div < 0 || o.block_nnz > 8192 || o.block_rows > 1024)
        return SPX_ERR_ARG;
    spx_status s = SPX_OK;
    spx_plan* P = new (std::nothrow) spx_plan();
    if (!P) return SPX_ERR_NOMEM;
    P->M = M;
    P->K = K;
    P->nnz = nnz;
    P->opts = o;
    P->stats = stats;
    try {
        s = dev ? spx_dev_make_plan(P, rp, nullptr) : make_plan(P, rp);
    } catch (const std::bad_alloc&) {
        s = SPX_ERR_NOMEM;
    }
    if (s == SPX_OK) {
        if (dev) s = spx_dev_rp_fingerprint(M, rp, &P->fingerprint, nullptr);
        else P->fingerprint = rp_fingerprint_host(M, rp);
    }
    if (s != SPX_OK) {
        delete P;
        return s;
    }
    P->magic = kPlanMagic;
    *plan_out = P;
    return SPX_OK;
}

spx_status spx_plan_fingerprint(const spx_plan* P, uint64_t* out) {
    if (!spx_plan_ok(P) || !out) return SPX_ERR_ARG;
    *out = P->fingerprint;
    return SPX_OK;
}

spx_status spx_plan_validate(const spx_plan* P, int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr,
                             spx_loc where, spx_stream_t stream) {
    if (!spx_plan_ok(P) || !row_ptr || (where != SPX_HOST && where != SPX_DEVICE)) return SPX_ERR_ARG;
    if (P->M != M || P->K != K || P->nnz != nnz) return SPX_ERR_ARG;
    uint64_t f = 0;
    if (where == SPX_DEVICE) {
        spx_status s = spx_dev_rp_fingerprint(M, row_ptr, &f, reinterpret_cast<cudaStream_t>(stream));
        if (s != SPX_OK) return s;
    } else {
        f = rp_fingerprint_host(M, row_ptr);
    }
    return f == P->fingerprint ? SPX_OK : SPX_ERR_ARG;
}

spx_status spx_plan_get_info(const spx_plan* P, spx_plan_info_t* out) {
    if (!spx_plan_ok(P) || !out) return SPX_ERR_ARG;
    out->M = P->M;
    out->K = P->K;
    out->nnz = P->nnz;
    out->tasks = P->counts[0];
    out->long_rows = P->counts[1];
    out->slots = P->counts[2];
    out->packed_rows = P->counts[3];
    out->cta_rows = P->counts[4];
    out->split_rows = P->counts[5];
    out->thread_groups = P->counts[6];
    out->lane_groups = P->counts[7];
    out->segmented_groups = P->counts[8];
    out->table_bytes = P->table_bytes;
    out->scratch_bytes = P->scratch_bytes;
    out->stats = P->stats;
    out->opts = P->opts;
    return SPX_OK;
}

spx_status spx_plan_get_tasks(const spx_plan* P, int32_t* tasks, int32_t* long_rows) {
    if (!spx_plan_ok(P)) return SPX_ERR_ARG;
    if (tasks) std::memcpy(tasks, P->tasks.data(), P->tasks.size() * sizeof(int32_t));
    if (long_rows) std::memcpy(long_rows, P->longrows.data(), P->longrows.size() * sizeof(int32_t));
    return SPX_OK;
}

spx_status spx_plan_get_table(const spx_plan* P, void* table) {
    if (!spx_plan_ok(P)) return SPX_ERR_ARG;
    if (P->table_bytes == 0) return SPX_OK;
    if (!table) return SPX_ERR_ARG;
    char* dst = static_cast<char*>(table);
    const size_t tb = P->dtasks.size() * sizeof(int32_t), lb = P->longrows.size() * sizeof(int32_t);
    if (tb) std::memcpy(dst, P->dtasks.data(), tb);
    if (lb) std::memcpy(dst + tb, P->longrows.data(), lb);
    if (!P->first.empty()) std::memcpy(dst + tb + lb, P->first.data(), P->first.size() * sizeof(uint16_t));
    return SPX_OK;
}

spx_status spx_plan_upload(spx_plan* P, void* table, size_t table_bytes, spx_stream_t stream) {
    if (!spx_plan_ok(P)) return SPX_ERR_ARG;
    if (P->table_bytes == 0) {
        P->d_table = table;
        return SPX_OK;
    }
    if (!table || table_bytes < P->table_bytes) return SPX_ERR_ARG;
    if (!spx_aligned(table, 16)) return SPX_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* dst = static_cast<char*>(table);
    const size_t tb = P->dtasks.size() * sizeof(int32_t), lb = P->longrows.size() * sizeof(int32_t);
    cudaError_t e = cudaSuccess;
    if (tb) e = cudaMemcpyAsync(dst, P->dtasks.data(), tb, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && lb) e = cudaMemcpyAsync(dst + tb, P->longrows.data(), lb, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && !P->first.empty())
        e = cudaMemcpyAsync(dst + tb + lb, P->first.data(), P->first.size() * sizeof(uint16_t), cudaMemcpyHostToDevice,
                            st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    P->d_table = table;
    return SPX_OK;
}

spx_status spx_plan_destroy(spx_plan* P) {
    if (!P) return SPX_OK;
    if (!spx_plan_ok(P)) return SPX_ERR_ARG;
    P->magic = 0;
    delete P;
    return SPX_OK;
}

}  // extern "C"

void spx_note_launches(uint64_t n) { g_launches.fetch_add(n); }

spx_status spx_cuda_status(int cuda_error) { return cuda_error == 0 ? SPX_OK : SPX_ERR_CUDA; }
