// spx_tune.cpp -- measured choice of the SpMV plan options, cached per matrix profile.
//
// [SpMM-ops] §4: profile the matrix once (row-length statistics as the
// dispatch key), choose the kernel mapping, and keep the choice with the
// matrix so later calls reuse it.  The row-statistics rule of
// spx_plan_opts_auto is a guess from the key alone; this routine times a
// handful of candidate option sets on the device with the caller's own
// matrix and vector and keeps the fastest, under a key made of the matrix's
// sizes and row-length profile.
#include <cuda_runtime.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "spx_internal.h"

namespace {

using Key = std::tuple<int, int32_t, int32_t, int64_t, int64_t, int32_t, int32_t, int32_t>;

std::mutex g_mu;
std::map<Key, spx_plan_opts_t> g_cache;

// The built-in candidates: the default lanes rule at two divisors and the
// segmented reduction at two group sizes.
constexpr int kBuiltin = 4;
void builtin_candidates(spx_plan_opts_t* c) {
    for (int i = 0; i < kBuiltin; ++i) spx_plan_opts_default(&c[i]);
    c[1].lanes_div = 4;
    c[2].block_nnz = 1024;
    c[2].lanes_div = 0;
    c[3].lanes_div = 0;
}

struct DevBuf {
    void* p = nullptr;
    ~DevBuf() {
        if (p) cudaFree(p);
    }
    cudaError_t alloc(size_t n) { return n ? cudaMalloc(&p, n) : cudaSuccess; }
};

struct PlanHolder {
    spx_plan* p = nullptr;
    ~PlanHolder() { spx_plan_destroy(p); }
};

}  // namespace

extern "C" {

spx_status spx_plan_autotune(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr_host, const int32_t* row_ptr,
                             const int32_t* col, const float* val, const float* x, float* y_scratch,
                             const spx_plan_opts_t* candidates, int32_t ncand, int32_t reps, spx_stream_t stream,
                             spx_plan_opts_t* best, float* times_ms, int32_t* cached) {
    if (M < 0 || K < 0 || nnz < 0 || !row_ptr_host || !best) return SPX_ERR_ARG;
    if (nnz > kI32Max) return SPX_ERR_INDEX_RANGE;
    if (reps < 1 || reps > 1000) return SPX_ERR_ARG;
    if (candidates && (ncand < 1 || ncand > 16)) return SPX_ERR_ARG;
    if (M > 0 && (!row_ptr || !y_scratch)) return SPX_ERR_ARG;
    if (nnz > 0 && (!col || !val || !x)) return SPX_ERR_ARG;
    spx_row_stats_t st;
    spx_status s = spx_row_stats(M, row_ptr_host, SPX_HOST, &st);
    if (s != SPX_OK) return s;
    if (st.nnz != nnz) return SPX_ERR_ARG;

    spx_plan_opts_t builtin[kBuiltin];
    builtin_candidates(builtin);
    const spx_plan_opts_t* cand = candidates ? candidates : builtin;
    const int n = candidates ? ncand : kBuiltin;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPX_ERR_CUDA;
    // Explicit candidates are part of the key: a different candidate list is a different question.
    int32_t cand_tag = 0;
    if (candidates) {
        uint32_t h = 2166136261u;
        const unsigned char* b = reinterpret_cast<const unsigned char*>(candidates);
        for (size_t i = 0; i < sizeof(spx_plan_opts_t) * static_cast<size_t>(n); ++i) h = (h ^ b[i]) * 16777619u;
        cand_tag = static_cast<int32_t>(h | 1u);
    }
    const Key key{dev, M, K, nnz, st.sumsq, st.max, st.p99, cand_tag};
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_cache.find(key);
        if (it != g_cache.end()) {
            *best = it->second;
            if (cached) *cached = 1;
            if (times_ms)
                for (int i = 0; i < n; ++i) times_ms[i] = -1.f;
            return SPX_OK;
        }
    }

    cudaStream_t stm = reinterpret_cast<cudaStream_t>(stream);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        return SPX_ERR_CUDA;
    }
    int pick = -1;
    float pick_ms = 0.f;
    for (int i = 0; i < n && s == SPX_OK; ++i) {
        PlanHolder P;
        s = spx_plan_csr(M, K, nnz, row_ptr_host, SPX_HOST, &cand[i], &P.p);
        if (s != SPX_OK) break;
        spx_plan_info_t info;
        spx_plan_get_info(P.p, &info);
        DevBuf table, scratch;
        if (table.alloc(info.table_bytes) != cudaSuccess || scratch.alloc(info.scratch_bytes) != cudaSuccess) {
            s = SPX_ERR_NOMEM;
            break;
        }
        s = spx_plan_upload(P.p, table.p, info.table_bytes, stream);
        auto call = [&] {
            return spx_spmv_csr(P.p, M, K, nnz, row_ptr, col, val, 1.f, x, 0.f, y_scratch, scratch.p,
                                info.scratch_bytes, stream);
        };
        if (s == SPX_OK) s = call();  // warm-up
        if (s != SPX_OK) break;
        if (cudaEventRecord(e0, stm) != cudaSuccess) {
            s = SPX_ERR_CUDA;
            break;
        }
        for (int r = 0; r < reps && s == SPX_OK; ++r) s = call();
        if (s != SPX_OK) break;
        float ms = 0.f;
        if (cudaEventRecord(e1, stm) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
            cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
            s = SPX_ERR_CUDA;
            break;
        }
        ms /= static_cast<float>(reps);
        if (times_ms) times_ms[i] = ms;
        if (pick < 0 || ms < pick_ms) {
            pick = i;
            pick_ms = ms;
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (s != SPX_OK) return s;
    *best = cand[pick];
    if (cached) *cached = 0;
    std::lock_guard<std::mutex> lock(g_mu);
    g_cache[key] = cand[pick];
    return SPX_OK;
}

spx_status spx_plan_autotune_forget(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    g_cache.clear();
    return SPX_OK;
}

}  // extern "C"
