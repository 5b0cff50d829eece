// spx_sell.cu -- SELL-C-sigma format (host builder) and its SpMV (sm_103a).
//
// [SpMM-ops] §1.4 and [Formats] §6: sliced ELLPACK -- rows are sorted by
// length inside windows of sigma rows, cut into slices of C rows, and each
// slice is padded to its longest row and stored column-major, so that the C
// threads of a slice read their j-th entries from C consecutive words.  Here
// C = 32 (one warp per slice, one thread per row).
//
// Rows longer than T are cut into pieces of T entries ("pseudo-rows") before
// the sort; a piece writes its sum to a partial slot and a second launch adds
// the pieces of each long row in piece order (the segment-plus-fix-up scheme of
// [SpMM-ops] §2.4).  Without the cut, one thread would walk a row of 10^5
// entries alone.  Rows of length 0 are pseudo-rows too (their output is
// beta * y).
//
// Device image (one caller-owned buffer, sections 16-byte aligned):
//   slice_ptr int32[S+1]   first padded entry of each slice (entries, not bytes)
//   prow      int32[32 S]  row of each pseudo-row; -1-slot for a piece of a
//                          long row; INT32_MIN for the unused tail of the last slice
//   longrows  int4[nlong]  {row, first slot, #pieces, 0}
//   scol      int32[padded] column of each padded entry, -1 for padding
//   sval      fp32[padded]  value, 0 for padding
// The kernel reads col/val with coalesced loads and needs no shared memory:
// the layout already gives each thread its own row.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <new>
#include <numeric>
#include <vector>

#include "spx_carveout.cuh"
#include "spx_gather.cuh"
#include "spx_check.cuh"
#include "spx_internal.h"

struct spx_sell {
    int32_t M = 0, K = 0;
    int64_t nnz = 0;
    spx_sell_opts_t opts{};
    std::vector<int32_t> slice_ptr, prow, longrows, scol;  // host-built image (empty when built on the GPU)
    std::vector<float> sval;
    int64_t nslices = 0, padded = 0, nlong = 0, pseudo_rows = 0, slots = 0;
    size_t off_prow = 0, off_long = 0, off_col = 0, off_val = 0, bytes = 0;
    bool gpu_built = false;         // built on the GPU: the host vectors stay empty
    void* d_own = nullptr;          // GPU-built image held by the library until the first upload
    const void* d_image = nullptr;  // the caller's uploaded copy
    uint64_t magic = 0;
};

namespace {

constexpr uint64_t kSellMagic = 0x5350585f53454c4cull;  // "SPX_SELL"
constexpr int kC = 32;
constexpr int kWarpsPerCta = 8;
constexpr int kU = 8;          // entries in flight per thread
constexpr int kMinBlocks = 6;  // register budget: 42 per thread (measured best of 4, 6, 8)

inline size_t align16(size_t n) { return (n + 15) & ~size_t(15); }

SPX_CHECK_WORD(g_sell_check)

// The checked build's tests of the uploaded image (caller memory): a column in
// [-1, K) (-1 is padding), a slice inside the padded entries, a row in [0, M),
// a piece slot in [0, slots).  A failed test skips the access.
struct SellBounds {
    int M, K;
    long long padded, slots;
};
__device__ __forceinline__ bool sell_fail() {
    check_fail();
    return false;
}

struct Pseudo {
    int32_t len, row, start, slot;
};

spx_status build(spx_sell* S, const int32_t* rp, const int32_t* col, const float* val) {
    const spx_sell_opts_t& o = S->opts;
    const int32_t M = S->M;
    std::vector<Pseudo> ps;
    ps.reserve(static_cast<size_t>(M));
    int64_t slots = 0;
    for (int32_t i = 0; i < M; ++i) {
        const int32_t l = rp[i + 1] - rp[i];
        if (l <= o.piece) {
            ps.push_back({l, i, rp[i], -1});
            continue;
        }
        const int32_t n = (l + o.piece - 1) / o.piece;
        if (slots + n > kI32Max) return SPX_ERR_INDEX_RANGE;
        S->longrows.insert(S->longrows.end(), {i, static_cast<int32_t>(slots), n, 0});
        for (int32_t k = 0; k < n; ++k)
            ps.push_back({std::min(o.piece, l - k * o.piece), i, rp[i] + k * o.piece, static_cast<int32_t>(slots + k)});
        slots += n;
    }
    const int64_t np = static_cast<int64_t>(ps.size());
    if (np > kI32Max - kC) return SPX_ERR_INDEX_RANGE;
    // sort inside each window of sigma pseudo-rows, longest first; stable, so equal lengths keep row order
    for (int64_t w0 = 0; w0 < np; w0 += o.sigma) {
        auto b = ps.begin() + w0, e = ps.begin() + std::min<int64_t>(w0 + o.sigma, np);
        std::stable_sort(b, e, [](const Pseudo& a, const Pseudo& c) { return a.len > c.len; });
    }
    const int64_t ns = (np + kC - 1) / kC;
    S->slice_ptr.assign(static_cast<size_t>(ns) + 1, 0);
    int64_t padded = 0;
    for (int64_t s = 0; s < ns; ++s) {
        int32_t L = 0;
        for (int64_t p = s * kC; p < std::min<int64_t>((s + 1) * kC, np); ++p) L = std::max(L, ps[p].len);
        padded += static_cast<int64_t>(L) * kC;
        if (padded > kI32Max) return SPX_ERR_INDEX_RANGE;
        S->slice_ptr[static_cast<size_t>(s) + 1] = static_cast<int32_t>(padded);
    }
    S->prow.assign(static_cast<size_t>(ns * kC), INT32_MIN);
    S->scol.assign(static_cast<size_t>(padded), -1);
    S->sval.assign(static_cast<size_t>(padded), 0.f);
    for (int64_t p = 0; p < np; ++p) {
        const Pseudo& q = ps[p];
        S->prow[p] = q.slot < 0 ? q.row : -1 - q.slot;
        const int64_t s = p / kC, r = p % kC, base = S->slice_ptr[s];
        for (int32_t j = 0; j < q.len; ++j) {
            S->scol[base + static_cast<int64_t>(j) * kC + r] = col[q.start + j];
            S->sval[base + static_cast<int64_t>(j) * kC + r] = val[q.start + j];
        }
    }
    S->pseudo_rows = np;
    S->slots = slots;
    S->nslices = ns;
    S->padded = padded;
    S->nlong = static_cast<int64_t>(S->longrows.size() / 4);
    S->off_prow = align16(sizeof(int32_t) * S->slice_ptr.size());
    S->off_long = S->off_prow + align16(sizeof(int32_t) * S->prow.size());
    S->off_col = S->off_long + align16(sizeof(int32_t) * S->longrows.size());
    S->off_val = S->off_col + align16(sizeof(int32_t) * S->scol.size());
    S->bytes = S->off_val + align16(sizeof(float) * S->sval.size());
    return SPX_OK;
}

// ---------------------------------------------------------------- kernels

__global__ void __launch_bounds__(kC * kWarpsPerCta, kMinBlocks) sell_kernel(int nslices, const int* __restrict__ slice_ptr,
                                                                 const int* __restrict__ prow,
                                                                 const int* __restrict__ scol,
                                                                 const float* __restrict__ sval,
                                                                 const float* __restrict__ x, float alpha, float beta,
                                                                 float* y, float* __restrict__ partials,
                                                                 SellBounds bd) {
    const int s = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= nslices) return;
    const int p0 = __ldg(slice_ptr + s);
    const int L = (__ldg(slice_ptr + s + 1) - p0) / kC;
    const int pr = __ldg(prow + s * kC + lane);
    if (SPX_CHECKED) {
        const long long p1 = p0 + static_cast<long long>(L) * kC;
        const bool slice_ok = p0 >= 0 && L >= 0 && p1 <= bd.padded;
        const bool row_ok = (pr >= 0 && pr < bd.M) || pr == INT_MIN || (pr < 0 && -1LL - pr < bd.slots);
        if (!slice_ok || !row_ok) {
            sell_fail();
            return;
        }
    }
    const float y_old = pr >= 0 && beta != 0.f ? y[pr] : 0.f;  // read up front, off the epilogue's path
    const int* cp = scol + p0 + lane;
    const float* vp = sval + p0 + lane;
    float acc = 0.f;
    int j = 0;
    for (; j + kU <= L; j += kU) {
        int c[kU];
        float v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            c[u] = spx_gather::ld_once(cp + (j + u) * kC);
            v[u] = spx_gather::ld_once(vp + (j + u) * kC);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (SPX_CHECKED && (c[u] < -1 || c[u] >= bd.K)) {
                sell_fail();
                c[u] = -1;
            }
            acc += v[u] * (c[u] >= 0 ? spx_gather::ld_x(x + c[u]) : 0.f);
        }
    }
    for (; j < L; ++j) {
        int c0 = spx_gather::ld_once(cp + j * kC);
        const float v0 = spx_gather::ld_once(vp + j * kC);
        if (SPX_CHECKED && (c0 < -1 || c0 >= bd.K)) {
            sell_fail();
            c0 = -1;
        }
        acc += v0 * (c0 >= 0 ? spx_gather::ld_x(x + c0) : 0.f);
    }
    if (pr >= 0) y[pr] = beta != 0.f ? alpha * acc + beta * y_old : alpha * acc;
    else if (pr != INT_MIN) partials[-1 - pr] = acc;
}

// One warp per long row: its pieces' sums in piece order (lane-strided, then a fixed tree).
__global__ void __launch_bounds__(256) sell_fixup_kernel(const int4* __restrict__ longrows, int nlong,
                                                         const float* __restrict__ partials, float alpha, float beta,
                                                         float* y, SellBounds bd) {
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= nlong) return;
    const int4 lr = longrows[w];
    if (SPX_CHECKED && !(lr.x >= 0 && lr.x < bd.M && lr.y >= 0 && lr.z >= 0 && lr.y + static_cast<long long>(lr.z) <= bd.slots)) {
        if (lane == 0) sell_fail();
        return;
    }
    float s = 0.f;
    for (int k = lane; k < lr.z; k += 32) s += partials[lr.y + k];
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) s += __shfl_down_sync(0xffffffffu, s, d);
    if (lane == 0) y[lr.x] = beta != 0.f ? alpha * s + beta * y[lr.x] : alpha * s;
}

inline bool sell_ok(const spx_sell* S) { return S && S->magic == kSellMagic; }

}  // namespace

int spx_sell_check_take() { return spx_check_take(g_sell_check); }

extern "C" {

spx_status spx_sell_opts_default(spx_sell_opts_t* o) {
    if (!o) return SPX_ERR_ARG;
    o->sigma = 1024;
    o->piece = 64;
    return SPX_OK;
}

spx_status spx_sell_build(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                          const float* val, spx_loc where, const spx_sell_opts_t* opts, spx_sell** out) {
    if (!out) return SPX_ERR_ARG;
    *out = nullptr;
    if (M < 0 || K < 0 || nnz < 0 || !row_ptr || (nnz > 0 && (!col || !val))) return SPX_ERR_ARG;
    if (nnz > kI32Max) return SPX_ERR_INDEX_RANGE;
    spx_sell_opts_t o;
    if (opts) o = *opts; else spx_sell_opts_default(&o);
    if (o.sigma < kC || o.sigma % kC || o.sigma > (1 << 20) || o.piece < 1 || o.piece > (1 << 24)) return SPX_ERR_ARG;
    if (where == SPX_DEVICE) {  // built on the GPU (spx_build.cu); the image stays in device memory
        spx_sell_dev_image img;
        spx_status s = spx_dev_build_sell(M, K, nnz, row_ptr, col, val, o.sigma, o.piece, &img, nullptr);
        if (s != SPX_OK) return s;
        spx_sell* S = new (std::nothrow) spx_sell();
        if (!S) {
            cudaFree(img.image);
            return SPX_ERR_NOMEM;
        }
        S->M = M;
        S->K = K;
        S->nnz = nnz;
        S->opts = o;
        S->gpu_built = true;
        S->d_own = img.image;
        S->bytes = img.bytes;
        S->off_prow = img.off_prow;
        S->off_long = img.off_long;
        S->off_col = img.off_col;
        S->off_val = img.off_val;
        S->nslices = img.nslices;
        S->padded = img.padded;
        S->nlong = img.nlong;
        S->pseudo_rows = img.pseudo_rows;
        S->slots = img.slots;
        S->magic = kSellMagic;
        *out = S;
        return SPX_OK;
    }
    if (where != SPX_HOST) return SPX_ERR_ARG;
    const int32_t* rp = row_ptr;
    const int32_t* cl = col;
    const float* vl = val;
    if (rp[0] != 0 || rp[M] != nnz) return SPX_ERR_ARG;
    for (int32_t i = 0; i < M; ++i)
        if (rp[i + 1] < rp[i]) return SPX_ERR_NOT_SORTED;
    for (int64_t p = 0; p < nnz; ++p)
        if (cl[p] < 0 || cl[p] >= K) return SPX_ERR_INDEX_RANGE;
    spx_sell* S = new (std::nothrow) spx_sell();
    if (!S) return SPX_ERR_NOMEM;
    S->M = M;
    S->K = K;
    S->nnz = nnz;
    S->opts = o;
    spx_status s;
    try {
        s = build(S, rp, cl, vl);
    } catch (const std::bad_alloc&) {
        s = SPX_ERR_NOMEM;
    }
    if (s != SPX_OK) {
        delete S;
        return s;
    }
    S->magic = kSellMagic;
    *out = S;
    return SPX_OK;
}

spx_status spx_sell_get_info(const spx_sell* S, spx_sell_info_t* out) {
    if (!sell_ok(S) || !out) return SPX_ERR_ARG;
    std::memset(out, 0, sizeof(*out));
    out->M = S->M;
    out->K = S->K;
    out->nnz = S->nnz;
    out->slices = S->nslices;
    out->pseudo_rows = S->pseudo_rows;
    out->padded = S->padded;
    out->long_rows = S->nlong;
    out->slots = S->slots;
    out->image_bytes = S->bytes;
    out->scratch_bytes = sizeof(float) * static_cast<size_t>(S->slots);
    out->opts = S->opts;
    return SPX_OK;
}

spx_status spx_sell_get_arrays(const spx_sell* S, int32_t* slice_ptr, int32_t* prow, int32_t* longrows, int32_t* scol,
                               float* sval) {
    if (!sell_ok(S)) return SPX_ERR_ARG;
    const char* dimg = static_cast<const char*>(S->d_own ? S->d_own : S->d_image);
    if (S->gpu_built) {  // copy the sections down
        if (!dimg) return SPX_ERR_NOT_READY;
        const size_t n[5] = {sizeof(int32_t) * static_cast<size_t>(S->nslices + 1),
                             sizeof(int32_t) * static_cast<size_t>(S->nslices * kC),
                             sizeof(int32_t) * static_cast<size_t>(4 * S->nlong),
                             sizeof(int32_t) * static_cast<size_t>(S->padded), sizeof(float) * static_cast<size_t>(S->padded)};
        const size_t off[5] = {0, S->off_prow, S->off_long, S->off_col, S->off_val};
        void* dst[5] = {slice_ptr, prow, longrows, scol, sval};
        for (int i = 0; i < 5; ++i)
            if (dst[i] && n[i] && cudaMemcpy(dst[i], dimg + off[i], n[i], cudaMemcpyDeviceToHost) != cudaSuccess)
                return SPX_ERR_CUDA;
        return SPX_OK;
    }
    auto cp = [](void* dst, const void* src, size_t n) {
        if (dst && n) std::memcpy(dst, src, n);
    };
    cp(slice_ptr, S->slice_ptr.data(), sizeof(int32_t) * S->slice_ptr.size());
    cp(prow, S->prow.data(), sizeof(int32_t) * S->prow.size());
    cp(longrows, S->longrows.data(), sizeof(int32_t) * S->longrows.size());
    cp(scol, S->scol.data(), sizeof(int32_t) * S->scol.size());
    cp(sval, S->sval.data(), sizeof(float) * S->sval.size());
    return SPX_OK;
}

spx_status spx_sell_upload(spx_sell* S, void* image, size_t image_bytes, spx_stream_t stream) {
    if (!sell_ok(S)) return SPX_ERR_ARG;
    if (!image || image_bytes < S->bytes) return SPX_ERR_ARG;
    if (!spx_aligned(image, 16)) return SPX_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* d = static_cast<char*>(image);
    if (S->gpu_built) {  // one device-to-device copy, then the library's copy is freed
        const void* src = S->d_own ? S->d_own : S->d_image;
        if (!src) return SPX_ERR_NOT_READY;
        cudaError_t e = src == image ? cudaSuccess : cudaMemcpyAsync(d, src, S->bytes, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return SPX_ERR_CUDA;
        if (S->d_own) cudaFree(S->d_own);
        S->d_own = nullptr;
        S->d_image = image;
        return SPX_OK;
    }
    struct Part {
        size_t off;
        const void* src;
        size_t n;
    } parts[] = {{0, S->slice_ptr.data(), sizeof(int32_t) * S->slice_ptr.size()},
                 {S->off_prow, S->prow.data(), sizeof(int32_t) * S->prow.size()},
                 {S->off_long, S->longrows.data(), sizeof(int32_t) * S->longrows.size()},
                 {S->off_col, S->scol.data(), sizeof(int32_t) * S->scol.size()},
                 {S->off_val, S->sval.data(), sizeof(float) * S->sval.size()}};
    cudaError_t e = cudaSuccess;
    for (const Part& p : parts)
        if (e == cudaSuccess && p.n) e = cudaMemcpyAsync(d + p.off, p.src, p.n, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPX_ERR_CUDA;
    S->d_image = image;
    return SPX_OK;
}

spx_status spx_sell_destroy(spx_sell* S) {
    if (!S) return SPX_OK;
    if (!sell_ok(S)) return SPX_ERR_ARG;
    S->magic = 0;
    if (S->d_own) cudaFree(S->d_own);
    delete S;
    return SPX_OK;
}

spx_status spx_spmv_sell(const spx_sell* S, int32_t M, int32_t K, float alpha, const float* x, float beta, float* y,
                         void* scratch, size_t scratch_bytes, spx_stream_t stream) {
    if (!sell_ok(S)) return SPX_ERR_ARG;
    if (M != S->M || K != S->K) return SPX_ERR_ARG;
    if (!S->d_image) return SPX_ERR_NOT_READY;
    if (M == 0) return SPX_OK;
    if (!y || (S->nnz > 0 && !x)) return SPX_ERR_ARG;
    if (!spx_aligned(y, 4) || (x && !spx_aligned(x, 4))) return SPX_ERR_ALIGN;
    const size_t need = sizeof(float) * static_cast<size_t>(S->slots);
    if (need && (!scratch || scratch_bytes < need)) return SPX_ERR_ARG;
    if (x) {
        const char* xb = reinterpret_cast<const char*>(x);
        const char* yb = reinterpret_cast<const char*>(y);
        if (xb < yb + 4 * static_cast<size_t>(M) && yb < xb + 4 * static_cast<size_t>(K)) return SPX_ERR_ARG;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const char* img = static_cast<const char*>(S->d_image);
    const int nslices = static_cast<int>(S->nslices);
    const int nlong = static_cast<int>(S->nlong);
    uint64_t launches = 0;
    if (nslices > 0) {
        spx_carve::fit(sell_kernel, kC * kWarpsPerCta, 0);
        sell_kernel<<<(nslices + kWarpsPerCta - 1) / kWarpsPerCta, kC * kWarpsPerCta, 0, st>>>(
            nslices, reinterpret_cast<const int*>(img), reinterpret_cast<const int*>(img + S->off_prow),
            reinterpret_cast<const int*>(img + S->off_col), reinterpret_cast<const float*>(img + S->off_val), x, alpha,
            beta, y, static_cast<float*>(scratch), SellBounds{M, K, S->padded, S->slots});
        ++launches;
    }
    if (nlong > 0) {
        sell_fixup_kernel<<<(nlong + 7) / 8, 256, 0, st>>>(reinterpret_cast<const int4*>(img + S->off_long), nlong,
                                                           static_cast<const float*>(scratch), alpha, beta, y,
                                                           SellBounds{M, K, S->padded, S->slots});
        ++launches;
    }
    spx_note_launches(launches);
    return spx_cuda_status(cudaGetLastError());
}

}  // extern "C"
