// spx_build.cu -- format builders on the GPU: COO -> CSR and CSR -> CSR(A^T).
//
// [Formats] §3 (COO -> CSR: histogram of the row indices, prefix sum, stable
// scatter, entries of a row in column order) and [LSMR-dual] §2, §4 (CSR(A^T)
// = CSC(A): a counting sort by column that keeps rows ascending inside each
// output row).  Both are stable sorts of the entries by an integer key, done
// here as an LSD radix sort with 8-bit digits:
//   per tile of 2048 keys, a 256-bin histogram (shared-memory integer
//   atomics -- exact counts); an exclusive scan over (digit, tile); a scatter
//   that ranks each key among equal digits in input order (warp match + per-
//   warp counts), so every pass is stable and the result is the unique
//   stable order.
// COO -> CSR sorts by column, then by row (LSD over the pair); CSR -> CSR(A^T)
// sorts by column only (the entries already come in row order).  The sort
// carries each entry's source index; columns and values (1, 2, 4 or 8 bytes)
// are gathered through it at the end.  Row offsets come from exact per-row
// counts and a scan.  Indices are validated first (SPX_ERR_INDEX_RANGE, like
// the host builders).  Temporary device memory is taken from the stream-
// ordered allocator and returned before the call ends.
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "spx_internal.h"

namespace {

constexpr int kT = 256;              // threads per CTA
constexpr int kPer = 8;              // keys per thread per tile
constexpr int kTile = kT * kPer;     // 2048 keys per tile
constexpr int kScanBlock = 2048;     // elements per scan block (256 threads x 8)

// ---------------------------------------------------------------- validation
__global__ void check_indices(const int* __restrict__ a, long long n, int lim, int* __restrict__ bad) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        const int v = a[i];
        if (v < 0 || v >= lim) atomicOr(bad, 1);
    }
}

// row_ptr must start at 0, end at nnz and never decrease.
__global__ void check_row_ptr(const int* __restrict__ rp, int M, long long nnz, int* __restrict__ bad) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < M;
         i += static_cast<long long>(gridDim.x) * kT)
        if (rp[i + 1] < rp[i]) atomicOr(bad, 2);
    if (blockIdx.x == 0 && threadIdx.x == 0 && (rp[0] != 0 || static_cast<long long>(rp[M]) != nnz)) atomicOr(bad, 4);
}

// ---------------------------------------------------------------- scan (exclusive, uint32)
// Block b scans in[b*2048 .. +2048) into out and writes its total to sums[b].
__global__ void __launch_bounds__(kT) scan_blocks(const uint32_t* __restrict__ in, uint32_t* __restrict__ out,
                                                  long long n, uint32_t* __restrict__ sums) {
    __shared__ uint32_t s_w[kT / 32];
    const long long base = blockIdx.x * static_cast<long long>(kScanBlock) + threadIdx.x * kPer;
    uint32_t v[kPer], t = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        v[j] = base + j < n ? in[base + j] : 0u;
        t += v[j];
    }
    // exclusive scan of the per-thread totals across the block
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = t;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    uint32_t wp = 0;
    for (int w = 0; w < warp; ++w) wp += s_w[w];
    uint32_t run = wp + x - t;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (base + j < n) out[base + j] = run;
        run += v[j];
    }
    if (threadIdx.x == kT - 1) sums[blockIdx.x] = wp + x;
}

__global__ void __launch_bounds__(kT) scan_add(uint32_t* __restrict__ out, long long n,
                                               const uint32_t* __restrict__ offs) {
    const long long base = blockIdx.x * static_cast<long long>(kScanBlock) + threadIdx.x * kPer;
    const uint32_t o = offs[blockIdx.x];
#pragma unroll
    for (int j = 0; j < kPer; ++j)
        if (base + j < n) out[base + j] += o;
}

// ---------------------------------------------------------------- radix sort
// hist[d * ntiles + tile] = number of keys of this tile whose digit is d.
__global__ void __launch_bounds__(kT) radix_hist(const uint32_t* __restrict__ keys, long long n, int shift,
                                                 uint32_t* __restrict__ hist, int ntiles) {
    __shared__ uint32_t h[256];
    h[threadIdx.x] = 0;
    __syncthreads();
    const long long base = blockIdx.x * static_cast<long long>(kTile);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const long long i = base + j * kT + threadIdx.x;
        if (i < n) atomicAdd(&h[(keys[i] >> shift) & 255u], 1u);
    }
    __syncthreads();
    hist[static_cast<long long>(threadIdx.x) * ntiles + blockIdx.x] = h[threadIdx.x];
}

// Stable scatter of one tile: keys are taken in input order, 256 per round;
// a key's place = the tile's offset for its digit + keys of that digit in
// earlier rounds + in earlier warps of this round + in lower lanes of its warp.
__global__ void __launch_bounds__(kT) radix_scatter(const uint32_t* __restrict__ kin, const int* __restrict__ iin,
                                                    uint32_t* __restrict__ kout, int* __restrict__ iout, long long n,
                                                    int shift, const uint32_t* __restrict__ offs, int ntiles) {
    __shared__ uint32_t s_base[256];
    __shared__ uint32_t s_cnt[kT / 32][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    s_base[threadIdx.x] = offs[static_cast<long long>(threadIdx.x) * ntiles + blockIdx.x];
    const long long base = blockIdx.x * static_cast<long long>(kTile);
    const unsigned below = (1u << lane) - 1u;
    for (int r = 0; r < kPer; ++r) {
#pragma unroll
        for (int w = 0; w < kT / 32; ++w) s_cnt[w][threadIdx.x] = 0;
        __syncthreads();
        const long long i = base + r * kT + threadIdx.x;
        const bool valid = i < n;
        const uint32_t key = valid ? kin[i] : 0u;
        const int idx = valid ? iin[i] : 0;
        const uint32_t d = valid ? ((key >> shift) & 255u) : 256u;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        const int rank = __popc(peers & below);
        if (valid && rank == 0) s_cnt[warp][d] = __popc(peers);
        __syncthreads();
        if (valid) {
            uint32_t pos = s_base[d] + rank;
            for (int w = 0; w < warp; ++w) pos += s_cnt[w][d];
            kout[pos] = key;
            iout[pos] = idx;
        }
        __syncthreads();
        uint32_t add = 0;
#pragma unroll
        for (int w = 0; w < kT / 32; ++w) add += s_cnt[w][threadIdx.x];
        s_base[threadIdx.x] += add;
        __syncthreads();
    }
}

__global__ void iota_keys(const int* __restrict__ src, uint32_t* __restrict__ keys, int* __restrict__ idx, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT) {
        keys[i] = static_cast<uint32_t>(src[i]);
        idx[i] = static_cast<int>(i);
    }
}

// keys[i] = src[idx[i]] (the next, more significant key in source order of the current permutation)
__global__ void gather_keys(const int* __restrict__ src, const int* __restrict__ idx, uint32_t* __restrict__ keys,
                            long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT)
        keys[i] = static_cast<uint32_t>(src[idx[i]]);
}

template <class T>
__global__ void gather_values(const T* __restrict__ src, const int* __restrict__ idx, T* __restrict__ dst,
                              long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT)
        dst[i] = src[idx[i]];
}

__global__ void count_keys(const int* __restrict__ a, long long n, uint32_t* __restrict__ cnt) {
    for (long long i = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kT)
        atomicAdd(&cnt[a[i]], 1u);
}

// rowid[p] = the row holding entry p: the last i with rp[i] <= p (binary search).
__global__ void expand_rows(const int* __restrict__ rp, int M, long long n, int* __restrict__ rowid) {
    for (long long p = blockIdx.x * static_cast<long long>(kT) + threadIdx.x; p < n;
         p += static_cast<long long>(gridDim.x) * kT) {
        int lo = 0, hi = M;  // rp[lo] <= p < rp[hi]
        while (hi - lo > 1) {
            const int mid = lo + (hi - lo) / 2;
            if (rp[mid] <= p) lo = mid;
            else hi = mid;
        }
        rowid[p] = lo;
    }
}

int grid_for(long long n) {
    long long g = (n + kT - 1) / kT;
    if (g > 152 * 32) g = 152 * 32;
    return static_cast<int>(g < 1 ? 1 : g);
}

// ---------------------------------------------------------------- host helpers
struct Pool {
    cudaStream_t st;
    std::vector<void*> ptrs;
    cudaError_t err = cudaSuccess;
    explicit Pool(cudaStream_t s) : st(s) {}
    template <class T>
    T* get(long long n) {
        void* p = nullptr;
        if (err == cudaSuccess) err = cudaMallocAsync(&p, static_cast<size_t>(n > 0 ? n : 1) * sizeof(T), st);
        if (err == cudaSuccess) ptrs.push_back(p);
        return static_cast<T*>(p);
    }
    ~Pool() {
        for (void* p : ptrs) cudaFreeAsync(p, st);
    }
};

// Exclusive scan of n uint32 (in place allowed: out may equal in).
cudaError_t scan_exclusive(const uint32_t* in, uint32_t* out, long long n, Pool& pool) {
    if (n <= 0) return cudaSuccess;
    const long long nb = (n + kScanBlock - 1) / kScanBlock;
    uint32_t* sums = pool.get<uint32_t>(nb);
    if (pool.err != cudaSuccess) return pool.err;
    scan_blocks<<<static_cast<unsigned>(nb), kT, 0, pool.st>>>(in, out, n, sums);
    if (nb > 1) {
        cudaError_t e = scan_exclusive(sums, sums, nb, pool);
        if (e != cudaSuccess) return e;
        scan_add<<<static_cast<unsigned>(nb), kT, 0, pool.st>>>(out, n, sums);
    }
    return cudaGetLastError();
}

int bits_for(long long lim) {  // bits needed for keys in [0, lim)
    int b = 0;
    while (b < 32 && (1ll << b) < lim) ++b;
    return b;
}

// Stable LSD radix sort of (k, ix) by the low `bits` bits of the keys; the
// result ends in (k, ix) (the second buffers are scratch).
cudaError_t radix_sort(uint32_t*& k, int*& ix, uint32_t*& k2, int*& ix2, long long n, int bits, Pool& pool,
                       uint64_t& launches) {
    if (n <= 1) return cudaSuccess;
    const int ntiles = static_cast<int>((n + kTile - 1) / kTile);
    uint32_t* hist = pool.get<uint32_t>(256ll * ntiles);
    if (pool.err != cudaSuccess) return pool.err;
    for (int shift = 0; shift < bits; shift += 8) {
        radix_hist<<<ntiles, kT, 0, pool.st>>>(k, n, shift, hist, ntiles);
        cudaError_t e = scan_exclusive(hist, hist, 256ll * ntiles, pool);
        if (e != cudaSuccess) return e;
        radix_scatter<<<ntiles, kT, 0, pool.st>>>(k, ix, k2, ix2, n, shift, hist, ntiles);
        launches += 3;
        std::swap(k, k2);
        std::swap(ix, ix2);
    }
    return cudaGetLastError();
}

cudaError_t gather_vals(const void* src, const int* idx, void* dst, long long n, int vb, cudaStream_t st) {
    const int g = grid_for(n);
    switch (vb) {
        case 1: gather_values<uint8_t><<<g, kT, 0, st>>>(static_cast<const uint8_t*>(src), idx, static_cast<uint8_t*>(dst), n); break;
        case 2: gather_values<uint16_t><<<g, kT, 0, st>>>(static_cast<const uint16_t*>(src), idx, static_cast<uint16_t*>(dst), n); break;
        case 4: gather_values<uint32_t><<<g, kT, 0, st>>>(static_cast<const uint32_t*>(src), idx, static_cast<uint32_t*>(dst), n); break;
        default: gather_values<uint64_t><<<g, kT, 0, st>>>(static_cast<const uint64_t*>(src), idx, static_cast<uint64_t*>(dst), n); break;
    }
    return cudaGetLastError();
}

spx_status read_flag(const int* d_bad, cudaStream_t st, int* h) {
    if (cudaMemcpyAsync(h, d_bad, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SPX_ERR_CUDA;
    return SPX_OK;
}

// Row offsets from exact counts: ptr[0..lim] = exclusive scan of count(key == i), ptr[lim] = n.
cudaError_t offsets(const int* keys, long long n, int lim, int32_t* ptr, Pool& pool, uint64_t& launches) {
    uint32_t* cnt = reinterpret_cast<uint32_t*>(ptr);  // counted in place: lim + 1 slots
    cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(uint32_t) * (static_cast<size_t>(lim) + 1), pool.st);
    if (e != cudaSuccess) return e;
    if (n > 0) {
        count_keys<<<grid_for(n), kT, 0, pool.st>>>(keys, n, cnt);
        ++launches;
    }
    e = scan_exclusive(cnt, cnt, static_cast<long long>(lim) + 1, pool);
    ++launches;
    return e;
}

}  // namespace

spx_status spx_dev_build_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* coo_row, const int32_t* coo_col,
                             const void* coo_val, int32_t vb, int32_t* row_ptr, int32_t* col, void* val,
                             cudaStream_t st) {
    Pool pool(st);
    uint64_t launches = 0;
    int* bad = pool.get<int>(1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    if (cudaMemsetAsync(bad, 0, sizeof(int), st) != cudaSuccess) return SPX_ERR_CUDA;
    if (nnz > 0) {
        check_indices<<<grid_for(nnz), kT, 0, st>>>(coo_row, nnz, M, bad);
        check_indices<<<grid_for(nnz), kT, 0, st>>>(coo_col, nnz, K, bad);
        launches += 2;
    }
    int h = 0;
    spx_status s = read_flag(bad, st, &h);
    if (s != SPX_OK) return s;
    if (h) return SPX_ERR_INDEX_RANGE;
    uint32_t *k = pool.get<uint32_t>(nnz), *k2 = pool.get<uint32_t>(nnz);
    int *ix = pool.get<int>(nnz), *ix2 = pool.get<int>(nnz);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    cudaError_t e = cudaSuccess;
    if (nnz > 0) {
        // LSD over (row, col): stable by column first, then stable by row
        iota_keys<<<grid_for(nnz), kT, 0, st>>>(coo_col, k, ix, nnz);
        ++launches;
        e = radix_sort(k, ix, k2, ix2, nnz, bits_for(K), pool, launches);
        if (e == cudaSuccess) {
            gather_keys<<<grid_for(nnz), kT, 0, st>>>(coo_row, ix, k, nnz);
            ++launches;
            e = radix_sort(k, ix, k2, ix2, nnz, bits_for(M), pool, launches);
        }
        if (e == cudaSuccess) {
            gather_values<int32_t><<<grid_for(nnz), kT, 0, st>>>(coo_col, ix, col, nnz);
            e = gather_vals(coo_val, ix, val, nnz, vb, st);
            launches += 2;
        }
    }
    if (e == cudaSuccess) e = offsets(coo_row, nnz, M, row_ptr, pool, launches);
    if (e == cudaSuccess) e = cudaGetLastError();
    spx_note_launches(launches);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    return e == cudaSuccess ? SPX_OK : SPX_ERR_CUDA;
}

spx_status spx_dev_transpose_csr(int32_t M, int32_t K, int64_t nnz, const int32_t* row_ptr, const int32_t* col,
                                 const void* val, int32_t vb, int32_t* t_row_ptr, int32_t* t_col, void* t_val,
                                 cudaStream_t st) {
    Pool pool(st);
    uint64_t launches = 0;
    int* bad = pool.get<int>(1);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    if (cudaMemsetAsync(bad, 0, sizeof(int), st) != cudaSuccess) return SPX_ERR_CUDA;
    check_row_ptr<<<grid_for(M), kT, 0, st>>>(row_ptr, M, nnz, bad);
    ++launches;
    if (nnz > 0) {
        check_indices<<<grid_for(nnz), kT, 0, st>>>(col, nnz, K, bad);
        ++launches;
    }
    int h = 0;
    spx_status s = read_flag(bad, st, &h);
    if (s != SPX_OK) return s;
    if (h & 4) return SPX_ERR_ARG;
    if (h & 2) return SPX_ERR_NOT_SORTED;
    if (h & 1) return SPX_ERR_INDEX_RANGE;
    uint32_t *k = pool.get<uint32_t>(nnz), *k2 = pool.get<uint32_t>(nnz);
    int *ix = pool.get<int>(nnz), *ix2 = pool.get<int>(nnz), *rowid = pool.get<int>(nnz);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    cudaError_t e = cudaSuccess;
    if (nnz > 0) {
        expand_rows<<<grid_for(nnz), kT, 0, st>>>(row_ptr, M, nnz, rowid);
        iota_keys<<<grid_for(nnz), kT, 0, st>>>(col, k, ix, nnz);
        launches += 2;
        // entries come in row order: a stable sort by column keeps rows ascending in each column
        e = radix_sort(k, ix, k2, ix2, nnz, bits_for(K), pool, launches);
        if (e == cudaSuccess) {
            gather_values<int32_t><<<grid_for(nnz), kT, 0, st>>>(rowid, ix, t_col, nnz);
            e = gather_vals(val, ix, t_val, nnz, vb, st);
            launches += 2;
        }
    }
    if (e == cudaSuccess) e = offsets(col, nnz, K, t_row_ptr, pool, launches);
    if (e == cudaSuccess) e = cudaGetLastError();
    spx_note_launches(launches);
    if (pool.err != cudaSuccess) return SPX_ERR_NOMEM;
    return e == cudaSuccess ? SPX_OK : SPX_ERR_CUDA;
}
