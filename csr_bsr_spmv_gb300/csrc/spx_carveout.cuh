// spx_carveout.cuh -- L1 / shared-memory split for the gather-bound kernels.
//
// L1 and shared memory share one array per SM, and the split is chosen per
// kernel from a preference.  The SpMV-family kernels gather x (or rows of B)
// through L1, so they ask for just the shared memory their full occupancy
// needs -- resident CTAs x (dynamic + static + reserved shared memory) -- and
// leave the rest to L1.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

namespace spx_carve {

struct State {
    std::mutex mu;
    std::map<std::tuple<const void*, int, size_t>, int> pct;  // (kernel, device, dynamic smem) -> percent
    std::map<std::tuple<const void*, int>, int> current;      // (kernel, device) -> percent last set
};

inline State& state() {
    static State s;
    return s;
}

// Sets the kernel's carveout preference for a launch of `threads`-thread CTAs
// with `smem` bytes of dynamic shared memory (a no-op when already set).
template <class K>
inline cudaError_t fit(K* kernel, int threads, size_t smem) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const void* kp = reinterpret_cast<const void*>(kernel);
    State& S = state();
    std::lock_guard<std::mutex> lock(S.mu);
    auto key = std::make_tuple(kp, dev, smem);
    auto it = S.pct.find(key);
    int pct = 0;
    if (it != S.pct.end()) {
        pct = it->second;
    } else {
        // resident CTAs per SM with the largest shared-memory split, from the
        // thread, CTA, register and shared-memory limits (the occupancy
        // calculator itself would see the split already chosen)
        int per_sm = 0, reserved = 0, max_thr = 0, max_blk = 0, regs_sm = 0;
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, kernel);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&max_thr, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&max_blk, cudaDevAttrMaxBlocksPerMultiprocessor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
        if (e != cudaSuccess) return e;
        const uint64_t per_block = smem + fa.sharedSizeBytes + reserved;
        const int warps = (threads + 31) / 32;
        const int warp_regs = (fa.numRegs * 32 + 255) / 256 * 256;  // allocated per warp in units of 256
        int blocks = threads > 0 ? max_thr / threads : 0;
        if (max_blk < blocks) blocks = max_blk;
        if (warp_regs > 0 && regs_sm / (warp_regs * warps) < blocks) blocks = regs_sm / (warp_regs * warps);
        if (per_block > 0 && static_cast<int>(per_sm / per_block) < blocks) blocks = static_cast<int>(per_sm / per_block);
        const uint64_t need = static_cast<uint64_t>(blocks) * per_block;
        pct = per_sm > 0 ? static_cast<int>((need * 100 + per_sm - 1) / per_sm) : -1;
        if (pct > 100) pct = 100;
        S.pct[key] = pct;
    }
    auto ck = std::make_tuple(kp, dev);
    auto cur = S.current.find(ck);
    if (cur != S.current.end() && cur->second == pct) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, pct);
    if (e == cudaSuccess) S.current[ck] = pct;
    return e;
}

}  // namespace spx_carve
