// spx_bsr.cu -- BSR SpMM on the tensor cores (placeholder until the tcgen05 kernel lands).
#include <cuda_runtime.h>

#include "spx_internal.h"

extern "C" {

spx_status spx_spmm_bsr(int32_t, int32_t, int32_t, int32_t, int64_t, const int32_t*, const int32_t*, const uint16_t*,
                        int32_t, const uint16_t*, int64_t, float*, int64_t, spx_stream_t) {
    return SPX_ERR_UNSUPPORTED;
}

spx_status spx_last_device_error(spx_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPX_OK : SPX_ERR_CUDA;
}

}  // extern "C"
