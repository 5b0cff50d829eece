// spx_check.cuh -- the bounds-checked build (compiled with -DSPX_CHECK into
// libspx_check.so; the product library is built without it).
//
// A compute-sanitizer run reports an out-of-range access after the fact, by
// faulting; this build instead tests every index a kernel reads from the
// caller's arrays before it uses it -- a column against K, a row offset
// against the matrix and the plan -- skips the access when the test fails
// (the term counts as zero, a group with inconsistent offsets is not
// reduced) and records SPX_ERR_INDEX_RANGE in the calling translation unit's
// error word, which spx_last_device_error reports.  With valid inputs the
// checked build computes exactly what the product build computes.
#pragma once

#ifdef SPX_CHECK
#define SPX_CHECKED true
#else
#define SPX_CHECKED false
#endif

// One error word per translation unit that instruments its kernels:
//   SPX_CHECK_WORD(g_word)  defines the word and check_fail() setting it;
//   spx_check_take(g_word)  (host) reads and clears it: 0, or SPX_ERR_INDEX_RANGE.
#define SPX_CHECK_WORD(word)                                                         \
    __device__ int word;                                                             \
    __device__ __forceinline__ void check_fail() { atomicExch(&word, 1); }

#ifdef SPX_CHECK
#define spx_check_take(word)                                                                   \
    ([]() -> int {                                                                             \
        int h = 0;                                                                             \
        const int zero = 0;                                                                    \
        if (cudaMemcpyFromSymbol(&h, word, sizeof(int)) != cudaSuccess) return SPX_ERR_CUDA;   \
        if (h != 0 && cudaMemcpyToSymbol(word, &zero, sizeof(int)) != cudaSuccess)             \
            return SPX_ERR_CUDA;                                                               \
        return h ? static_cast<int>(SPX_ERR_INDEX_RANGE) : 0;                                  \
    }())
#else
#define spx_check_take(word) 0
#endif
