// Internal declarations shared by the host and device translation units of libspx.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "spx.h"

// Counts kernel launches (reported by spx_launch_count).
void spx_note_launches(uint64_t n);

// Status of the last CUDA runtime error, or SPX_OK.
spx_status spx_cuda_status(int cuda_error);

struct spx_plan {
    int32_t M = 0, K = 0;
    int64_t nnz = 0;
    spx_plan_opts_t opts{};
    std::vector<int32_t> tasks;     // 4 per task
    std::vector<int32_t> longrows;  // 4 per split row
    int64_t counts[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    spx_row_stats_t stats{};
    const void* d_table = nullptr;  // caller-owned copy of tasks + longrows
    size_t table_bytes = 0;
    size_t scratch_bytes = 0;
    uint64_t magic = 0;
};

constexpr uint64_t kPlanMagic = 0x5350585f504c414eull;  // "SPX_PLAN"

enum : int32_t { kTaskGroup = 0, kTaskCta = 1, kTaskSeg = 2 };

inline bool spx_plan_ok(const spx_plan* p) { return p && p->magic == kPlanMagic; }

inline bool spx_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t kI32Max = 2147483647LL;
