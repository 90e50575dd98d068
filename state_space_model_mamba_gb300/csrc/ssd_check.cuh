// ssd_check.cuh -- the optional finite-value check of a call's outputs and
// intermediates (ssd_check.cu; not part of the ABI).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssd {

struct CheckRegion {
    const void *ptr;  // device pointer, 4-byte aligned
    size_t count;     // elements
    int is_bf16;      // 1: bf16 elements, 0: fp32 elements
};

constexpr int kMaxCheckRegions = 16;
struct CheckList {
    CheckRegion r[kMaxCheckRegions];
    int n;
};

// Adds the number of NaN / infinite elements of every region to *count (a
// device int).  One launch; nothing is enqueued when list.n == 0.
cudaError_t launch_check_finite(const CheckList &list, int *count, cudaStream_t s);

}  // namespace ssd
