// ssd_check.cu -- the optional finite-value check (SSD_FLAG_CHECK_FINITE).
//
// burn-mamba, "combined_backward.rs": every intermediate of the recompute
// backward is passed through `san(..)` right after it is formed.  Its body is not
// on the page; it is read here as a debug-time check that the tensor holds only
// finite values, with no numerical effect.  With the flag set, the last kernel
// of a call counts the non-finite elements of every output and of the
// intermediates that the call writes in full (cumA, endA, the chunk states and,
// in the backward, the chunk-state gradients) into status word 2 of the
// workspace.  Without the flag nothing here runs.
#include "ssd_check.cuh"

namespace ssd {

namespace {

__device__ __forceinline__ bool nonfinite_f32(uint32_t u) { return (u & 0x7F800000u) == 0x7F800000u; }
__device__ __forceinline__ bool nonfinite_bf16(uint32_t u16) { return (u16 & 0x7F80u) == 0x7F80u; }

// blockIdx.y selects the region; a grid-stride loop over its 32-bit words
// (a bf16 region's words hold two elements); one atomic per warp that saw
// something.
__global__ void check_finite_kernel(CheckList list, int *count) {
    const CheckRegion r = list.r[blockIdx.y];
    const size_t nwords = r.is_bf16 ? r.count / 2 : r.count;
    const uint32_t *w = (const uint32_t *)r.ptr;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    int bad = 0;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nwords; i += stride) {
        const uint32_t u = __ldg(w + i);
        bad += r.is_bf16 ? (int)nonfinite_bf16(u & 0xFFFFu) + (int)nonfinite_bf16(u >> 16)
                         : (int)nonfinite_f32(u);
    }
    // an odd bf16 element count leaves one element after the last whole word
    if (r.is_bf16 && (r.count & 1) && blockIdx.x == 0 && threadIdx.x == 0)
        bad += (int)nonfinite_bf16(((const unsigned short *)r.ptr)[r.count - 1]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(count, bad);
}

}  // namespace

cudaError_t launch_check_finite(const CheckList &list, int *count, cudaStream_t s) {
    if (list.n <= 0) return cudaSuccess;
    size_t biggest = 0;
    for (int i = 0; i < list.n; ++i) biggest = list.r[i].count > biggest ? list.r[i].count : biggest;
    const int threads = 256;
    // at most 2 waves of 152 SMs x 8 blocks across all regions
    size_t blocks = (biggest + threads - 1) / threads;
    const size_t cap = (size_t)(2 * 152 * 8) / (size_t)list.n + 1;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    check_finite_kernel<<<dim3((unsigned)blocks, (unsigned)list.n), threads, 0, s>>>(list, count);
    return cudaGetLastError();
}

}  // namespace ssd
