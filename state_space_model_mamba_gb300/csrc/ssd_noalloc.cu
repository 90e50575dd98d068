// ssd_noalloc.cu -- ssd_forward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a memory
// pool or arena that owns every device allocation, plug-ins whose host
// framework forbids allocation on the hot path, and code that must not
// allocate while another component is capturing or replaying work.  They can
// still run the forward through ssd_forward_noalloc, whose scratch (the
// workspace ssd_forward otherwise takes from the caller) is a fixed array in
// this library's device memory.
//
// The array below is created when the library's code is loaded onto a GPU
// and stays there until the process exits, on every GPU that loads it.
#include <mutex>
#include <stdio.h>

#include "ssd.h"
#include "ssd_internal.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)SSD_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (the lookup may load this module onto the device).
ssd_status scratch_for_current_device(void **out) {
    char msg[256];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg), "ssd_forward_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
        ssd::record_error(msg);
        return SSD_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            snprintf(msg, sizeof(msg), "ssd_forward_noalloc: cudaGetSymbolAddress(scratch) failed on device %d: %s",
                     dev, cudaGetErrorString(e));
            ssd::record_error(msg);
            return SSD_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SSD_OK;
}

}  // namespace

extern "C" {

ssd_status ssd_forward_noalloc(const ssd_dims *dims, ssd_dtype dtype, const void *x, const float *dt,
                               const float *A, const void *B, const void *C, const float *D,
                               const float *init_state, const int32_t *valid_len, void *y,
                               float *final_state, void *stream) {
    ssd_status st = ssd_supported(dims, dtype);
    if (st != SSD_OK) return st;
    const size_t need = ssd_workspace_bytes(dims, dtype, 0);
    if (need > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "ssd_forward_noalloc: this shape needs %zu bytes of scratch, more than the %zu-byte "
                 "static array (SSD_NOALLOC_SCRATCH_BYTES); use ssd_forward with a caller workspace",
                 need, kScratchBytes);
        ssd::record_error(msg);
        return SSD_ERR_UNSUPPORTED;
    }
    void *scratch = nullptr;
    st = scratch_for_current_device(&scratch);
    if (st != SSD_OK) return st;
    // ssd_forward clears the only part of the workspace that must start at
    // zero (the device status word); everything else is written before it is read.
    return ssd_forward(dims, dtype, x, dt, A, B, C, D, init_state, valid_len, y, final_state, scratch,
                       kScratchBytes, stream);
}

}  // extern "C"
