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

#include <cuda.h>

#include "ssd.h"
#include "ssd_internal.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)SSD_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct CachedAddress {
    void *ptr = nullptr;
    unsigned long long ctx_id = 0;  // the driver's ID of the context the address belongs to
};
CachedAddress g_cache[kMaxDevices];

// The driver's ID of the calling thread's current context (0 when there is none
// or the driver does not offer the query).  Taken through the runtime's driver
// entry points, so the library does not link the driver library directly.
unsigned long long current_context_id() {
    typedef CUresult (*GetCurrent)(CUcontext *);
    typedef CUresult (*GetId)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = (GetCurrent)f;
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = (GetId)f;
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array on the current device, looked up once
// per device and context (the lookup may load this module onto the device and
// makes the device's primary context current).  `lookup` false: report the
// cached address only (SSD_ERR_INVALID_ARG when there is none).
ssd_status scratch_for_current_device(void **out, bool lookup) {
    char msg[256];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "ssd_forward_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
        ssd::record_error(msg);
        return SSD_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg), "ssd_forward_noalloc: device %d is beyond the library's %d-device table",
                 dev, kMaxDevices);
        ssd::record_error(msg);
        return SSD_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    CachedAddress &c = g_cache[dev];
    const unsigned long long id = current_context_id();
    if (c.ptr && id == c.ctx_id) {
        *out = c.ptr;
        return SSD_OK;
    }
    if (!lookup) {
        snprintf(msg, sizeof(msg), "ssd_noalloc_status: no ssd_forward_noalloc call yet on device %d", dev);
        ssd::record_error(msg);
        return SSD_ERR_INVALID_ARG;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
        snprintf(msg, sizeof(msg), "ssd_forward_noalloc: cudaGetSymbolAddress(scratch) failed on device %d: %s",
                 dev, cudaGetErrorString(e));
        ssd::record_error(msg);
        return SSD_ERR_CUDA;
    }
    c.ptr = p;
    c.ctx_id = current_context_id();  // the lookup has made the primary context current
    *out = p;
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
    st = scratch_for_current_device(&scratch, true);
    if (st != SSD_OK) return st;
    // ssd_forward clears the only part of the workspace that must start at
    // zero (the status words at its start); everything else is written before
    // it is read.
    return ssd_forward(dims, dtype, x, dt, A, B, C, D, init_state, valid_len, y, final_state, scratch,
                       kScratchBytes, stream);
}

ssd_status ssd_noalloc_status(void *stream) {
    void *scratch = nullptr;
    const ssd_status st = scratch_for_current_device(&scratch, false);
    if (st != SSD_OK) return st;
    return ssd::read_status_words(scratch, (cudaStream_t)stream);
}

}  // extern "C"
