// ssd_tc.cuh -- tcgen05 tensor-core kernels of the bf16 path (ssd_tc.cu).
#pragma once
#include "ssd.h"
#include "ssd_internal.cuh"

namespace ssd {

// True when the tensor-core kernels cover (headdim, dstate, chunk_len).
bool tc_supported(int64_t P, int64_t N, int64_t Q);
// dD partials per (b, chunk, head) written by the tensor-core main backward.
int tc_dD_per(int64_t Q);
// Head slices of the group-level backward: d_cb partial sums (first) and the
// dB / dC partial sums (second).
int tc_dcb_slices(const ssd_dims &d);
// Head slices of the persistent per-group kernels (K5, K3 and ORANGE backward).
int tc_k5_slices(const ssd_dims &d);
// Head slices of the streaming per-group kernels (K3 forward, BLUE backward).
int tc_k3_slices(const ssd_dims &d);
int tc_group_slices(const ssd_dims &d);

// Fused K1 + K3 + K4 (cumA, endA and the bf16 chunk-input states; final state when asked).
cudaError_t launch_tc_state_scan(const Params &p, bool write_final, cudaStream_t s);
// CTAs of the chunk-state scan's grid (one per (b, group, head pair or head))
long long tc_state_scan_ctas(const Params &p);
// one bounded wait (the kernels' own) that gives up after limit_ns unless arrive
cudaError_t launch_wait_selftest(int *status, uint64_t limit_ns, int arrive, cudaStream_t s);
// Closed-form state moments per (b, h, chunk range): partial A and m1 into p.mom_A, p.mom_m1.
cudaError_t launch_tc_moments(const Params &p, cudaStream_t s);
cudaError_t launch_tc_k2(const Params &p, cudaStream_t s);
cudaError_t launch_tc_k3(const Params &p, cudaStream_t s);
cudaError_t launch_tc_k5(const Params &p, cudaStream_t s);
cudaError_t launch_tc_bwd_blue(const Params &p, cudaStream_t s);
cudaError_t launch_tc_bwd_k3(const Params &p, cudaStream_t s);
cudaError_t launch_tc_bwd_orange(const Params &p, cudaStream_t s);
cudaError_t launch_tc_bwd_dcb(const Params &p, cudaStream_t s);         // G1: d_cb over the group's heads
cudaError_t launch_tc_bwd_dbc(const Params &p, cudaStream_t s);         // G2: dB, dC partial sums
cudaError_t launch_tc_bwd_dbc_reduce(const Params &p, cudaStream_t s);  // G3: sum of the partials

}  // namespace ssd
