// ssd_tc.cu -- tcgen05 tensor-core kernels of the bf16 path.
#include "ssd_tc.cuh"

namespace ssd {

bool tc_supported(int64_t, int64_t, int64_t) { return false; }
int tc_dD_per(int64_t) { return 1; }
int tc_group_slices(const ssd_dims &) { return 1; }

cudaError_t launch_tc_k2(const Params &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_k3(const Params &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_k5(const Params &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_bwd_blue(const Params &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_bwd_main(const Params &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_bwd_group(const Params &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ssd
