// Diagnostic used by the failure-detection tests: shows that a bounded wait
// that can never complete ends with SP_DEV_TIMEOUT in the caller's status
// word instead of hanging the GPU, using the same wait as the attention
// kernels.  One warp waits on an mbarrier that nothing ever arrives at.
#include <cuda_runtime.h>

#include "internal.h"
#include "pipeline.cuh"
#include "sm103_ptx.cuh"

namespace spc {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint32_t limit, int32_t *d_status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncwarp();
  const Ctl ctl{b, &abort_flag, d_status, limit};
  ctl.wait_warp(0, 0);  // phase 0 never completes: expires after `limit` polls
}

}  // namespace
}  // namespace spc

extern "C" int sp_debug_wait_timeout(int32_t spin_limit, int32_t *d_status, void *stream) {
  if (spin_limit < 256 || !d_status) return SP_ERR_INVALID_ARG;
  spc::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(uint32_t(spin_limit), d_status);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}
