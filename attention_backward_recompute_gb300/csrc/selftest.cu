// attn_selftest_wait_timeout: exercises the failure detection every kernel of
// the library relies on.  Each spin of a kernel on an mbarrier is bounded:
// after ATTN_WAIT_TIMEOUT_NS it gives up, raises the CTA's abort flag, ORs
// DEV_ERR_TIMEOUT into the device error word and returns, so a lost producer
// or a stalled pipeline ends as an error status the host reads with
// attn_check_device_error, never as a hung GPU.  This kernel waits on a
// barrier that nothing arrives on, so that path can be tested on a GPU without
// any fault: it returns after one bounded wait and leaves the context usable.
#include <cuda_runtime.h>

#include "api_internal.h"
#include "sm103.cuh"

namespace {

__global__ void wait_timeout_kernel(uint32_t* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    sm103::mbar_init(&bar, 1);
    sm103::mbar_fence_init();
  }
  __syncwarp();
  const sm103::Abort ab{&abort_flag, err};
  sm103::mbar_wait_warp(&bar, 0, ab);  // phase 0 never completes: the wait expires
}

}  // namespace

ATTN_API attn_status_t attn_selftest_wait_timeout(void* stream) {
  uint32_t* err = attn::device_error_word();
  if (!err) return attn::api_fail(ATTN_ERR_CUDA, "no CUDA device");
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return attn::api_fail(ATTN_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
  return attn::api_ok();
}
