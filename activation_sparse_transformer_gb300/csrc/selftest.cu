// Self-test of the pipelines' failure detection: every mbarrier wait in the
// GEMM and SpMM kernels is bounded (mbar_wait gives up after a time limit and
// the kernel reports TWELL_ERR_WAIT_TIMEOUT on the status word instead of
// hanging).  This kernel runs that same wait on a barrier nothing ever
// arrives on, so a test can see the limit expire, the status set and the
// context stay usable, without faulting or hanging the GPU.
#include <cuda_runtime.h>

#include "sm103.cuh"
#include "twell_internal.h"

namespace twell {
namespace {

__global__ void wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns, &abort_flag)) report_error(status, TWELL_ERR_WAIT_TIMEOUT);
}

}  // namespace
}  // namespace twell

extern "C" int twell_selftest_wait_timeout(int32_t* status, uint64_t limit_ns, twell_stream_t stream) {
  if (!status || limit_ns == 0 || limit_ns > 10000000000ull) return TWELL_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(status) & 3u) != 0) return TWELL_ERR_MISALIGNED;
  if (!twell::device_is_sm103()) return TWELL_ERR_NO_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  twell::wait_timeout_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}
