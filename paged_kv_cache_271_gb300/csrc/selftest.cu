// Self-test of failure detection in the kernels' waits. Every copy and MMA barrier wait in the
// decode and cascade kernels goes through mbar_wait, which gives up after its limit, records
// PKV_DEVERR_TIMEOUT and returns false, so a copy that never lands ends the kernel with a
// status instead of hanging the GPU. This launch makes that happen on purpose, safely: one
// thread waits on a barrier that nothing will ever complete (no copy, no arrival), the wait
// runs out after its limit (2 s), and the kernel reports what it saw and returns.
#include <cuda_runtime.h>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

__global__ void wait_timeout_kernel(int* err, int* done) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool got = mbar_wait(&bar, 0, err);  // no arrival: the wait runs out
    *done = got ? 2 : 1;
  }
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_selftest_wait_timeout(int32_t* err_dev, int32_t* done_dev, void* stream) {
  if (!err_dev || !done_dev)
    return pkv::set_error(PKV_EINVAL, "pkv_selftest_wait_timeout: null pointer");
  pkv::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err_dev, done_dev);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return pkv::set_error(PKV_ECUDA, "pkv_selftest_wait_timeout: %s", cudaGetErrorString(e));
  return PKV_OK;
}
