// Self-test of the bounded pipeline waits.  Every mbarrier wait in the library's
// kernels gives up after a wall-clock limit (about one second), records
// DLLM_DEV_TIMEOUT in the cache's status word and lets the kernel end, so a stalled
// pipeline never hangs the device.  This kernel waits on an mbarrier that nothing
// arrives at, with the same wait routine, to show that path end to end.
#include "internal.h"
#include "ptx.cuh"

namespace dllm {
namespace {

__global__ void wait_timeout_kernel(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none will come
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag)) atomicOr(status, DLLM_DEV_TIMEOUT);
}

}  // namespace
}  // namespace dllm

extern "C" int dllm_selftest_wait_timeout(dllm_cache* c, void* stream) {
  if (!c) return DLLM_EINVAL;
  int dev = -1;  // the cache's device must be current (its status word lives there)
  if (cudaGetDevice(&dev) != cudaSuccess || dev != c->device) {
    cudaGetLastError();
    return DLLM_EINVAL;
  }
  dllm::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(c->status);
  return cudaGetLastError() == cudaSuccess ? DLLM_OK : DLLM_ECUDA;
}
