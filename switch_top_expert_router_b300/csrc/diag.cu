// Diagnostic kernel for the failure-detection path: a bounded wait that is
// bound to expire.  See switch_moe_selftest_wait_timeout in switch_moe.h.
#include "common.cuh"
#include "ptx.cuh"

namespace smoe {
namespace {

__global__ void selftest_wait_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // No thread or copy ever arrives on `bar`: phase 0 never completes.
    mbar_wait(&bar, 0u, &abort_flag, status, SWITCH_MOE_ERR_DEVICE_TIMEOUT, timeout_ns);
  }
}

}  // namespace

cudaError_t launch_selftest_wait(int* status, unsigned long long timeout_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace smoe
