// Small kernels used by kmoe_check_device (does the sm_103a image load?) and
// by kmoe_selftest_wait_timeout (a bounded wait on a barrier nobody arrives
// at must give up and raise the timeout bit, leaving the context usable).
#include "common.cuh"

namespace kmoe {

__global__ void kmoe_probe_kernel() {}

__global__ void wait_selftest_kernel(uint32_t* err, uint64_t budget_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, budget_ns, err, nullptr);
}

cudaError_t launch_wait_selftest(uint32_t* err, uint64_t budget_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, budget_ns);
  return cudaGetLastError();
}

}  // namespace kmoe
