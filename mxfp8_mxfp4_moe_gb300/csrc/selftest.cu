// Small kernels used by kmoe_check_device (does the sm_103a image load?), by
// kmoe_selftest_wait_timeout (a bounded wait on a barrier nobody arrives at
// must give up and raise the timeout bit, leaving the context usable) and by
// kmoe_selftest_activation (the FC1 epilogue's activation, elementwise).
#include "gemm_dev.cuh"

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

// out[i] = the activation the FC1 epilogue applies to (gate[i], up[i]): the
// same device functions with the same parameters.
__global__ void activation_selftest_kernel(const float* __restrict__ g, const float* __restrict__ u, int n, int act,
                                           float kg, float ku, float bb, float alpha, float beta, float limit,
                                           float* __restrict__ out) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = act == 0 ? situ_f32(g[i], u[i], kg, ku, bb) : swiglu_f32(g[i], u[i], alpha, beta, limit);
}

cudaError_t launch_activation_selftest(const float* g, const float* u, int n, int act, float kg, float ku, float bb,
                                       float alpha, float beta, float limit, float* out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
  activation_selftest_kernel<<<blocks, 256, 0, st>>>(g, u, n, act, kg, ku, bb, alpha, beta, limit, out);
  return cudaGetLastError();
}

}  // namespace kmoe
