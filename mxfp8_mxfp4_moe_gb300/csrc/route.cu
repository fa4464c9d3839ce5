// Routing kernel for given logits (the per-token selection is in
// route_dev.cuh).
#include "route_dev.cuh"

namespace kmoe {

// One warp per token; the token's logits and the bias are staged through
// shared memory so that all loads are independent and in flight together
// before any key is computed.
template <int KPL>
__global__ void __launch_bounds__(32) route_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                    int T, int E, int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ wts) {
  chain_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* lg = logits + static_cast<size_t>(warp) * E;
  __shared__ float s_lg[KPL * 32], s_b[KPL * 32];
  __shared__ int s_idx[32];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      s_lg[e] = __ldg(lg + e);
      s_b[e] = __ldg(bias + e);
    }
  }
  __syncwarp();
  route_token<KPL>(s_lg, s_b, E, k, lane, ids + static_cast<size_t>(warp) * k, wts + static_cast<size_t>(warp) * k,
                   s_idx);
}

cudaError_t launch_route(const float* logits, const float* bias, int T, int E, int k, int32_t* ids, float* wts,
                         cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  // one warp per block: the double-precision sigmoids of a few tokens spread over many SMs
  const int blocks = T;
  const int kpl = (E + 31) / 32;
#define KMOE_ROUTE(N)                                                             \
  if (kpl <= N) {                                                                 \
    route_kernel<N><<<blocks, 32, 0, st>>>(logits, bias, T, E, k, ids, wts);      \
    return cudaGetLastError();                                                    \
  }
  KMOE_ROUTE(1)
  KMOE_ROUTE(2)
  KMOE_ROUTE(4)
  KMOE_ROUTE(8)
  KMOE_ROUTE(16)
  KMOE_ROUTE(32)
#undef KMOE_ROUTE
  return cudaErrorInvalidValue;
}

}  // namespace kmoe
