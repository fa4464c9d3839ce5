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

// Small batches (a few hundred tokens at most): one block of G warps per
// token (group_local_topk / group_merge_topk), the token's logits and the
// bias staged through shared memory; a token whose candidates do not fit the
// group's pass is routed by warp 0 alone (route_token).
constexpr int kGroupWarps = 4;
constexpr int kGroupMaxT = 512;

template <int KPL, int G>
__global__ void __launch_bounds__(32 * G) route_group_kernel(const float* __restrict__ logits,
                                                             const float* __restrict__ bias, int E, int k,
                                                             int32_t* __restrict__ ids, float* __restrict__ wts) {
  constexpr int KPLG = (KPL + G - 1) / G;  // 32-expert blocks per warp
  __shared__ float s_lg[KPL * 32], s_b[KPL * 32];
  __shared__ float s_lk[G * kMaxK], s_ls[G * kMaxK];
  __shared__ int s_li[G * kMaxK];
  __shared__ int s_idx[G * 32];
  __shared__ int s_ok[G];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const float* lg = logits + static_cast<size_t>(t) * E;
  for (int e = threadIdx.x; e < E; e += 32 * G) {
    s_lg[e] = __ldg(lg + e);
    s_b[e] = __ldg(bias + e);
  }
  __syncthreads();
  const bool ok = group_local_topk<KPLG>(s_lg, s_b, E, k, lane, warp, G, s_lk + warp * k, s_li + warp * k,
                                         s_ls + warp * k, s_idx + warp * 32);
  if (lane == 0) s_ok[warp] = ok ? 1 : 0;
  __syncthreads();
  if (warp != 0) return;
  int all = 1;
  for (int q = 0; q < G; ++q) all &= s_ok[q];
  int32_t* ids_row = ids + static_cast<size_t>(t) * k;
  float* w_row = wts + static_cast<size_t>(t) * k;
  if (all)
    group_merge_topk(s_lk, s_li, s_ls, G, k, lane, ids_row, w_row);
  else
    route_token<KPL>(s_lg, s_b, E, k, lane, ids_row, w_row, s_idx);
}

cudaError_t launch_route(const float* logits, const float* bias, int T, int E, int k, int32_t* ids, float* wts,
                         cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (T <= kGroupMaxT && E >= 32 * kGroupWarps && k <= kMaxK) {
    // every warp of a group holds at least one whole block of 32 experts (at least k of them)
    const int kpl = (E + 31) / 32;
#define KMOE_ROUTE_GROUP(N)                                                                            \
  if (kpl <= N) {                                                                                      \
    route_group_kernel<N, kGroupWarps><<<T, 32 * kGroupWarps, 0, st>>>(logits, bias, E, k, ids, wts);  \
    return cudaGetLastError();                                                                         \
  }
    KMOE_ROUTE_GROUP(8)
    KMOE_ROUTE_GROUP(16)
    KMOE_ROUTE_GROUP(32)
#undef KMOE_ROUTE_GROUP
  }
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
