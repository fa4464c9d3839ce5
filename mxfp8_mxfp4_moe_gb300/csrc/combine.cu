// Routing-weighted combine (the non-fused, deterministic finalize of the
// Kimi-K3 SM120 FlashInfer MXFP4 page, Phase 2):
//   out[t, h] = bf16_rn( rsf * sum_{j=0..k-1} w[t, j] * y[t*k + j, h] )
// summed in fp32 in slot order; slots with a negative expert id are skipped.
// Blocks cover (token, slice of H): enough blocks to fill the GPU even for a
// handful of tokens; 16-byte loads of the fp32 rows.
#include <cuda_bf16.h>

#include "common.cuh"

namespace kmoe {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ ids,
                                                      const float* __restrict__ w, int H, int k, int E, float rsf,
                                                      __nv_bfloat16* __restrict__ out) {
  chain_wait();
  __shared__ float s_w[kMaxK];
  const int t = blockIdx.x;
  const int H4 = H / 4;
  const int h_begin = blockIdx.y * blockDim.x;  // one float4 per thread per slice
  if (threadIdx.x < k) {
    const int id = ids[static_cast<size_t>(t) * k + threadIdx.x];
    s_w[threadIdx.x] = (id >= 0 && id < E) ? w[static_cast<size_t>(t) * k + threadIdx.x] : 0.f;
  }
  __syncthreads();
  const float4* y4 = reinterpret_cast<const float4*>(y + static_cast<size_t>(t) * k * H);
  for (int h = h_begin + threadIdx.x; h < H4; h += blockDim.x * gridDim.y) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float wj = s_w[j];
      if (wj == 0.f) continue;  // masked slot: its y row was never written
      const float4 v = __ldcs(y4 + static_cast<size_t>(j) * H4 + h);
      acc.x = fmaf(wj, v.x, acc.x);
      acc.y = fmaf(wj, v.y, acc.y);
      acc.z = fmaf(wj, v.z, acc.z);
      acc.w = fmaf(wj, v.w, acc.w);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * rsf, acc.y * rsf);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * rsf, acc.w * rsf);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * H)[h] = pk;
  }
}

cudaError_t launch_combine(const float* y, const int32_t* ids, const float* w, int T, int H, int k, int E, float rsf,
                           void* out, cudaStream_t st, bool pdl) {
  if (T == 0) return cudaSuccess;
  const int slices = (H / 4 + 255) / 256;
  const int split = T >= 1024 ? 1 : slices;  // few tokens: one block per (token, H slice)
  return launch_chained(combine_kernel, dim3(T, split), dim3(256), 0, st, pdl, y, ids, w, H, k, E, rsf,
                        static_cast<__nv_bfloat16*>(out));
}

}  // namespace kmoe
