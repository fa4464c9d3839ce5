// Routing: sigmoid scores + e_score_correction_bias top-k with renormalised
// weights (Kimi-K3 SM120 FlashInfer MXFP4 page, serving call chain: the bias
// only takes part in choosing experts; the weights come from the un-biased
// sigmoid scores and are renormalised).
//
// One warp per token.  Lane l holds the keys of experts l, l+32, l+64, ...
// The selection key is fp32(sigmoid(logit)) + fp32(bias) with the sigmoid
// correctly rounded to fp32 (evaluated in double).  Double precision is slow
// on this part, so a first pass ranks cheap fp32 keys, and only experts whose
// cheap key lies within a safety margin of the k-th largest (the margin is
// far above the error of expf) get the exact key; the final top-k is taken
// over exact keys, equal keys going to the lower expert index.
#include "common.cuh"

namespace kmoe {

__device__ __forceinline__ float sigmoid_exact_f32(float x) {
  return static_cast<float>(1.0 / (1.0 + exp(-static_cast<double>(x))));
}

// warp arg-max of (key, idx): larger key wins, equal keys -> lower index
__device__ __forceinline__ void warp_argmax(float& key, int& idx) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ok = __shfl_xor_sync(0xffffffffu, key, off);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
    if (ok > key || (ok == key && oi < idx)) {
      key = ok;
      idx = oi;
    }
  }
}

template <int KPL>
__global__ void __launch_bounds__(32) route_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                    int T, int E, int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ wts) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* lg = logits + static_cast<size_t>(warp) * E;
  const float NEG_INF = -__int_as_float(0x7f800000);

  float lgt[KPL], b[KPL], key[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    lgt[i] = e < E ? lg[e] : 0.f;
    b[i] = e < E ? bias[e] : 0.f;
    float s = 1.f / (1.f + expf(-lgt[i]));
    float kf = s + b[i];
    key[i] = (e < E && !isnan(kf)) ? kf : NEG_INF;
  }
  // pass 1: k-th largest cheap key
  uint32_t taken = 0;
  float kth = NEG_INF;
  for (int j = 0; j < k; ++j) {
    float bk = NEG_INF;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (key[i] > bk || (key[i] == bk && e < bi))) {
        bk = key[i];
        bi = e;
      }
    }
    warp_argmax(bk, bi);
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    kth = bk;
  }
  // pass 2: exact keys for the candidates.  Each lane evaluates one candidate
  // per round (all lanes in step), so the double-precision work per warp is
  // the largest candidate count of any lane rather than the candidate total.
  const float margin = 1e-5f * fmaxf(1.f, fabsf(kth));
  const float cut = (kth == NEG_INF) ? NEG_INF : kth - margin;
  uint32_t cand = 0;
  float sx[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    sx[i] = 0.f;
    if (e < E && key[i] >= cut) cand |= 1u << i;
  }
  const uint32_t cand0 = cand;
  while (__any_sync(0xffffffffu, cand != 0)) {
    const int pick = cand ? __ffs(cand) - 1 : -1;
    float lv = 0.f, bv = 0.f;
#pragma unroll
    for (int i = 0; i < KPL; ++i)
      if (i == pick) {
        lv = lgt[i];
        bv = b[i];
      }
    const float sv = sigmoid_exact_f32(lv);
    float kx = sv + bv;
    if (isnan(kx)) kx = NEG_INF;
#pragma unroll
    for (int i = 0; i < KPL; ++i)
      if (i == pick) {
        sx[i] = sv;
        key[i] = kx;
      }
    if (pick >= 0) cand &= cand - 1;
  }
#pragma unroll
  for (int i = 0; i < KPL; ++i)
    if (!((cand0 >> i) & 1u)) key[i] = NEG_INF;  // not a candidate: cannot be chosen
  taken = 0;
  float mys = 0.f;
  int myid = -1;
  double sum = 0.0;
  for (int j = 0; j < k; ++j) {
    float bk = NEG_INF;
    int bi = 0x7fffffff;
    float bs = 0.f;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (key[i] > bk || (key[i] == bk && e < bi))) {
        bk = key[i];
        bi = e;
        bs = sx[i];
      }
    }
    warp_argmax(bk, bi);
    const int owner = bi & 31;
    bs = __shfl_sync(0xffffffffu, bs, owner);
    if (owner == lane) taken |= 1u << (bi >> 5);
    if (j == lane) {
      mys = bs;
      myid = bi;
    }
    sum += static_cast<double>(bs);
  }
  if (lane < k) {
    ids[static_cast<size_t>(warp) * k + lane] = myid;
    wts[static_cast<size_t>(warp) * k + lane] = static_cast<float>(static_cast<double>(mys) / sum);
  }
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
