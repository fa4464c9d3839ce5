// Routing: sigmoid scores + e_score_correction_bias top-k with renormalised
// weights (Kimi-K3 SM120 FlashInfer MXFP4 page, serving call chain: the bias
// only takes part in choosing experts; the weights come from the un-biased
// sigmoid scores and are renormalised).
//
// One warp per token.  Lane l holds the keys of experts l, l+32, l+64, ...
// The selection key is fp32(sigmoid(logit)) + fp32(bias) with the sigmoid
// correctly rounded to fp32 (evaluated in double).  Double precision is slow
// on this part, so a radix select first finds the k-th largest cheap fp32
// key, and only experts whose cheap key lies within a safety margin of it
// (the margin is far above the error of expf) get the exact key; the final
// top-k is taken over exact keys, equal keys going to the lower expert index.
// Usually the candidates fit one per lane and are ranked in one pass; with
// more than 32 (many equal keys) k rounds of warp arg-max are used instead.
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
  // pass 1: the k-th largest cheap key, by a bitwise radix select over
  // order-preserving integer images of the keys (32 counting rounds)
  uint32_t okey[KPL];  // 0 for absent experts: below every probe
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const uint32_t u = __float_as_uint(key[i]);
    okey[i] = (lane + 32 * i < E) ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
  }
  uint32_t prefix = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t probe = prefix | (1u << bit);
    unsigned cnt = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) cnt += okey[i] >= probe;
    if (static_cast<int>(__reduce_add_sync(0xffffffffu, cnt)) >= k) prefix = probe;
  }
  const float kth = __uint_as_float((prefix & 0x80000000u) ? (prefix & 0x7fffffffu) : ~prefix);

  // fast path: gather the candidates (cheap key within the margin of the k-th)
  // into one lane each, take their exact keys and rank them across the warp
  {
    const float margin = 1e-5f * fmaxf(1.f, fabsf(kth));
    const float cut = (kth == NEG_INF) ? NEG_INF : kth - margin;
    __shared__ int s_idx[32];
    __shared__ float s_lg[32], s_b[32];
    int base = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int e = lane + 32 * i;
      const bool pred = e < E && key[i] >= cut;
      const unsigned m = __ballot_sync(0xffffffffu, pred);
      const int pos = base + __popc(m & ((1u << lane) - 1u));
      if (pred && pos < 32) {
        s_idx[pos] = e;
        s_lg[pos] = lgt[i];
        s_b[pos] = b[i];
      }
      base += __popc(m);
    }
    __syncwarp();
    if (base <= 32) {
      const bool have = lane < base;
      const int idx = have ? s_idx[lane] : 0x7fffffff;
      const float sv = have ? sigmoid_exact_f32(s_lg[lane]) : 0.f;
      float kx = have ? sv + s_b[lane] : NEG_INF;
      if (isnan(kx)) kx = NEG_INF;
      int rank = 0;
      for (int j = 0; j < 32; ++j) {
        const float kj = __shfl_sync(0xffffffffu, kx, j);
        const int ij = __shfl_sync(0xffffffffu, idx, j);
        rank += (kj > kx || (kj == kx && ij < idx)) ? 1 : 0;
      }
      const bool sel = have && rank < k;
      double sum = sel ? static_cast<double>(sv) : 0.0;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (sel) {
        ids[static_cast<size_t>(warp) * k + rank] = idx;
        wts[static_cast<size_t>(warp) * k + rank] = static_cast<float>(static_cast<double>(sv) / sum);
      }
      return;
    }
  }
  // general path (more than 32 candidates, e.g. many equal keys): k rounds of
  // warp arg-max over the exact keys of all candidates
  uint32_t taken = 0;
  // exact keys for the candidates: each lane evaluates one candidate per
  // round (all lanes in step)
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
