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

// Order-preserving image of a non-NaN float as an unsigned integer (-0 and
// +0 map to the same value).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_inverse(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// Exact selection key of expert e (NaN -> -inf) and its sigmoid score.
__device__ __forceinline__ float exact_key(const float* lg, const float* bias, int e, float& score) {
  score = sigmoid_exact_f32(lg[e]);
  const float kx = score + bias[e];
  return isnan(kx) ? -__int_as_float(0x7f800000) : kx;
}

// Only the integer images of the cheap keys live in registers (KPL per
// lane); the candidates' exact keys are computed from the shared-memory copy
// of the token's logits and the bias.
template <int KPL>
__global__ void __launch_bounds__(32) route_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                    int T, int E, int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ wts) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* lg = logits + static_cast<size_t>(warp) * E;
  const float NEG_INF = -__int_as_float(0x7f800000);

  // the token's logits and the bias through shared memory: all loads are
  // independent and in flight together before any key is computed
  __shared__ float s_lg[KPL * 32], s_b[KPL * 32];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      s_lg[e] = __ldg(lg + e);
      s_b[e] = __ldg(bias + e);
    }
  }
  __syncwarp();
  uint32_t okey[KPL];  // 0 for absent experts: below every probe
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    okey[i] = 0u;
    if (e < E) {
      const float kf = 1.f / (1.f + expf(-s_lg[e])) + s_b[e];
      okey[i] = order_key(isnan(kf) ? NEG_INF : kf);
    }
  }
  // pass 1: the k-th largest cheap key, by a bitwise radix select over the
  // integer images (32 counting rounds)
  uint32_t prefix = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t probe = prefix | (1u << bit);
    unsigned cnt = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) cnt += okey[i] >= probe;
    if (static_cast<int>(__reduce_add_sync(0xffffffffu, cnt)) >= k) prefix = probe;
  }
  const float kth = order_key_inverse(prefix);
  // candidates: cheap key within the margin of the k-th
  const float margin = 1e-5f * fmaxf(1.f, fabsf(kth));
  const uint32_t ocut = order_key((kth == NEG_INF) ? NEG_INF : kth - margin);

  // fast path: the candidates one per lane, exact keys ranked across the warp
  {
    __shared__ int s_idx[32];
    int base = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int e = lane + 32 * i;
      const bool pred = e < E && okey[i] >= ocut;
      const unsigned m = __ballot_sync(0xffffffffu, pred);
      const int pos = base + __popc(m & ((1u << lane) - 1u));
      if (pred && pos < 32) s_idx[pos] = e;
      base += __popc(m);
    }
    __syncwarp();
    if (base <= 32) {
      const bool have = lane < base;
      const int idx = have ? s_idx[lane] : 0x7fffffff;
      float sv = 0.f;
      const float kx = have ? exact_key(s_lg, s_b, idx, sv) : NEG_INF;
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
  // warp arg-max over the exact keys of the candidates not taken yet (exact
  // keys recomputed each round: this path is rare)
  uint32_t taken = 0;
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
      if (e < E && okey[i] >= ocut && !((taken >> i) & 1u)) {
        float sv;
        const float kx = exact_key(s_lg, s_b, e, sv);
        if (kx > bk || (kx == bk && e < bi)) {
          bk = kx;
          bi = e;
          bs = sv;
        }
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
