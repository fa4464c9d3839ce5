// Routing of one token by one warp: sigmoid scores + e_score_correction_bias
// top-k with renormalised weights (Kimi-K3 SM120 FlashInfer MXFP4 page,
// serving call chain: the bias only takes part in choosing experts; the
// weights come from the un-biased sigmoid scores and are renormalised).
//
// Lane l holds the keys of experts l, l+32, l+64, ...  The selection key is
// fp32(sigmoid(logit)) + fp32(bias) with the sigmoid correctly rounded to fp32
// (evaluated in double).  Double precision is slow on this part, so the top-k
// is first narrowed with cheap fp32 keys (fast exponential, see
// candidate_cut) and only the candidates get the exact key; the final top-k
// is taken over exact keys, equal keys going to the lower expert index.
//   1. A lower bound of the k-th largest cheap key: the k-th largest of the
//      32 lane maxima (k lanes each hold a key at least that large).  Experts
//      whose cheap key is within the margin of it are the candidates; usually
//      they fit one per lane and are ranked by exact key in one pass.
//   2. Otherwise (more than 32 candidates), the exact k-th largest cheap key
//      by a bitwise radix select, and the candidates within the margin of it.
//   3. If those are still more than 32 (many equal keys): k rounds of warp
//      arg-max over the candidates' exact keys.
//
// Used by the routing kernel (logits given) and by the fused router kernel
// (logits produced by its own GEMM phase).
#pragma once
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

// Cut (an order key) for the candidates of a k-th largest cheap key `kth`:
// everything within the safety margin below it.  The margin, 1e-5 x
// max(1, |kth|), is at least twice the largest difference between a cheap
// key and its exact key (below 2e-6: the fast exponential's relative error,
// at most |x| 2^-24 plus a few ulp for |x| <= 88, moves the sigmoid by at
// most a quarter of it; beyond, both sigmoids are 0 or 1 to fp32 accuracy),
// so every expert of the exact top k is a candidate: its cheap key is at
// least the k-th largest cheap key minus twice that difference.
__device__ __forceinline__ uint32_t candidate_cut(float kth) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float margin = 1e-5f * fmaxf(1.f, fabsf(kth));
  return order_key((kth == NEG_INF) ? NEG_INF : kth - margin);
}

// Bitonic sort of one value per lane across the warp into descending order
// (lane 0 the largest): 15 compare-exchange steps of one shuffle each, in
// place of 32 rounds of broadcast-and-count.  `before(a, i, b, j)` says
// whether (a, i) precedes (b, j); the payload p travels with its key.
template <class K, class Before>
__device__ __forceinline__ void warp_sort_desc(K& key, int& idx, float& p, int lane, Before before) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const K ok = __shfl_xor_sync(0xffffffffu, key, stride);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, stride);
      const float op = __shfl_xor_sync(0xffffffffu, p, stride);
      const bool lower = (lane & stride) == 0;   // lower lane of the pair
      const bool desc = (lane & size) == 0;      // this block sorts descending
      const bool mine_first = before(key, idx, ok, oi);
      if (mine_first != (lower == desc)) {
        key = ok;
        idx = oi;
        p = op;
      }
    }
  }
}

// Candidates (order key >= ocut) one per lane, ranked by exact key across the
// warp; writes the top k and returns true, or returns false (nothing written)
// when there are more than 32 candidates.
template <int KPL>
__device__ __forceinline__ bool select_ranked(const uint32_t (&okey)[KPL], uint32_t ocut, const float* lg,
                                              const float* bias, int E, int k, int lane, int32_t* ids_row,
                                              float* wts_row, int* s_idx) {
  const float NEG_INF = -__int_as_float(0x7f800000);
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
  if (base > 32) {
    __syncwarp();
    return false;
  }
  const bool have = lane < base;
  int idx = have ? s_idx[lane] : 0x7fffffff;
  float sv = 0.f;
  float kx = have ? exact_key(lg, bias, idx, sv) : NEG_INF;
  // sorted by exact key (equal keys: lower expert id first); lane r holds rank r
  warp_sort_desc(kx, idx, sv, lane,
                 [](float a, int i, float b, int j) { return a > b || (a == b && i < j); });
  const bool sel = lane < k;  // base >= k: every rank below k is a candidate
  double sum = sel ? static_cast<double>(sv) : 0.0;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (sel) {
    ids_row[lane] = idx;
    wts_row[lane] = __fdiv_rn(sv, static_cast<float>(sum));
  }
  __syncwarp();  // s_idx is reused by this warp's next token
  return true;
}

// Routes one token.  `lg` (the token's E logits) and `bias` may be in shared
// or global memory (generic pointers; global data must already be visible to
// this thread).  `s_idx` is 32 ints of this warp's shared memory.  Writes the
// k ids in descending key order and their weights to ids_row / wts_row.
template <int KPL>
__device__ __forceinline__ void route_token(const float* lg, const float* bias, int E, int k, int lane,
                                            int32_t* ids_row, float* wts_row, int* s_idx) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  // only the integer images of the cheap keys live in registers
  uint32_t okey[KPL];  // 0 for absent experts: below every key
  float lv[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    lv[i] = e < E ? lg[e] : 0.f;
  }
  uint32_t lmax = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    okey[i] = 0u;
    if (e < E) {
      const float kf = __fdividef(1.f, 1.f + __expf(-lv[i])) + bias[e];
      okey[i] = order_key(isnan(kf) ? NEG_INF : kf);
    }
    lmax = okey[i] > lmax ? okey[i] : lmax;
  }
  // 1. the k-th largest lane maximum (ranks 0..31, ties by lane) bounds the
  //    k-th largest cheap key from below
  {
    uint32_t sk = lmax;
    int sl = lane;
    float unused = 0.f;
    warp_sort_desc(sk, sl, unused, lane, [](uint32_t a, int i, uint32_t b, int j) { return a > b || (a == b && i < j); });
    const float lb = order_key_inverse(__shfl_sync(0xffffffffu, sk, k - 1));
    if (select_ranked<KPL>(okey, candidate_cut(lb), lg, bias, E, k, lane, ids_row, wts_row, s_idx)) return;
  }
  // 2. the exact k-th largest cheap key, by a bitwise radix select over the
  //    integer images (32 counting rounds)
  uint32_t prefix = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t probe = prefix | (1u << bit);
    unsigned cnt = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) cnt += okey[i] >= probe;
    if (static_cast<int>(__reduce_add_sync(0xffffffffu, cnt)) >= k) prefix = probe;
  }
  const uint32_t ocut = candidate_cut(order_key_inverse(prefix));
  if (select_ranked<KPL>(okey, ocut, lg, bias, E, k, lane, ids_row, wts_row, s_idx)) return;
  // 3. more than 32 candidates (e.g. many equal keys): k rounds of warp
  //    arg-max over the exact keys of the candidates not taken yet (exact keys
  //    recomputed each round: this path is rare)
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
        const float kx = exact_key(lg, bias, e, sv);
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
    ids_row[lane] = myid;
    wts_row[lane] = static_cast<float>(static_cast<double>(mys) / sum);
  }
  __syncwarp();
}

}  // namespace kmoe
