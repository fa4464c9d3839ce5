// Device pieces shared by the one-CTA and the CTA-pair expert GEMM kernels:
// work-item decoding, the SiTU activation (and the SwiGLU control) and the
// epilogue of one 32-column accumulator chunk.
#pragma once
#include <cuda_fp8.h>

#include "gemm.cuh"

namespace kmoe {

struct Work {
  int e, m, tile, r0, n;  // m: weight-tile group (tiles NT*m + j)
};

// Shared-memory bytes of the tile_start copy (E+1 <= kMaxE+1 ints).
constexpr int kTileStartBytes = ((kMaxE + 1) * 4 + 255) / 256 * 256;

// Copy tile_start[0..E] into shared memory; every thread of the CTA takes
// part, before the CTA's first barrier.
__device__ __forceinline__ void stage_tile_start(const GemmArgs& a, int32_t* ts) {
  for (int i = threadIdx.x; i <= a.E; i += blockDim.x) ts[i] = __ldg(a.tile_start + i);
}

// Item w -> expert, weight-tile group m (tiles NT*m .. NT*m+NT-1), token tile.
// `tsm` is the shared-memory copy of tile_start.
__device__ __forceinline__ void decode_work(const GemmArgs& a, const int32_t* tsm, int BN, int NT, int w, Work& wk) {
  const int MG = a.MT / NT;  // weight-tile groups per expert
  int lo = 0, hi = a.E;      // largest e with MG*tile_start[e] <= w
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (MG * tsm[mid] <= w) lo = mid; else hi = mid;
  }
  const int ts = tsm[lo];
  const int nt = tsm[lo + 1] - ts;
  const int local = w - MG * ts;
  const int t = local % nt;
  wk.e = lo;
  wk.m = local / nt;
  wk.tile = ts + t;
  wk.r0 = __ldg(a.seg_start + lo) + t * BN;
  const int left = __ldg(a.counts + lo) - t * BN;
  wk.n = left < BN ? left : BN;
}

__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// e^(-y) for y >= 0, accurate to a few ulp over the whole range.  The fast
// form 2^(-fl(y log2 e)) loses accuracy as y grows: the product's rounding is
// up to |y log2 e| 2^-24 in absolute terms, which becomes the result's
// relative error.  Here y log2 e is carried as t + tl (tl: the product's
// rounding residual from an fma plus y times the tail of log2 e), 2^(-t) is
// taken on the hardware's base-2 exponential and multiplied by
// 2^(-tl) = 1 - tl ln 2 (|tl| <= 2^-23 |t|).  y is clamped to 128 (e^-128 is
// below the smallest subnormal; results below 2^-126 flush to zero), so
// +Inf gives 0 (and so does NaN).
__device__ __forceinline__ float exp_neg(float y) {
  constexpr float kLog2e = 1.44269502162933349609375f;  // fp32(log2 e)
  constexpr float kLog2eLo = 1.925963033500011e-08f;   // fp32(log2 e - kLog2e)
  constexpr float kLn2 = 0.693147182464599609375f;     // fp32(ln 2)
  y = fminf(y, 128.0f);
  const float t = y * kLog2e;
  const float tl = fmaf(y, kLog2eLo, fmaf(y, kLog2e, -t));
  const float p = ex2_approx(-t);
  return fmaf(p, -tl * kLn2, p);
}

// 1 - exp(-x) for x >= 0 given q = exp(-x): a Taylor polynomial below 1/4
// (no cancellation; the first omitted term, x^7/8!, is below 2e-9 relative),
// 1 - q above.
__device__ __forceinline__ float one_minus_exp_neg(float x, float q) {
  float p = 1.0f / 5040.0f;
  p = fmaf(p, x, -1.0f / 720.0f);
  p = fmaf(p, x, 1.0f / 120.0f);
  p = fmaf(p, x, -1.0f / 24.0f);
  p = fmaf(p, x, 1.0f / 6.0f);
  p = fmaf(p, x, -0.5f);
  p = fmaf(p, x, 1.0f);
  return x < 0.25f ? x * p : 1.0f - q;
}

// SiTU(g, u) = beta*tanh(g/beta)*sigmoid(g) * beta_lin*tanh(u/beta_lin) in fp32
// from exponentials of non-positive arguments only:
//   tanh(|v|/b) = (1 - q)/(1 + q),  q = exp(-2|v|/b)
//   sigmoid(g) = 1/(1 + r) (g >= 0) or r/(1 + r) (g < 0),  r = exp(-|g|)
// so the product is one quotient: no cancellation, no overflow, a few ulp.
// The sigmoid of a large negative g is r itself, so r's relative error is
// the result's: r comes from the accurate exp_neg, and for beta = 4
// (kg = 1/2, the method's value) as qg^2 with qg = exp_neg(|g|/2) exact in
// its argument, which saves an exponential.  qu's error only moves
// tanh(|u|/b) by about qu times it (fast exponential).
// kg = 2/beta, ku = 2/beta_lin, bb = beta*beta_lin.
__device__ __forceinline__ float situ_f32(float g, float u, float kg, float ku, float bb) {
  const float ag = fabsf(g), au = fabsf(u);
  const float xg = ag * kg, xu = au * ku;
  const float qg = exp_neg(xg);
  const float qu = __expf(-xu);
  const float omg = one_minus_exp_neg(xg, qg);
  const float omu = one_minus_exp_neg(xu, qu);
  float r;
  if (kg == 0.5f)
    r = qg * qg;
  else
    r = exp_neg(ag);
  const float num = (omg * omu) * (g >= 0.0f ? 1.0f : r);
  const float den = ((1.0f + qg) * (1.0f + qu)) * (1.0f + r);
  const float mag = bb * __fdividef(num, den);
  return ((g < 0.0f) != (u < 0.0f)) ? -mag : mag;
}

// The clamped SwiGLU control: g' = min(g, limit), u' = clamp(u, -limit,
// limit), out = g' * sigmoid(alpha*g') * (u' + beta), the sigmoid from the
// exponential of a non-positive argument (1/(1+e) or e/(1+e), e = exp(-|z|)).
// alpha*g' = z + zl exactly (zl from an fma); the sigmoid's relative error
// grows like |z| times the error of z, so e is corrected by the factor
// exp(-sign(z) zl) = 1 - sign(z) zl (|zl| <= 2^-24 |z|).
__device__ __forceinline__ float swiglu_f32(float g, float u, float alpha, float beta, float limit) {
  const float gc = fminf(g, limit);
  const float uc = fminf(fmaxf(u, -limit), limit);
  const float z = alpha * gc;
  const float zl = fmaf(alpha, gc, -z);
  float e = exp_neg(fabsf(z));
  e = fmaf(e, z >= 0.0f ? -zl : zl, e);
  const float sig = __fdividef(z >= 0.0f ? 1.0f : e, 1.0f + e);
  return gc * sig * (uc + beta);
}

// Epilogue staging tile: 128 rows x 32 floats, unpadded.  The 16-byte unit u
// of row r is stored at unit u ^ (r & 7) ^ ((r >> 3) & 7).  Row-wise float4
// writes: any 8 consecutive lanes (rows) hit 8 distinct units.  Column reads
// of the activation step: a warp reads, for one value index i, rows
// UV*uu + i (and 64 + that) of 8 or 4 columns; the lane bits that select uu
// (rows bits 3-5) and the column's unit reach the three unit bits through
// the (r >> 3) term, and the column within the unit picks the bank inside
// it, so the 32 lanes hit 32 distinct banks for both 8- and 16-value units.
constexpr int kStgFloats = 128 * 32;
__device__ __forceinline__ int stg_unit(int r, int u) { return r * 32 + ((u ^ (r & 7) ^ ((r >> 3) & 7)) << 2); }
__device__ __forceinline__ int stg_at(int r, int c) { return stg_unit(r, c >> 2) + (c & 3); }

// One 32-column chunk (token columns c0..c0+31) of the 128 x BN accumulator
// of weight tile mt, read from TMEM at `tacc` (the accumulator's first column,
// lane quarter included).  Called by the four warps of one epilogue group
// (warp eq of the group reads lane quarter q).
//   FC2: fp32 stores of rows 128*mt + lane to y of each column's routed slot.
//   FC1: the group stages the chunk in smem (`stg`, 128 x 32 floats), then
//        each math thread takes UV (8 or 16) consecutive intermediate columns
//        of a token:
//        the activation (SiTU, or the SwiGLU control when a.act is set) of
//        (gate, up) = (tile rows i, 64 + i), the MXFP8 scale of the 32-group
//        (amax over 32/UV threads), E4M3 codes as one 8- or 16-byte store.
template <bool FC1, int NCH, int UV = 16>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs& a, const Work& wk, int mt, uint32_t tacc, int c0,
                                               float* stg, int q, int eq, int lane, int grp, int skip_eq = -1,
                                               int heavy_eq = -1) {
  uint32_t r[32];
  tmem_ld_32x32b_x32(tacc + c0, r);
  tmem_ld_wait();
  if (!FC1) {
    const int h = 128 * mt + 32 * q + lane;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const int col = c0 + jj;
      if (col < wk.n) {
        const int slot = __ldg(a.slot_of_row + wk.r0 + col);
        a.y[static_cast<size_t>(slot) * a.H + h] = __uint_as_float(r[jj]);
      }
    }
    return;
  }
  {
    const int rr = 32 * q + lane;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<float4*>(stg + stg_unit(rr, u)) =
          make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]), __uint_as_float(r[4 * u + 2]),
                      __uint_as_float(r[4 * u + 3]));
  }
  named_barrier(2 + grp, 128);
  // 32*64/UV work units = (column, UV consecutive intermediate values of the
  // 64), spread over the group's warps except warp `skip_eq` (the one that
  // shares the MMA warp's scheduler); with three math warps, the warps of the
  // lowest ranks (warp `heavy_eq` first) take the extra pass.  The 32/UV units
  // of a quantisation group sit on consecutive lanes of one warp in the same
  // pass.  UV = 8 spreads the work more evenly over the three math warps (the
  // busiest thread evaluates 24 values instead of 32): it pays where the main
  // loop is short.
  constexpr int kUnits = 32 * 64 / UV;
  constexpr int kPer = 64 / UV;  // units per column
  constexpr int kQ = 32 / UV;    // units per quantisation group
  if (eq != skip_eq) {
    int wm = eq;  // rank among the math warps (0 takes the extra pass)
    if (skip_eq >= 0) {
      const int r = eq > skip_eq ? eq - 1 : eq;             // 0..2
      const int h = heavy_eq > skip_eq ? heavy_eq - 1 : heavy_eq;
      wm = r == h ? 0 : (r < h ? r + 1 : r);
    }
    const int stride = skip_eq >= 0 ? 96 : 128;
    for (int t = wm * 32 + lane; t < kUnits; t += stride) {
      const int cl = t / kPer;
      const int uu = t % kPer;
      const int col = c0 + cl;
      const int i0 = UV * uu;
      float act[UV];
      float amax = 0.0f;
      if (a.act == 0) {
#pragma unroll
        for (int i = 0; i < UV; ++i) {
          const float g = stg[stg_at(i0 + i, cl)];
          const float u = stg[stg_at(64 + i0 + i, cl)];
          act[i] = situ_f32(g, u, a.kg, a.ku, a.bb);
          amax = fmaxf(amax, fabsf(act[i]));
        }
      } else {
#pragma unroll
        for (int i = 0; i < UV; ++i) {
          const float g = stg[stg_at(i0 + i, cl)];
          const float u = stg[stg_at(64 + i0 + i, cl)];
          act[i] = swiglu_f32(g, u, a.sw_alpha, a.sw_beta, a.sw_limit);
          amax = fmaxf(amax, fabsf(act[i]));
        }
      }
#pragma unroll
      for (int m = 1; m < kQ; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
      const int e = e4m3_scale_exp(amax);
      const float inv = exp2i(-e);
      uint32_t w[UV / 4];
#pragma unroll
      for (int k4 = 0; k4 < UV / 4; ++k4) {
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(act[4 * k4] * inv, act[4 * k4 + 1] * inv),
                                                     __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(act[4 * k4 + 2] * inv, act[4 * k4 + 3] * inv),
                                                     __NV_SATFINITE, __NV_E4M3);
        w[k4] = (lo & 0xFFFFu) | (hi << 16);
        // a NaN activation (from an accumulator that overflowed to +Inf and
        // -Inf, possible only for inputs near the bf16 maximum) becomes +0,
        // the MXFP8 rule for NaN elements: the E4M3 NaN codes 0x7F / 0xFF
        w[k4] &= ~__vcmpeq4(w[k4] & 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      }
      if (col < wk.n) {
        uint8_t* dst = a.iq + static_cast<size_t>(wk.r0 + col) * a.I + 64 * mt + i0;
        if constexpr (UV == 16)
          *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        else
          *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
        if (uu % kQ == 0)
          a.isf[tile_sf_offset(wk.tile, col, 2 * mt + uu / kQ, NCH, a.I / 128)] = static_cast<uint8_t>(e + 127);
      }
    }
  }
  named_barrier(2 + grp, 128);
}

}  // namespace kmoe
