// Microscaling quantisation of bf16 activations (MoE path analysis page,
// SM100 pre-dispatch: per-32 absmax -> UE8M0 scale -> FP8 E4M3 codes; the
// SM120 page's NaN/Inf record: saturating-finite codes, never the 0xFF
// scale).  One thread per 32-element group: four 16-byte loads, an absmax,
// the exact power-of-two scale, and the hardware's round-to-nearest-even
// saturating conversion.
//
//   quant_rows_kernel     token-major output (kmoe_quantize_mx), E4M3 or E2M1
//   quant_scatter_kernel  forward path: codes of token t written to each of
//                         its k expert-sorted rows, scales in the token-tile
//                         layout the GEMM copies into TMEM
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace kmoe {

__device__ __forceinline__ void load_group_bf16(const __nv_bfloat16* p, float (&v)[32]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = __ldg(q + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ float group_amax(const float (&v)[32]) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[i]));  // fmaxf drops NaN
  return a;
}

__device__ __forceinline__ uint8_t e4m3_code(float x, float inv_scale) {
  if (isnan(x)) return 0;
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x * inv_scale, __NV_SATFINITE, __NV_E4M3));
}

// 32 E4M3 codes of a group, packed little-endian into 8 words
__device__ __forceinline__ void e4m3_group(const float (&v)[32], float inv_scale, uint32_t (&out)[8]) {
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) word |= static_cast<uint32_t>(e4m3_code(v[4 * w + b], inv_scale)) << (8 * b);
    out[w] = word;
  }
}

__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16* __restrict__ x, int rows, int cols,
                                                         int fmt, uint8_t* __restrict__ codes,
                                                         uint8_t* __restrict__ scales) {
  const int gpr = cols / 32;
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= static_cast<long long>(rows) * gpr) return;
  const long long r = gid / gpr;
  const int g = static_cast<int>(gid % gpr);
  float v[32];
  load_group_bf16(x + r * cols + 32 * g, v);
  const float amax = group_amax(v);
  if (fmt == KMOE_MXFP8_E4M3) {
    const int e = e4m3_scale_exp(amax);
    uint32_t out[8];
    e4m3_group(v, exp2i(-e), out);
    uint4* dst = reinterpret_cast<uint4*>(codes + r * cols + 32 * g);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    scales[r * gpr + g] = static_cast<uint8_t>(e + 127);
  } else {
    const int e = e2m1_scale_exp(amax);
    const float inv = exp2i(-e);
    uint32_t out[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const float xv = v[8 * w + b];
        const uint32_t c =
            isnan(xv) ? 0u : static_cast<uint32_t>(__nv_cvt_float_to_fp4(xv * inv, __NV_E2M1, cudaRoundNearest));
        word |= (c & 0xFu) << (4 * b);
      }
      out[w] = word;
    }
    uint4* dst = reinterpret_cast<uint4*>(codes + r * (cols / 2) + 16 * g);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    scales[r * gpr + g] = static_cast<uint8_t>(e + 127);
  }
}

cudaError_t launch_quant_rows(const void* x, int rows, int cols, int fmt, uint8_t* codes, uint8_t* scales,
                              cudaStream_t st) {
  const long long groups = static_cast<long long>(rows) * (cols / 32);
  if (groups == 0) return cudaSuccess;
  const long long blocks = (groups + 255) / 256;
  quant_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), rows,
                                                                   cols, fmt, codes, scales);
  return cudaGetLastError();
}

// One block per token.  Threads 0..k-1 first resolve the token's k slots to
// expert-sorted rows and token tiles (of the expert's tile class: BN rows for
// experts with at most `thr` rows, kBigTileRows rows and the xsf_big scale
// array for the others); then each thread quantises one
// 32-element group.  A warp's 32 groups form one contiguous 1 KB run of code
// bytes per routed slot: the lanes exchange their codes once (shuffles) so
// that each store instruction writes 512 contiguous bytes (lane l: 16-byte
// chunk l, then chunk 32 + l), and the run is stored once per slot.  The
// four groups of a 128-wide K block sit in an aligned quad of lanes and their
// scale bytes are adjacent in the token-tile scale layout, so the quad merges
// them and its first lane writes one 32-bit word per slot.
__global__ void __launch_bounds__(256) quant_scatter_kernel(
    const __nv_bfloat16* __restrict__ x, int H, int k, int E, int BN, int thr, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ rank, const int32_t* __restrict__ chunk_prefix, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ seg_start, const int32_t* __restrict__ tile_start,
    const int32_t* __restrict__ tile_start_big, int32_t* __restrict__ row_of_slot, int32_t* __restrict__ slot_of_row,
    uint8_t* __restrict__ xq, uint8_t* __restrict__ xsf, uint8_t* __restrict__ xsf_big) {
  chain_wait();
  __shared__ int s_row[kMaxK], s_tile[kMaxK], s_local[kMaxK], s_big[kMaxK];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    const int j = threadIdx.x;
    const int s = t * k + j;
    const int id = ids[s];
    int row = -1, tile = -1, local = -1, big = 0;
    if (id >= 0 && id < E) {
      const int c = s / kRankChunk;
      const int in_seg = chunk_prefix[static_cast<size_t>(c) * E + id] + rank[s];
      row = seg_start[id] + in_seg;
      big = counts[id] > thr;
      const int bn = big ? kBigTileRows : BN;
      tile = (big ? tile_start_big[id] : tile_start[id]) + in_seg / bn;
      local = in_seg % bn;
      slot_of_row[row] = s;
    }
    row_of_slot[s] = row;
    s_row[j] = row;
    s_tile[j] = tile;
    s_local[j] = local;
    s_big[j] = big;
  }
  __syncthreads();
  const int lane = static_cast<int>(threadIdx.x) & 31;
  const int gpr = H / 32;  // a multiple of 4: quads are wholly in or out of range
  const int KB = H / 128;
  for (int g0 = 0; g0 < gpr; g0 += blockDim.x) {
    const int g = g0 + static_cast<int>(threadIdx.x);
    const int gw = g - lane;                     // first group of this warp's run
    if (gw >= gpr) continue;                     // the whole warp is past the row
    const int nact = min(32, gpr - gw);          // groups of the run (a multiple of 4)
    const bool active = lane < nact;
    uint32_t out[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int e = 0;
    if (active) {
      float v[32];
      load_group_bf16(x + static_cast<size_t>(t) * H + 32 * g, v);
      e = e4m3_scale_exp(group_amax(v));
      e4m3_group(v, exp2i(-e), out);
    }
    // chunk c of the run (16 bytes) = half (c & 1) of group c >> 1
    uint32_t c0[4], c1[4];
    const int src0 = lane >> 1, src1 = 16 + (lane >> 1);
    const bool hi = lane & 1;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t a0 = __shfl_sync(0xffffffffu, out[w], src0), a1 = __shfl_sync(0xffffffffu, out[4 + w], src0);
      const uint32_t b0 = __shfl_sync(0xffffffffu, out[w], src1), b1 = __shfl_sync(0xffffffffu, out[4 + w], src1);
      c0[w] = hi ? a1 : a0;
      c1[w] = hi ? b1 : b0;
    }
    const uint4 v0 = make_uint4(c0[0], c0[1], c0[2], c0[3]);
    const uint4 v1 = make_uint4(c1[0], c1[1], c1[2], c1[3]);
    const bool st0 = src0 < nact, st1 = src1 < nact;
    uint32_t sc = active ? static_cast<uint32_t>(e + 127) << (8 * (g & 3)) : 0u;
    sc |= __shfl_xor_sync(0xffffffffu, sc, 1);
    sc |= __shfl_xor_sync(0xffffffffu, sc, 2);
    for (int j = 0; j < k; ++j) {
      const int row = s_row[j];
      if (row < 0) continue;
      uint4* run = reinterpret_cast<uint4*>(xq + static_cast<size_t>(row) * H + 32 * gw);
      if (st0) run[lane] = v0;
      if (st1) run[32 + lane] = v1;
      if (active && (g & 3) == 0) {
        // small tiles (at most 64 rows) hold one 128-row scale chunk, big tiles two
        uint8_t* base = s_big[j] ? xsf_big : xsf;
        *reinterpret_cast<uint32_t*>(base + tile_sf_offset(s_tile[j], s_local[j], g, s_big[j] ? 2 : 1, KB)) = sc;
      }
    }
  }
}

cudaError_t launch_quant_scatter(const void* x, int T, int H, int k, int E, int BN, int thr, const int32_t* ids,
                                 const int32_t* rank, const int32_t* chunk_prefix, const int32_t* counts,
                                 const int32_t* seg_start, const int32_t* tile_start, const int32_t* tile_start_big,
                                 int32_t* row_of_slot, int32_t* slot_of_row, uint8_t* xq, uint8_t* xsf,
                                 uint8_t* xsf_big, cudaStream_t st, bool pdl) {
  if (T == 0) return cudaSuccess;
  return launch_chained(quant_scatter_kernel, dim3(T), dim3(256), 0, st, pdl, static_cast<const __nv_bfloat16*>(x),
                        H, k, E, BN, thr, ids, rank, chunk_prefix, counts, seg_start, tile_start, tile_start_big,
                        row_of_slot, slot_of_row, xq, xsf, xsf_big);
}

}  // namespace kmoe
