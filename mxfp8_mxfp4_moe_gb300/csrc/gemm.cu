// Grouped block-scaled expert GEMMs on the 5th-generation tensor cores.
//
//   FC1: per expert e and token tile, D = W13_tile (128 weight rows: 64 gate
//        rows and the matching 64 up rows) x X_tile^T over K = H, followed by
//        SiTU(gate, up) and MXFP8 requantisation of the result (epilogue).
//   FC2: D = W2_tile (128 rows of H) x INTER_tile^T over K = I, stored as
//        fp32 per routed slot.
//
// Both use tcgen05.mma .kind::mxf8f6f4 with block scaling (scale_vec::1X):
// A = E2M1 weights (TMA in the 16-byte-aligned unpacked FP4 smem format,
// 128-byte swizzle), B = E4M3 token rows (TMA, 128-byte swizzle), UE8M0
// scales copied into TMEM by tcgen05.cp (32x128b, replicated into the four
// lane quarters), fp32 accumulators in TMEM.  Weights sit in the M=128 slot
// so a tile holds as few as 16 routed rows (decode) and up to BN (prefill).
//
// Warp roles (192 threads, persistent, one CTA per SM):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM owner and MMA issuer (one lane)
//   warps 2..5  epilogue; warp w reads TMEM lane quarter w % 4
// Pipelines: STAGES smem stages (full/empty mbarriers) and two TMEM
// accumulator buffers (acc_full/acc_empty) so the epilogue of one work item
// overlaps the main loop of the next.  Every wait is bounded.
//
// Work items: for expert e with nt_e = ceil(rows_e / BN) token tiles and MT
// weight tiles, items MT*tile_start[e] .. MT*tile_start[e+1]-1 are ordered
// weight-tile-major, so the token tiles sharing one weight tile run side by
// side (their weight reads meet in L2).  CTA b takes items b, b+grid, ...
#include <cuda_fp8.h>

#include "gemm.cuh"

namespace kmoe {



template <int BN_, int STAGES_, bool FC1_>
struct GemmCfg {
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static constexpr bool FC1 = FC1_;
  static constexpr int A_BYTES = 16384;  // 128 rows x 128 FP4 in the unpacked smem format
  static constexpr int A_TX = 8192;      // transaction bytes of that tile (packed source)
  static constexpr int B_BYTES = BN * 128;
  static constexpr int NCH = (BN + 127) / 128;
  static constexpr int SF_OFF = A_BYTES + B_BYTES;
  static constexpr int STAGE = (A_BYTES + B_BYTES + 512 + NCH * 512 + 1023) / 1024 * 1024;
  static constexpr int STG_BYTES = FC1 ? 128 * 33 * 4 : 0;
  static constexpr int BAR_OFF = STAGES * STAGE + STG_BYTES;
  static constexpr int SMEM = 1024 + BAR_OFF + 256;
  static constexpr int SF_COL0 = 2 * BN;
  static constexpr int TMEM_NEED = 2 * BN + STAGES * 16;
  static constexpr int TMEM_COLS =
      TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
  static_assert(BN % 32 == 0 && BN <= 256, "token tile must be a multiple of 32 rows, at most 256");
  static_assert(TMEM_NEED <= 512, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct Work {
  int e, m, tile, r0, n;
};

__device__ __forceinline__ void decode_work(const GemmArgs& a, int BN, int w, Work& wk) {
  int lo = 0, hi = a.E;  // largest e with MT*tile_start[e] <= w
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.MT * __ldg(a.tile_start + mid) <= w) lo = mid; else hi = mid;
  }
  const int ts = __ldg(a.tile_start + lo);
  const int nt = __ldg(a.tile_start + lo + 1) - ts;
  const int local = w - a.MT * ts;
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

__device__ __forceinline__ float situ_f32(float g, float u, float beta, float beta_lin) {
  const float gate = beta * tanhf(g / beta) * (1.0f / (1.0f + expf(-g)));
  const float up = beta_lin * tanhf(u / beta_lin);
  return gate * up;
}

template <class C>
__global__ void __launch_bounds__(192, 1) moe_gemm_kernel(const __grid_constant__ CUtensorMap mapA,
                                                          const __grid_constant__ CUtensorMap mapB,
                                                          const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* stg = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&mapA);
    prefetch_tmap(&mapB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = a.MT * __ldg(a.tile_start + a.E);
  const uint64_t budget = a.budget_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        Work wk;
        decode_work(a, C::BN, w, wk);
        const int ng = (wk.n + 31) >> 5;
        const int nch = (wk.n + 127) >> 7;
        const uint32_t tx = C::A_TX + ng * 4096 + 512 + nch * 512;
        const uint8_t* wsf = a.wsf + (static_cast<size_t>(wk.e) * a.MT + wk.m) * a.KB * 512;
        const uint8_t* bsf = a.bsf + static_cast<size_t>(wk.tile) * C::NCH * 512;
        const size_t bsf_kb = static_cast<size_t>(a.max_tiles) * C::NCH * 512;
        int rowA0, rowA1 = 0;
        if (C::FC1) {
          rowA0 = wk.e * 2 * a.I + 64 * wk.m;
          rowA1 = rowA0 + a.I;
        } else {
          rowA0 = wk.e * a.H + 128 * wk.m;
        }
        for (int kb = 0; kb < a.KB; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, budget, a.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::STAGE;
          mbar_arrive_expect_tx(&full[s], tx);
          if (C::FC1) {
            tma_load_2d(st, &mapA, &full[s], kb * 128, rowA0, pol_w);
            tma_load_2d(st + 8192, &mapA, &full[s], kb * 128, rowA1, pol_w);
          } else {
            tma_load_2d(st, &mapA, &full[s], kb * 128, rowA0, pol_w);
          }
          for (int b = 0; b < ng; ++b)
            tma_load_2d(st + C::A_BYTES + b * 4096, &mapB, &full[s], kb * 128, wk.r0 + 32 * b, pol_x);
          bulk_load(st + C::SF_OFF, wsf + static_cast<size_t>(kb) * 512, 512, &full[s]);
          bulk_load(st + C::SF_OFF + 512, bsf + kb * bsf_kb, nch * 512, &full[s]);
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA can exit
        const uint32_t first = it > static_cast<uint32_t>(C::STAGES) ? it - C::STAGES : 0u;
        for (uint32_t i = first; i < it; ++i)
          mbar_wait_bounded(&full[i % C::STAGES], (i / C::STAGES) & 1u, 20000000ull, nullptr, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, li = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x, ++li) {
        Work wk;
        decode_work(a, C::BN, w, wk);
        const uint32_t acc = li & 1u;
        const uint32_t aph = (li >> 1) & 1u;
        if (!mbar_wait_bounded(&acc_empty[acc], aph ^ 1u, budget, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * C::BN;
        const uint32_t nmma = (static_cast<uint32_t>(wk.n) + 15u) & ~15u;
        const int nch = (wk.n + 127) >> 7;
        for (int kb = 0; kb < a.KB; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait_bounded(&full[s], ph, budget, a.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t* st = smem + s * C::STAGE;
          const uint32_t sfc = tmem + C::SF_COL0 + s * 16;
          tc_cp_32x128b_warpx4(sfc, sdesc_sf_32x16(smem_u32(st + C::SF_OFF)));
          for (int c = 0; c < nch; ++c)
            tc_cp_32x128b_warpx4(sfc + 4 + 4 * c, sdesc_sf_32x16(smem_u32(st + C::SF_OFF + 512 + 512 * c)));
          const uint32_t aaddr = smem_u32(st);
          const uint32_t baddr = smem_u32(st + C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_mxf8f6f4(d, sdesc_kmajor_sw128(aaddr + 32 * kk), sdesc_kmajor_sw128(baddr + 32 * kk),
                         idesc_mxf8f6f4(128, nmma, MX_E2M1, MX_E4M3, kk, kk), sfc, sfc + 4, (kb | kk) != 0);
          }
          tc_commit(&empty[s]);
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
      }
      tc_commit(done);
      mbar_wait_bounded(done, 0, budget, a.err, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;   // TMEM lane quarter of this warp
    const int eq = warp - 2;  // 0..3
    uint32_t li = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x, ++li) {
      Work wk;
      decode_work(a, C::BN, w, wk);
      const uint32_t acc = li & 1u;
      const uint32_t aph = (li >> 1) & 1u;
      bool ok = mbar_wait_bounded(&acc_full[acc], aph, budget, a.err, abort_flag);
      ok = named_barrier_and(1, 128, ok && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * C::BN;
      for (int c0 = 0; c0 < wk.n; c0 += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tbase + c0, r);
        tmem_ld_wait();
        if (!C::FC1) {
          const int h = 128 * wk.m + 32 * q + lane;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int col = c0 + jj;
            if (col < wk.n) {
              const int slot = __ldg(a.slot_of_row + wk.r0 + col);
              a.y[static_cast<size_t>(slot) * a.H + h] = __uint_as_float(r[jj]);
            }
          }
        } else {
          float* row = stg + (32 * q + lane) * 33;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) row[jj] = __uint_as_float(r[jj]);
          named_barrier(2, 128);
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            const int cl = 8 * eq + cc;
            const int col = c0 + cl;
            if (col >= wk.n) break;
#pragma unroll
            for (int grp = 0; grp < 2; ++grp) {
              const float g = stg[(32 * grp + lane) * 33 + cl];
              const float u = stg[(64 + 32 * grp + lane) * 33 + cl];
              const float act = situ_f32(g, u, a.beta, a.beta_lin);
              float amax = fabsf(act);
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
              const int e = e4m3_scale_exp(amax);
              const uint8_t code = static_cast<uint8_t>(
                  __nv_cvt_float_to_fp8(act * exp2i(-e), __NV_SATFINITE, __NV_E4M3));
              a.iq[static_cast<size_t>(wk.r0 + col) * a.I + 64 * wk.m + 32 * grp + lane] = code;
              if (lane == 0)
                a.isf[tile_sf_offset(wk.tile, col, 2 * wk.m + grp, C::NCH, a.max_tiles)] =
                    static_cast<uint8_t>(e + 127);
            }
          }
          named_barrier(2, 128);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- weight scale re-layout
// out[((e*MT + m)*KB + kb)*512 + j*16 + c*4 + g] = scale of weight-tile row
// 32c+j for K group 4kb+g.  FC1 tile m holds gate rows 64m..64m+63 then up
// rows I+64m..I+64m+63; FC2 tile m holds rows 128m..128m+127.
__global__ void prep_wsf_kernel(const uint8_t* __restrict__ sf, uint8_t* __restrict__ out, int E, int MT, int KB,
                                int rows_per_expert, int gpr, int fc1, int I) {
  const size_t total = static_cast<size_t>(E) * MT * KB * 512;
  for (size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int byte = static_cast<int>(idx & 511);
    size_t rest = idx >> 9;
    const int kb = static_cast<int>(rest % KB);
    rest /= KB;
    const int m = static_cast<int>(rest % MT);
    const int e = static_cast<int>(rest / MT);
    const int j = byte >> 4, c = (byte >> 2) & 3, g = byte & 3;
    const int tr = 32 * c + j;
    int row;
    if (fc1) row = tr < 64 ? 64 * m + tr : I + 64 * m + (tr - 64);
    else row = 128 * m + tr;
    out[idx] = sf[(static_cast<size_t>(e) * rows_per_expert + row) * gpr + 4 * kb + g];
  }
}

cudaError_t launch_prep_wsf(const uint8_t* sf, uint8_t* out, int E, int MT, int KB, int rows_per_expert, int gpr,
                            int fc1, int I, cudaStream_t st) {
  prep_wsf_kernel<<<1024, 256, 0, st>>>(sf, out, E, MT, KB, rows_per_expert, gpr, fc1, I);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- launch
template <class C>
static cudaError_t launch_one(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmArgs& a, int grid,
                              cudaStream_t st) {
  static bool attr_set = false;  // per instantiation; benign race (idempotent)
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  moe_gemm_kernel<C><<<grid, 192, C::SMEM, st>>>(mapA, mapB, a);
  return cudaGetLastError();
}

cudaError_t launch_moe_gemm(bool fc1, int BN, const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmArgs& a,
                            int grid, cudaStream_t st) {
  if (fc1) {
    if (BN == 32) return launch_one<GemmCfg<32, 8, true>>(mapA, mapB, a, grid, st);
    if (BN == 64) return launch_one<GemmCfg<64, 7, true>>(mapA, mapB, a, grid, st);
    if (BN == 224) return launch_one<GemmCfg<224, 4, true>>(mapA, mapB, a, grid, st);
  } else {
    if (BN == 32) return launch_one<GemmCfg<32, 8, false>>(mapA, mapB, a, grid, st);
    if (BN == 64) return launch_one<GemmCfg<64, 7, false>>(mapA, mapB, a, grid, st);
    if (BN == 224) return launch_one<GemmCfg<224, 4, false>>(mapA, mapB, a, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kmoe
