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
// Weights are read from the load-time layout of kmoe_prepare_weights: per
// (expert, 128-row weight tile, 128-wide K block) one contiguous block of
// 8192 code bytes (128 rows x 64 B) followed by its 512 scale bytes, blocks
// ordered by K block.  A work item therefore streams one contiguous range.
//
// Warp roles (persistent; one CTA per SM for the 224-row tiles, two for the
// 32- and 64-row tiles):
//   warp 0      TMA producer of the weight codes and scales
//   warp 1      TMEM owner and MMA issuer
//   warps 2..   epilogue, EPI_WARPS in groups of four; warp w reads TMEM lane
//               quarter w % 4, group g = (w - 2) / 4 takes the 32-column
//               chunks NGRP*i + g of the tile
//   last warp   TMA producer of the token rows and their scales
// The producer and MMA warps run their loops with all lanes converged; one
// lane, elected inside each instruction sequence, issues every copy and
// tcgen05 operation (a lone lane in a divergent branch issues them several
// times more slowly).  Two producer warps keep more bulk copies in flight
// than one thread can.
// Pipelines: STAGES smem stages (full/empty mbarriers) and NACC TMEM
// accumulator sets (acc_full/acc_empty); with two, the epilogue of one work
// item overlaps the main loop of the next.  Every wait is bounded.
//
// Work items: for expert e with nt_e = ceil(rows_e / BN) token tiles and MT
// weight tiles taken NT at a time (NT = 2 for the 224-row prefill tiles: two
// 128-row weight tiles share each token-tile load, cutting the bytes moved per
// MMA by 39%; one accumulator set then, as two do not fit in TMEM), items
// (MT/NT)*tile_start[e] .. are ordered weight-tile-major, so the token tiles
// sharing weight tiles run side by side (their weight reads meet in L2).
// CTA b takes items b, b+grid, ...
#include "gemm_dev.cuh"

namespace kmoe {

// Weight stages fetched into L2 ahead of their TMA loads by the small-tile
// (decode) kernels, which are bound by HBM: the shared-memory ring alone keeps
// too few weight bytes in flight per SM to cover the memory latency.
#ifndef KMOE_DECODE_PF_STAGES
#define KMOE_DECODE_PF_STAGES 2
#endif

template <int BN_, int KPS_, int STAGES_, bool FC1_, int EPI_WARPS_ = 8, int CTAS_PER_SM_ = 1, int NT_ = 1,
          int PF_ = 0>
struct GemmCfg {
  static constexpr int BN = BN_;
  static constexpr int PF = PF_;          // stages of weights prefetched into L2 ahead of the loads (0: none)
  static constexpr int KPS = KPS_;        // 128-wide K blocks per pipeline stage
  static constexpr int STAGES = STAGES_;
  static constexpr bool FC1 = FC1_;
  static constexpr int CTAS_PER_SM = CTAS_PER_SM_;
  static constexpr int NT = NT_;          // 128-row weight tiles per work item (sharing the token tile)
  static constexpr int NACC = NT == 1 ? 2 : 1;  // TMEM accumulator sets (2: epilogue overlaps next item)
  static constexpr int A_KB = 16384;     // 128 rows x 128 FP4 in the unpacked smem format
  static constexpr int A_TX_KB = 8192;   // transaction bytes of that tile (packed source)
  static constexpr int B_KB = BN * 128;  // token rows x 128 E4M3
  static constexpr int NCH = (BN + 127) / 128;
  static constexpr int B_OFF = NT * KPS * A_KB;  // A: [tile][kbi][16 KB]
  static constexpr int SFA_OFF = B_OFF + KPS * B_KB;
  static constexpr int SFB_OFF = SFA_OFF + NT * KPS * 512;
  static constexpr int STAGE = (SFB_OFF + KPS * NCH * 512 + 1023) / 1024 * 1024;
  static constexpr int SFW = 4 * NT + 4 * NCH;  // TMEM scale columns per K block (A tiles, then B chunks)
  static_assert(KPS * SFW <= 16, "scale columns per stage");
  static constexpr int EPI_WARPS = EPI_WARPS_;  // a multiple of 4 (one warp per TMEM lane quarter)
  static constexpr int NGRP = EPI_WARPS / 4;      // epilogue groups (column-chunk interleave)
  static constexpr int PRODB_WARP = 2 + EPI_WARPS;  // second producer: token rows and their scales
  static constexpr int THREADS = 32 * (3 + EPI_WARPS);
  static constexpr int STG_FLOATS = kStgFloats;  // one 128 x 32 staging tile per group
  static constexpr int STG_BYTES = FC1 ? NGRP * STG_FLOATS * 4 : 0;
  static constexpr int BAR_OFF = STAGES * STAGE + STG_BYTES;
  static constexpr int TS_OFF = BAR_OFF + 256;  // shared copy of tile_start
  static constexpr int SMEM = 1024 + TS_OFF + kTileStartBytes;
  static constexpr int SF_COL0 = NACC * NT * BN;
  static constexpr int TMEM_NEED = SF_COL0 + STAGES * 16;
  static constexpr int TMEM_COLS =
      TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
  static_assert(BN % 32 == 0 && BN <= 256, "token tile must be a multiple of 32 rows, at most 256");
  static_assert(TMEM_NEED <= 512, "TMEM budget");
  static_assert(SMEM * CTAS_PER_SM <= 232448, "shared memory budget");
  static_assert(TMEM_COLS * CTAS_PER_SM <= 512, "TMEM budget per SM");
  static_assert(EPI_WARPS % 4 == 0, "epilogue warps cover the four lane quarters");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, C::CTAS_PER_SM) moe_gemm_kernel(const __grid_constant__ GemmMaps maps,
                                                                 const GemmArgs a) {
  chain_wait();
  if (__ldg(a.tile_start + a.E) == 0) return;  // no tiles of this launch's class: leave before any set-up
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* tsm = reinterpret_cast<int32_t*>(smem + C::TS_OFF);
  stage_tile_start(a, tsm);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 2);  // one arrival per producer warp
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::NACC; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], C::EPI_WARPS);
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
    prefetch_tmap(&maps.a);
    for (int i = 0; i < 4; ++i) prefetch_tmap(&maps.b[i]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = (a.MT / C::NT) * tsm[a.E];
  const uint64_t budget = a.budget_ns;

  if (warp == 0 || warp == C::PRODB_WARP) {
    // ------------------------------------------------------------ producers
    // warp 0: weight codes and scales; warp PRODB_WARP: token rows and their
    // scales.  Both arrive on the stage's full barrier with their own bytes.
    // The whole warp runs the loop converged and one elected lane issues each
    // copy and arrival (ptx.cuh, the _el forms).
    {
      const bool is_a = warp == 0;
      const uint64_t pol = is_a ? policy_evict_normal() : policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      // L2 prefetch cursor (weight producer, PF > 0): walks the same item and
      // K-block sequence as the loads, up to PF stages ahead of them
      int pw = blockIdx.x, pkb = 0;
      uint32_t pit = 0;
      Work pwk;
      if (C::PF > 0 && is_a && pw < total) decode_work(a, tsm, C::BN, C::NT, pw, pwk);
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        Work wk;
        decode_work(a, tsm, C::BN, C::NT, w, wk);
        const int ng = (wk.n + 31) >> 5;  // 32-row groups of the token tile
        const uint32_t tx = is_a ? C::NT * C::KPS * (C::A_TX_KB + 512) : C::KPS * (ng * 4096 + C::NCH * 512);
        const int blk0 = (wk.e * a.MT + C::NT * wk.m) * a.KB;  // first block of the item's first tile
        const uint8_t* bsf = a.bsf + static_cast<size_t>(wk.tile) * a.KB * C::NCH * 512;
        for (int kb = 0; kb < a.KB; kb += C::KPS, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (C::PF > 0 && is_a) {
            while (pw < total && pit <= it + C::PF) {
              const int pblk0 = (pwk.e * a.MT + C::NT * pwk.m) * a.KB + pkb;
#pragma unroll
              for (int j = 0; j < C::NT; ++j) {
                const size_t blk = static_cast<size_t>(pblk0 + j * a.KB);
                bulk_prefetch_l2_el(a.wq + blk * 8192, C::KPS * 8192);
                bulk_prefetch_l2_el(a.wsf + blk * 512, C::KPS * 512);
              }
              ++pit;
              pkb += C::KPS;
              if (pkb >= a.KB) {
                pkb = 0;
                pw += gridDim.x;
                if (pw < total) decode_work(a, tsm, C::BN, C::NT, pw, pwk);
              }
            }
          }
          if (!mbar_wait_warp(&empty[s], ph ^ 1u, budget, a.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::STAGE;
          mbar_arrive_expect_tx_el(&full[s], tx);
          if (is_a) {
#pragma unroll
            for (int j = 0; j < C::NT; ++j) {
              const int blk = blk0 + j * a.KB + kb;
              tma_load_3d_el(st + j * C::KPS * C::A_KB, &maps.a, &full[s], 0, 0, blk, pol);
              bulk_load_el(st + C::SFA_OFF + j * C::KPS * 512, a.wsf + static_cast<size_t>(blk) * 512, C::KPS * 512,
                        &full[s]);
            }
          } else {
#pragma unroll
            for (int kbi = 0; kbi < C::KPS; ++kbi) {
              uint8_t* sb = st + C::B_OFF + kbi * C::B_KB;
              const int x = (kb + kbi) * 128;
              if (ng == C::BN / 32) {
                tma_load_2d_el(sb, &maps.b[3], &full[s], x, wk.r0, pol);  // a whole tile in one box
              } else {
                int g = 0;  // the tile's token rows in boxes of 128, 64 and 32 rows
                for (int lv = 2; lv >= 0; --lv) {
                  const int rows_g = 1 << lv;
                  while (ng - g >= rows_g) {
                    tma_load_2d_el(sb + g * 4096, &maps.b[lv], &full[s], x, wk.r0 + 32 * g, pol);
                    g += rows_g;
                  }
                }
              }
            }
            bulk_load_el(st + C::SFB_OFF, bsf + static_cast<size_t>(kb) * C::NCH * 512, C::KPS * C::NCH * 512,
                      &full[s]);
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA can exit
        const uint32_t first = it > static_cast<uint32_t>(C::STAGES) ? it - C::STAGES : 0u;
        for (uint32_t i = first; i < it; ++i)
          mbar_wait_warp(&full[i % C::STAGES], (i / C::STAGES) & 1u, 20000000ull, nullptr, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged and one elected lane issues each
    // tcgen05 operation (ptx.cuh, the _el forms); the loop stays lean:
    // descriptors are formed once and advanced by adds (the start-address
    // field holds smem offset >> 4).
    {
      constexpr uint32_t kStageD = C::STAGE >> 4;
      const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(smem));
      const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(smem + C::B_OFF));
      const uint64_t sfadesc0 = sdesc_sf_32x16(smem_u32(smem + C::SFA_OFF));
      const uint64_t sfbdesc0 = sdesc_sf_32x16(smem_u32(smem + C::SFB_OFF));
      int s = 0;
      uint32_t ph = 0, li = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x, ++li) {
        Work wk;
        decode_work(a, tsm, C::BN, C::NT, w, wk);
        const uint32_t acc = li % C::NACC;
        const uint32_t aph = (li / C::NACC) & 1u;
        if (!mbar_wait_warp(&acc_empty[acc], aph ^ 1u, budget, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * C::NT * C::BN;  // tile j accumulates at d + j*BN
        const uint32_t nmma = (static_cast<uint32_t>(wk.n) + 15u) & ~15u;
        const int nch = static_cast<int>((nmma + 127u) >> 7);
        const uint32_t id0 = idesc_mxf8f6f4(128, nmma, MX_E2M1, MX_E4M3, 0, 0);
        for (int kb = 0; kb < a.KB; kb += C::KPS) {
          if (!mbar_wait_warp(&full[s], ph, budget, a.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = static_cast<uint64_t>(s) * kStageD;
          const uint32_t sf0 = tmem + C::SF_COL0 + static_cast<uint32_t>(s) * 16;
#pragma unroll
          for (int kbi = 0; kbi < C::KPS; ++kbi) {
            const uint32_t sfc = sf0 + kbi * C::SFW;
            const uint32_t sfb = sfc + 4 * C::NT;
#pragma unroll
            for (int j = 0; j < C::NT; ++j)
              tc_cp_32x128b_warpx4_el(sfc + 4 * j, sfadesc0 + so + (j * C::KPS + kbi) * 32);
            tc_cp_32x128b_warpx4_el(sfb, sfbdesc0 + so + kbi * C::NCH * 32);
            if (C::NCH > 1 && nch > 1) tc_cp_32x128b_warpx4_el(sfb + 4, sfbdesc0 + so + kbi * C::NCH * 32 + 32);
            const uint64_t bd = bdesc0 + so + kbi * (C::B_KB >> 4);
#pragma unroll
            for (int j = 0; j < C::NT; ++j) {
              const uint64_t ad = adesc0 + so + (j * C::KPS + kbi) * (C::A_KB >> 4);
              mma_mxf8f6f4_el(d + j * C::BN, ad, bd, id0, sfc + 4 * j, sfb, (kb | kbi) != 0);
              mma_mxf8f6f4_el(d + j * C::BN, ad + 2, bd + 2, id0 | (1u << 4) | (1u << 29), sfc + 4 * j, sfb, 1u);
              mma_mxf8f6f4_el(d + j * C::BN, ad + 4, bd + 4, id0 | (2u << 4) | (2u << 29), sfc + 4 * j, sfb, 1u);
              mma_mxf8f6f4_el(d + j * C::BN, ad + 6, bd + 6, id0 | (3u << 4) | (3u << 29), sfc + 4 * j, sfb, 1u);
            }
          }
          tc_commit_el(&empty[s]);
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_el(&acc_full[acc]);
      }
      tc_commit_el(done);
      mbar_wait_warp(done, 0, budget, a.err, nullptr);
    }
  } else if (warp < C::PRODB_WARP) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;   // TMEM lane quarter of this warp
    const int ew = warp - 2;  // 0..EPI_WARPS-1
    const int grp = ew >> 2;  // chunk group
    const int eq = ew & 3;    // warp within the group
    float* stg = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE) + grp * C::STG_FLOATS;
    uint32_t li = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x, ++li) {
      Work wk;
      decode_work(a, tsm, C::BN, C::NT, w, wk);
      const uint32_t acc = li % C::NACC;
      const uint32_t aph = (li / C::NACC) & 1u;
      bool ok = mbar_wait_bounded(&acc_full[acc], aph, budget, a.err, abort_flag);
      ok = named_barrier_and(1, 32 * C::EPI_WARPS, ok && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      // chunks of 32 columns of the NT accumulators, round-robin over the groups
      const int nchunk = (wk.n + 31) >> 5;
      for (int ci = grp; ci < C::NT * nchunk; ci += C::NGRP) {
        const int j = ci / nchunk;             // weight tile of the item
        const int c0 = (ci - j * nchunk) * 32;  // first column of the chunk
        const int mt = C::NT * wk.m + j;        // weight tile index within the expert
        const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + (acc * C::NT + j) * C::BN;
        epilogue_chunk<C::FC1, C::NCH>(a, wk, mt, tbase, c0, stg, q, eq, lane, grp);
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

// ---------------------------------------------------------------- weight re-layout
// Block (e, m, kb) of the prepared weights = 128 tile rows x 64 code bytes
// (K elements 128kb..128kb+127 of each row) at blk*8192 in the code region,
// and 512 scale bytes at nblk*8192 + blk*512 in the scale region, byte
// j*16 + c*4 + g holding tile row 32c+j for K group 4kb+g.  FC1 tile m holds
// gate rows 64m..64m+63 then up rows I+64m..I+64m+63; FC2 tile m holds rows
// 128m..128m+127.  Blocks are ordered (e, m, kb).
__device__ __forceinline__ int tile_row_src(int fc1, int m, int tr, int I) {
  if (fc1) return tr < 64 ? 64 * m + tr : I + 64 * m + (tr - 64);
  return 128 * m + tr;
}

__global__ void prep_weights_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ sf,
                                    uint8_t* __restrict__ out, int E, int MT, int KB, int rows_per_expert, int K,
                                    int fc1, int I) {
  // one thread per 16 bytes of a block (8192 code bytes = 512 x 16, scales = 32 x 16)
  constexpr int kPieces = kWeightBlockBytes / 16;
  const size_t nblk = static_cast<size_t>(E) * MT * KB;
  const size_t total = nblk * kPieces;
  const size_t row_bytes = static_cast<size_t>(K) / 2;
  const int gpr = K / 32;
  for (size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t blk = idx / kPieces;
    const int piece = static_cast<int>(idx % kPieces);
    const int kb = static_cast<int>(blk % KB);
    const int m = static_cast<int>((blk / KB) % MT);
    const int e = static_cast<int>(blk / (static_cast<size_t>(KB) * MT));
    if (piece < 512) {
      uint8_t* dst = out + blk * 8192 + static_cast<size_t>(piece) * 16;
      const int tr = piece >> 2;
      const int src_row = tile_row_src(fc1, m, tr, I);
      const uint8_t* src =
          codes + (static_cast<size_t>(e) * rows_per_expert + src_row) * row_bytes + kb * 64 + (piece & 3) * 16;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    } else {
      const int j = piece - 512;  // lane j: rows j, 32+j, 64+j, 96+j
      uint8_t* dst = out + nblk * 8192 + blk * 512 + static_cast<size_t>(j) * 16;
      uint32_t v[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int src_row = tile_row_src(fc1, m, 32 * c + j, I);
        const uint8_t* s = sf + (static_cast<size_t>(e) * rows_per_expert + src_row) * gpr + 4 * kb;
        v[c] = static_cast<uint32_t>(s[0]) | (static_cast<uint32_t>(s[1]) << 8) |
               (static_cast<uint32_t>(s[2]) << 16) | (static_cast<uint32_t>(s[3]) << 24);
      }
      *reinterpret_cast<uint4*>(dst) = make_uint4(v[0], v[1], v[2], v[3]);
    }
  }
}

cudaError_t launch_prep_weights(const uint8_t* codes, const uint8_t* sf, uint8_t* out, int E, int MT, int KB,
                                int rows_per_expert, int K, int fc1, int I, cudaStream_t st) {
  prep_weights_kernel<<<2048, 256, 0, st>>>(codes, sf, out, E, MT, KB, rows_per_expert, K, fc1, I);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- launch
template <class C>
static cudaError_t launch_one(const GemmMaps& maps, const GemmArgs& a, int grid, cudaStream_t st, bool pdl) {
  static bool attr_set[kMaxDevices] = {};  // per instantiation and device; benign race (idempotent)
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  return launch_chained(moe_gemm_kernel<C>, dim3(grid * C::CTAS_PER_SM), dim3(C::THREADS), C::SMEM, st, pdl, maps, a);
}

cudaError_t launch_moe_gemm(bool fc1, int BN, int kps, const GemmMaps& maps, const GemmArgs& a, int grid,
                            cudaStream_t st, bool pdl) {
  if (a.KB % kps != 0) return cudaErrorInvalidValue;
  constexpr int PF = KMOE_DECODE_PF_STAGES;
  if (fc1) {
    if (BN == 32) return kps == 2 ? launch_one<GemmCfg<32, 2, 2, true, 4, 2, 1, PF>>(maps, a, grid, st, pdl)
                                  : launch_one<GemmCfg<32, 1, 8, true, 8, 1, 1, 2 * PF>>(maps, a, grid, st, pdl);
    if (BN == 64 && kps == 1) return launch_one<GemmCfg<64, 1, 3, true, 4, 2, 1, 2 * PF>>(maps, a, grid, st, pdl);
    if (BN == 224 && kps == 1)
      return pair_gemm_supported(a.MT, a.KB) ? launch_moe_gemm_pair(true, maps, a, grid, st, pdl)
                           : launch_one<GemmCfg<224, 1, 4, true>>(maps, a, grid, st, pdl);
  } else {
    if (BN == 32) return kps == 2 ? launch_one<GemmCfg<32, 2, 2, false, 4, 2, 1, PF>>(maps, a, grid, st, pdl)
                                  : launch_one<GemmCfg<32, 1, 8, false, 8, 1, 1, 2 * PF>>(maps, a, grid, st, pdl);
    if (BN == 64 && kps == 1) return launch_one<GemmCfg<64, 1, 4, false, 4, 2, 1, 2 * PF>>(maps, a, grid, st, pdl);
    if (BN == 224 && kps == 1)
      return pair_gemm_supported(a.MT, a.KB) ? launch_moe_gemm_pair(false, maps, a, grid, st, pdl)
                           : launch_one<GemmCfg<224, 1, 4, false>>(maps, a, grid, st, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kmoe
