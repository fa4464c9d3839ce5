// CTA-pair variant of the grouped expert GEMMs for the 224-row token tiles
// of prefill-sized layers.
//
// A cluster of two CTAs (two SMs) runs one work item = (expert e, weight
// tiles 2m and 2m+1, token tile of up to 224 rows) as 56 (FC1) or 28 (FC2)
// K blocks of tcgen05.mma.cta_group::2 with M = 256: CTA r supplies weight
// tile 2m+r (its 128 A rows) and half of the token rows, and its TMEM receives
// the 128 x 224 accumulator of its own weight tile.  Compared with one CTA
// computing both weight tiles, every SM loads half the token rows per K block
// and its shared memory serves the token operand once for both tensor cores,
// and each TMEM holds one 224-column accumulator, so two fit: the epilogue of
// one item overlaps the main loop of the next.
//
// Roles in each CTA of the pair:
//   warp 0      TMA of the CTA's weight block and its 512 scale bytes
//   warp 1      TMEM allocation (both CTAs); in the even CTA it issues the
//               pair MMAs (converged, one elected lane per instruction)
//   warps 2..9  epilogue on the CTA's own accumulator (as in the one-CTA kernel)
//   warp 10     TMA of the CTA's token rows (token tile rows [rN/2, rN/2+112))
//               and of the scales of all token rows of the tile
// Barriers: every load of both CTAs completes on full[s] of the even CTA (TMA
// .cta_group::2), whose two producers expect the bytes of both CTAs; the MMA
// commit multicasts empty[s] and acc_full[b] to both CTAs; acc_empty[b] of the
// even CTA counts the epilogue warps of both CTAs.  Every wait is bounded.
#include "gemm_dev.cuh"

namespace kmoe {

template <bool FC1_, int STAGES_, bool DYN_, int UV_ = 16>
struct PairCfg {
  static constexpr bool FC1 = FC1_;
  static constexpr int STAGES = STAGES_;
  static constexpr bool DYN = DYN_;  // work items claimed dynamically (else pair p takes p, p + npairs, ...)
  static constexpr int UV = UV_;     // FC1 activation values per epilogue work unit (8 or 16)
  // the short-K instantiation (8-value units): all four warps of an epilogue
  // group do activation math, the one on the MMA warp's scheduler included
  // (the epilogue is the limit there; at long K that warp only stages)
  static constexpr bool SHORT_K = UV_ == 8;
  static constexpr int KPS = 2;          // 128-wide K blocks per stage (8 pair MMAs)
  static constexpr int BN = 224;         // token rows per item (both CTAs)
  static constexpr int HALF = BN / 2;    // token rows loaded by each CTA
  static constexpr int NCH = 2;          // 128-row scale chunks of a token tile
  static constexpr int NT = 2;           // weight tiles per item (one per CTA)
  static constexpr int A_KB = 16384;     // 128 rows x 128 FP4 in the unpacked smem format
  static constexpr int A_TX = 8192;      // transaction bytes of that tile (packed source)
  static constexpr int B_BYTES = HALF * 128;
  // stage: A[kbi] (16 KB each), B[kbi] (112 rows), SFA[kbi] (512 B), SFB[kbi] (1 KB)
  static constexpr int B_OFF = KPS * A_KB;
  static constexpr int SFA_OFF = B_OFF + KPS * B_BYTES;
  static constexpr int SFB_OFF = SFA_OFF + KPS * 512;
  static constexpr int STAGE = (SFB_OFF + KPS * NCH * 512 + 1023) / 1024 * 1024;
  // two groups of four warps (one per TMEM lane quarter) taking alternate
  // 32-column chunks: FC1's SiTU epilogue must stay shorter than a short-K
  // main loop, and FC2's scattered fp32 stores with one group were on the
  // critical path (FC2 3.15 -> 2.76 ms at T=8192; 12 or 16 warps: 2.79, 2.83)
  static constexpr int EPI_WARPS = 8;
  static constexpr int NGRP = EPI_WARPS / 4;
  static constexpr int PRODB_WARP = 2 + EPI_WARPS;
  static constexpr int THREADS = 32 * (3 + EPI_WARPS);
  static constexpr int STG_FLOATS = kStgFloats;
  static constexpr int STG_BYTES = FC1 ? NGRP * STG_FLOATS * 4 : 0;
  static constexpr int BAR_OFF = STAGES * STAGE + STG_BYTES;
  static constexpr int TS_OFF = BAR_OFF + 256;  // shared copy of tile_start
  static constexpr int SMEM = 1024 + TS_OFF + kTileStartBytes;
  static constexpr int NACC = 2;
  static constexpr int SF_COL0 = NACC * BN;  // scale columns after the two accumulators
  static constexpr int SFW = 4 + 4 * NCH;    // per K block: own A scales, then all token-row scales
  static constexpr int SF_SLOT = KPS * SFW;  // per stage
  static constexpr int TMEM_COLS = 512;
  // Two scale slots alternate by stage: the copies into a slot are issued
  // after the MMAs that read its previous contents (the tcgen05 operations
  // of one thread run in issue order).
  static_assert(SF_COL0 + 2 * SF_SLOT <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(B_OFF % 1024 == 0 && B_BYTES % 1024 == 0 && STAGE % 1024 == 0,
                "128-byte-swizzled operands start on 1 KB");
};

constexpr int kRing = 8;  // work-item ring slots
// FC1 with at most this many 128-wide K blocks (H = 3584: 28) has a main loop
// short enough that the epilogue is on the critical path: its kernel uses
// 8-value activation units on all four warps of an epilogue group (FC1 3.54
// -> 3.25 ms at H = 3584, I = 3072, T = 8192 with 8-value units on three
// warps, 3.00 -> 2.87 ms on four once the MMA warp issued converged; at
// H = 7168 16-value units on three warps are faster).
constexpr int kShortKBlocks = 32;

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1) moe_gemm_pair_kernel(const __grid_constant__ GemmMaps maps,
                                                                     const GemmArgs a) {
  chain_wait();
  // no tiles of this launch's class: leave before any set-up (every CTA of
  // the cluster reads the same count)
  if (__ldg(a.tile_start + a.E) == 0) return;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done = acc_empty + 2;
  uint64_t* item_full = done + 1;  // [kRing]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(item_full + kRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // MMA width of item li in item_n[li & 3], written by the token producer
  // before it arrives on the item's first stage (so the MMA thread decodes nothing)
  volatile uint32_t* item_n = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);
  // work-item ring: index of the pair's li-th item in item_w[li % kRing]
  volatile int* item_w = reinterpret_cast<volatile int*>(tmem_slot + 6);
  int32_t* tsm = reinterpret_cast<int32_t*>(smem + C::TS_OFF);
  stage_tile_start(a, tsm);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool lead = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 2);  // the even CTA's two producers (plus both CTAs' bytes)
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::NACC; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * C::EPI_WARPS);  // epilogue warps of both CTAs
    }
    mbar_init(done, 1);
    for (int i = 0; i < kRing; ++i) mbar_init(&item_full[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.b[4]);
    prefetch_tmap(&maps.asf);
    prefetch_tmap(&maps.bsf);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = (a.MT / C::NT) * tsm[a.E];
  const uint64_t budget = a.budget_ns;
  // Work items are claimed dynamically (balance across pairs): the even CTA's
  // token producer takes them from a global counter, two ahead of its own
  // progress, and publishes each index to both CTAs' rings (item_full[slot]
  // completes once per publication); every role reads the same sequence, and
  // -1 ends it.  A slot is rewritten only kRing publications later, when every
  // role has long passed it (producers run at most a few stages ahead of the
  // MMA, the MMA at most two items ahead of the epilogues).
  // With DYN off the pair takes items p, p + npairs, ... (no ring).
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const bool fetcher = C::DYN && lead && warp == C::PRODB_WARP;  // the whole warp; lane 0 claims and publishes
  auto get_item = [&](uint32_t li) -> int {
    if (!C::DYN) {
      const int w = pair + static_cast<int>(li) * npairs;
      return w < total ? w : -1;
    }
    const uint32_t sl = li % kRing;
    if (!mbar_wait_bounded<true>(&item_full[sl], (li / kRing) & 1u, budget, a.err, abort_flag)) return -1;
    return item_w[sl];
  };
  // the same, called by every lane of a converged warp
  auto get_item_warp = [&](uint32_t li) -> int {
    if (!C::DYN) {
      const int w = pair + static_cast<int>(li) * npairs;
      return w < total ? w : -1;
    }
    const uint32_t sl = li % kRing;
    if (!mbar_wait_warp<true>(&item_full[sl], (li / kRing) & 1u, budget, a.err, abort_flag)) return -1;
    return item_w[sl];
  };

  if (warp == 0 || warp == C::PRODB_WARP) {
    // ------------------------------------------------------------ producers
    // The whole warp runs the loop converged and one elected lane issues each
    // copy and arrival (ptx.cuh, the _el forms).  Both CTAs' loads complete on
    // the even CTA's full barrier (the TMA .cta_group::2 form); its producers
    // expect the bytes of both CTAs.
    {
      const bool is_a = warp == 0;
      const uint64_t pol = is_a ? policy_evict_normal() : policy_evict_last();
      const uint32_t tx2 = 2u * C::KPS * (is_a ? C::A_TX + 512 : C::B_BYTES + C::NCH * 512);
      const uint32_t lead_full = cluster_map(full, 0);
      uint32_t it = 0;
      bool ok = true;
      // the fetcher's publication state (the same in every lane); each claim
      // (atomicAdd, lane 0) is issued one item before its value is needed, so
      // its latency overlaps the loads
      uint32_t published = 0;
      bool ended = false;
      int claimed = 0;  // lane 0's
      const uint32_t peer_item_full = cluster_map(item_full, 1);
      const uint32_t peer_item_w = cluster_map(const_cast<int*>(item_w), 1);
      auto publish = [&](int w_lane0) {
        int w = __shfl_sync(0xffffffffu, w_lane0, 0);
        if (ended) return;
        if (w >= total) {
          w = -1;
          ended = true;
        }
        const uint32_t sl = published % kRing;
        if (lane == 0) {
          item_w[sl] = w;
          st_shared_cluster_u32(peer_item_w + 4u * sl, static_cast<uint32_t>(w));
          mbar_arrive(&item_full[sl]);                    // release: orders the local store
          mbar_arrive_remote(peer_item_full + 8u * sl);   // release.cluster: orders the remote store
        }
        __syncwarp();
        ++published;
      };
      if (fetcher) {
        int c0 = 0, c1 = 0;
        if (lane == 0) {
          c0 = atomicAdd(a.sched, 1);
          c1 = atomicAdd(a.sched, 1);
          claimed = atomicAdd(a.sched, 1);
        }
        publish(c0);
        publish(c1);
      }
      for (uint32_t li = 0; ok; ++li) {
        int w;
        if (fetcher) {
          w = item_w[li % kRing];  // published by this warp
          if (w >= 0 && !ended) {
            publish(claimed);      // keep two items published ahead
            if (!ended && lane == 0) claimed = atomicAdd(a.sched, 1);
          }
        } else {
          w = get_item_warp(li);
        }
        if (w < 0) break;
        Work wk;
        decode_work(a, tsm, C::BN, C::NT, w, wk);
        const uint32_t nmma = (static_cast<uint32_t>(wk.n) + 15u) & ~15u;
        const int half = static_cast<int>(nmma >> 1);
        const int blk0 = (wk.e * a.MT + C::NT * wk.m + static_cast<int>(rank)) * a.KB;
        const int sfrow0 = wk.tile * a.KB * C::NCH * 4;  // token-tile scale rows of K block 0
        const int brow = wk.r0 + static_cast<int>(rank) * half;
        for (int kb = 0; kb < a.KB; kb += C::KPS, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait_warp(&empty[s], ph ^ 1u, budget, a.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::STAGE;
          const uint32_t bar = lead_full + 8u * s;
          if (lead) {
            if (!is_a && kb == 0) item_n[li & 3u] = nmma;  // every lane stores the same value
            mbar_arrive_expect_tx_el(&full[s], tx2);
          }
#pragma unroll
          for (int kbi = 0; kbi < C::KPS; ++kbi) {
            if (is_a) {
              tma_load_3d_pair_el(st + kbi * C::A_KB, &maps.a, bar, 0, 0, blk0 + kb + kbi, pol);
              tma_load_2d_pair_el(st + C::SFA_OFF + kbi * 512, &maps.asf, bar, 0, 4 * (blk0 + kb + kbi), pol);
            } else {
              // this CTA's half of the MMA's token rows (rows past the tile are
              // loaded but not used; rows past the tensor read as zero)
              tma_load_2d_pair_el(st + C::B_OFF + kbi * C::B_BYTES, &maps.b[4], bar, (kb + kbi) * 128, brow, pol);
              tma_load_2d_pair_el(st + C::SFB_OFF + kbi * C::NCH * 512, &maps.bsf, bar, 0,
                                  sfrow0 + (kb + kbi) * C::NCH * 4, pol);
            }
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA can exit
        if (lead) {
          const uint32_t first = it > static_cast<uint32_t>(C::STAGES) ? it - C::STAGES : 0u;
          for (uint32_t i = first; i < it; ++i)
            mbar_wait_warp(&full[i % C::STAGES], (i / C::STAGES) & 1u, 20000000ull, nullptr, nullptr);
        } else {
          spin_ns(100000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lead) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      // The whole warp runs this loop converged and one elected lane issues
      // each tcgen05 operation (ptx.cuh, the _el forms); the loop stays lean:
      // descriptors are formed once and advanced by adds (the start-address
      // field holds smem offset >> 4), stage and phase advance incrementally,
      // the item's MMA width comes from smem.
      constexpr uint32_t kStageD = C::STAGE >> 4;
      constexpr uint32_t kAD = C::A_KB >> 4, kBD = C::B_BYTES >> 4;
      const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(smem));
      const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(smem + C::B_OFF));
      const uint64_t sfadesc0 = sdesc_sf_32x16(smem_u32(smem + C::SFA_OFF));
      const uint64_t sfbdesc0 = sdesc_sf_32x16(smem_u32(smem + C::SFB_OFF));
      const uint32_t sf_base = tmem + C::SF_COL0;
      int s = 0;
      uint32_t ph = 0, slot = 0;
      bool ok = true;
      for (uint32_t li = 0; ok; ++li) {
        if (get_item_warp(li) < 0) break;
        const uint32_t acc = li & 1u;
        if (!mbar_wait_warp<true>(&acc_empty[acc], ((li >> 1) & 1u) ^ 1u, budget, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * C::BN;
        uint32_t id0 = 0;
        bool two_chunks = false;
        for (int kb = 0; kb < a.KB; kb += C::KPS) {
          if (!mbar_wait_warp(&full[s], ph, budget, a.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (kb == 0) {
            const uint32_t nmma = item_n[li & 3u];
            two_chunks = nmma > 128u;
            id0 = idesc_mxf8f6f4(256, nmma, MX_E2M1, MX_E4M3, 0, 0);
          }
          const uint64_t so = static_cast<uint64_t>(s) * kStageD;
          const uint32_t sf = sf_base + slot;
#pragma unroll
          for (int kbi = 0; kbi < C::KPS; ++kbi) {
            const uint32_t sfa = sf + kbi * C::SFW;
            tc_cp_32x128b_warpx4_pair_el(sfa, sfadesc0 + so + kbi * 32);
            tc_cp_32x128b_warpx4_pair_el(sfa + 4, sfbdesc0 + so + kbi * C::NCH * 32);
            if (two_chunks) tc_cp_32x128b_warpx4_pair_el(sfa + 8, sfbdesc0 + so + kbi * C::NCH * 32 + 32);
            const uint64_t ad = adesc0 + so + kbi * kAD, bd = bdesc0 + so + kbi * kBD;
            mma_mxf8f6f4_pair_el(d, ad, bd, id0, sfa, sfa + 4, (kb | kbi) != 0);
            mma_mxf8f6f4_pair_el(d, ad + 2, bd + 2, id0 | (1u << 4) | (1u << 29), sfa, sfa + 4, 1u);
            mma_mxf8f6f4_pair_el(d, ad + 4, bd + 4, id0 | (2u << 4) | (2u << 29), sfa, sfa + 4, 1u);
            mma_mxf8f6f4_pair_el(d, ad + 6, bd + 6, id0 | (3u << 4) | (3u << 29), sfa, sfa + 4, 1u);
          }
          tc_commit_pair_el(&empty[s]);
          slot ^= C::SF_SLOT;
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_el(&acc_full[acc]);
      }
      tc_commit_pair_el(done);
      mbar_wait_warp(done, 0, budget, a.err, nullptr);
    }
  } else if (warp < C::PRODB_WARP) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int ew = warp - 2;
    const int grp = ew >> 2;
    const int eq = ew & 3;
    // Warp w runs on scheduler w % 4: the MMA warp (1) shares one with the
    // epilogue warp of lane quarter 1, the token producer (PRODB_WARP) with
    // quarter 2's.  At long K the quarter-1 warp leaves the activation math
    // to the other three, and the extra pass goes to the warp whose
    // scheduler hosts no other role; at short K all four do math.
    constexpr int kMmaSchedEq = (1 + 4 - 2) & 3;
    constexpr int kHeavyEq = 1;  // warp 3, scheduler 3
    static_assert(((kHeavyEq + 2) & 3) != (C::PRODB_WARP & 3) && ((kHeavyEq + 2) & 3) != 0 &&
                      ((kHeavyEq + 2) & 3) != 1,
                  "the extra SiTU pass goes to a scheduler without a producer or the MMA warp");
    float* stg = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE) + grp * C::STG_FLOATS;
    const uint32_t lead_acc_empty = cluster_map(acc_empty, 0);
    for (uint32_t li = 0;; ++li) {
      const int w = get_item(li);
      if (w < 0) break;
      Work wk;
      decode_work(a, tsm, C::BN, C::NT, w, wk);
      const uint32_t acc = li & 1u;
      const uint32_t aph = (li >> 1) & 1u;
      bool ok = mbar_wait_bounded(&acc_full[acc], aph, budget, a.err, abort_flag);
      ok = named_barrier_and(1, 32 * C::EPI_WARPS, ok && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      const int mt = C::NT * wk.m + static_cast<int>(rank);  // this CTA's weight tile
      const uint32_t tacc = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * C::BN;
      const int nchunk = (wk.n + 31) >> 5;
      for (int ci = grp; ci < nchunk; ci += C::NGRP)
        epilogue_chunk<C::FC1, C::NCH, C::UV>(a, wk, mt, tacc, ci * 32, stg, q, eq, lane, grp,
                                              C::SHORT_K ? -1 : kMmaSchedEq, C::SHORT_K ? -1 : kHeavyEq);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (lead)
          mbar_arrive(&acc_empty[acc]);
        else
          mbar_arrive_remote(lead_acc_empty + 8u * acc);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no MMA of the pair and no remote arrive is outstanding past here
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

template <class C>
static cudaError_t launch_pair(const GemmMaps& maps, const GemmArgs& a, int sms, cudaStream_t st, bool pdl) {
  static int pairs_of[kMaxDevices] = {};  // co-resident clusters of two (per instantiation and device)
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  int& pairs = pairs_of[dev];
  if (pairs == 0) {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_pair_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, moe_gemm_pair_kernel<C>, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    pairs = n < sms / 2 ? n : sms / 2;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see chain_wait
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, moe_gemm_pair_kernel<C>, maps, a);
}

bool pair_gemm_supported(int MT, int KB) { return MT % 2 == 0 && KB % 2 == 0; }

cudaError_t launch_moe_gemm_pair(bool fc1, const GemmMaps& maps, const GemmArgs& a, int sms, cudaStream_t st,
                                 bool pdl) {
  if (!pair_gemm_supported(a.MT, a.KB)) return cudaErrorInvalidValue;
  // FC1 claims items dynamically (in the fixed order its pairs finished up to
  // 4 % apart at H = 7168, and it is ahead at H = 3584 too); FC2's items do
  // better in the fixed order.
  if (!fc1) return launch_pair<PairCfg<false, 3, false>>(maps, a, sms, st, pdl);
  return a.KB <= kShortKBlocks ? launch_pair<PairCfg<true, 3, true, 8>>(maps, a, sms, st, pdl)
                               : launch_pair<PairCfg<true, 3, true, 16>>(maps, a, sms, st, pdl);
}

}  // namespace kmoe
