// The fused router: the gate GEMM (logits = x W_g^T, bf16 operands, fp32
// accumulation) and the sigmoid + correction-bias top-k of every token in one
// kernel (Kimi-K3 SM120 FlashInfer MXFP4 page, "Phase 1: serving call chain":
// the TopK step consumes the gate's logits).
//
// One persistent CTA per SM, all co-resident (cooperative launch).
//   warp 0        TMA producer: per K step of 64, the x tile (128 tokens, or
//                 32 / 64 when T is that small) and the EN-expert gate tile
//                 (both bf16, 128-byte swizzle); as many pipeline stages as
//                 192 KB holds, up to 24 (4 at EN = 256 with 128-token x
//                 tiles, 24 at EN = 32 with 32-token tiles), since the loop
//                 is bound by the bytes in flight per SM; the warp runs
//                 converged and one elected lane issues each copy
//   warp 1        TMEM owner and MMA issuer: tcgen05.mma .kind::f16 (bf16 x
//                 bf16 -> fp32), M = 128 tokens, N = EN experts, K = 16 per
//                 instruction; two 256-column accumulators so that the
//                 epilogue of one item overlaps the next item's main loop
//   warps 2..5    epilogue: TMEM -> registers -> a swizzled smem tile ->
//                 coalesced fp32 rows of the logits; then the item's token
//                 tile completion counter is bumped (fence + atomic).  With K
//                 split S ways (few items: decode) each split writes a
//                 partial tile and the last split of a (tile, chunk) to
//                 finish sums the S partials in split order into the logits
//   warps 6..15   routing: first copy the correction bias into shared
//                 memory, then take tokens one at a time from a global
//                 counter, wait (bounded) until every expert chunk of the
//                 token's tile is written, route the token (route_dev.cuh)
// The GEMM warps join the routing pool when their work runs out, so routing
// of finished token tiles overlaps the gate GEMM of the rest.  Every wait is
// bounded; a wait that gives up sets the timeout bit and the token is left
// masked (ids -1).  When there are enough token tiles (prefill), the plan
// takes router_pair_kernel instead: the same roles on clusters of two CTAs
// with M = 256 tensor-core pairs.
#include "gemm_dev.cuh"  // named_barrier_and
#include "route_dev.cuh"
#include "router.cuh"

namespace kmoe {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kFirstRouteWarp = 6;
constexpr int kMaxStages = 24;
constexpr int kATile = 128 * 128;        // 128 tokens x 64 bf16 (the MMA's M = 128 rows)
constexpr int kStageArea = 192 * 1024;   // stages of the x tile + EN x 128 bytes, 1 KB aligned
constexpr int kStgOff = kStageArea;      // epilogue staging: 32 x 32 fp32 per warp
constexpr int kBarOff = kStgOff + 4 * 4096;
constexpr int kBiasOff = kBarOff + 512;
constexpr int kIdxOff = kBiasOff + 4 * kMaxE;
constexpr int kSmem = 1024 + kIdxOff + kWarps * 32 * 4;
constexpr uint32_t kTmemCols = 512;  // two accumulators of up to 256 columns
static_assert(kSmem <= 232448, "shared memory budget");

// bf16 instruction descriptor of tcgen05.mma .kind::f16: fp32 D (bits 4-5 =
// 1), A and B bf16 (bits 7-9, 10-12 = 1), both K-major, N>>3 at bit 17, M>>4
// at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A x B^T over K = 16 (32 bytes of each smem row), executed by
// every lane of a converged warp; one elected lane issues (see the
// warp-converged forms in ptx.cuh).  The _pair form (M = 256, issued by the
// even CTA): CTA r supplies A rows [128r, 128r+128) and B rows
// [rN/2, (r+1)N/2) from its own shared memory; each CTA's TMEM gets its
// 128 x N accumulator.
__device__ __forceinline__ void mma_bf16_el(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred e, p;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_bf16_pair_el(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred e, p;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One warp's 32 token rows of an item's accumulator (TMEM columns
// [0, EN) at `tacc`, lane quarter included) to fp32 logits rows t0..t0+31,
// columns e_base..e_base+EN-1 of dst [T, E]: TMEM -> registers -> a
// swizzled 32 x 32 smem tile (row `lane`'s 16-byte unit u at u ^ (lane & 7))
// -> 8 lanes per row, 128 contiguous bytes, 4 rows per store.
__device__ __forceinline__ void store_logit_tile(uint32_t tacc, int EN, float* stg, int lane, int t0, int e_base,
                                                 int T, int E, float* dst) {
  for (int c0 = 0; c0 < EN; c0 += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(tacc + c0, r);
    tmem_ld_wait();
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<float4*>(stg + lane * 32 + ((u ^ (lane & 7)) << 2)) =
          make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]), __uint_as_float(r[4 * u + 2]),
                      __uint_as_float(r[4 * u + 3]));
    __syncwarp();
    const int e0 = e_base + c0 + 4 * (lane & 7);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = 4 * i + (lane >> 3);
      const int t = t0 + rr;
      const float4 v = *reinterpret_cast<const float4*>(stg + rr * 32 + (((lane & 7) ^ (rr & 7)) << 2));
      if (t < T && e0 < E) *reinterpret_cast<float4*>(dst + static_cast<size_t>(t) * E + e0) = v;
    }
    __syncwarp();
  }
}

// The bias is read by the routing warps after the set-up, off the path of
// the GEMM roles (a cold read takes over a microsecond); each thread arrives
// on bias_bar after its stores, and every warp waits on it before routing.
__device__ __forceinline__ void load_bias(const RouterArgs& a, float* s_b, uint64_t* bias_bar, int warp) {
  if (warp < kFirstRouteWarp) return;
  for (int e = threadIdx.x - 32 * kFirstRouteWarp; e < a.E; e += 32 * (kWarps - kFirstRouteWarp)) s_b[e] = a.bias[e];
  mbar_arrive(bias_bar);
}

// Routing warps: tokens are handed out in increasing order, so the first
// tiles' tokens are routed while later tiles are still in the GEMM.
template <int KPL>
__device__ void route_pool(const RouterArgs& a, const float* s_b, uint64_t* bias_bar, int* s_idx, int lane) {
  if (!mbar_wait_warp(bias_bar, 0, a.budget_ns, a.err, nullptr)) return;
  int* next = a.sync;
  const int* tile_done = a.sync + 2;
  const int need = a.plan.nch;  // one count per expert chunk of the tile
  for (;;) {
    int t = 0;
    if (lane == 0) t = atomicAdd(next, 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t >= a.T) break;
    // Every lane polls (an acquire load each) and the loop exits together:
    // a wait run by one lane left the warp executing the routing diverged,
    // at about three times the time per token.
    const int* c = tile_done + (t >> 7);
    int ready = 1;
    const uint64_t t0 = globaltimer_ns();
    while (!__all_sync(0xffffffffu, ld_acquire_gpu(c) >= need)) {
      __nanosleep(256);
      const bool late = (*reinterpret_cast<volatile uint32_t*>(a.err) & KMOE_DEVERR_TIMEOUT) ||
                        globaltimer_ns() - t0 > a.budget_ns;
      if (__any_sync(0xffffffffu, late)) {
        if (lane == 0) atomicOr(a.err, KMOE_DEVERR_TIMEOUT);
        ready = 0;
        break;
      }
    }
    int32_t* ids_row = a.ids + static_cast<size_t>(t) * a.k;
    float* w_row = a.wts + static_cast<size_t>(t) * a.k;
    if (!ready) {
      if (lane < a.k) {
        ids_row[lane] = -1;
        w_row[lane] = 0.f;
      }
      continue;
    }
    route_token<KPL>(a.logits + static_cast<size_t>(t) * a.E, s_b, a.E, a.k, lane, ids_row, w_row, s_idx);
  }
}

template <int KPL>
__global__ void __launch_bounds__(kThreads, 1) router_kernel(const __grid_constant__ RouterMaps maps,
                                                             const RouterArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kMaxStages;
  uint64_t* acc_full = empty + kMaxStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done = acc_empty + 2;
  uint64_t* bias_bar = done + 1;  // the routing warps' copy of the bias is in s_b
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bias_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);  // epilogue: last split
  float* s_b = reinterpret_cast<float*>(smem + kBiasOff);
  int* s_idx = reinterpret_cast<int*>(smem + kIdxOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int EN = a.plan.EN, nch = a.plan.nch, items = a.plan.items, S = a.plan.S, kper = a.plan.kper;
  // a stage holds the x tile (xrows of the MMA's 128 A rows: the MMA reads
  // past it into the rest of shared memory for the rows >= T, whose
  // accumulator lanes are never stored) and the EN-expert gate tile; small
  // batches thus fit more stages in flight
  const int atile = a.xrows * 128;
  const int stride = (atile + EN * 128 + 1023) & ~1023;  // bytes per pipeline stage
  const int nst = kStageArea / stride < kMaxStages ? kStageArea / stride : kMaxStages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(done, 1);
    mbar_init(bias_bar, 32 * (kWarps - kFirstRouteWarp));
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.x);
    prefetch_tmap(&maps.g);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  load_bias(a, s_b, bias_bar, warp);
  const int KS = a.H / 64;
  const uint64_t budget = a.budget_ns;
  int* tile_done = a.sync + 2;
  int* split_done = a.sync + 2 + a.plan.tiles;
  // item it -> (token tile mt, expert chunk nc, K split sp), splits fastest
  auto decode = [&](int it, int& mt, int& nc, int& sp) {
    const int b = it / S;
    sp = it - b * S;
    mt = b / nch;
    nc = b - mt * nch;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // the whole warp runs the loop converged; one elected lane issues
    {
      const uint32_t tx = static_cast<uint32_t>(a.xrows + EN) * 128;
      const uint64_t pol_x = policy_evict_normal();
      const uint64_t pol_g = policy_evict_last();  // the gate weight is re-read by every token tile
      uint32_t n = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        int mt, nc, sp;
        decode(it, mt, nc, sp);
        const int ks1 = (sp + 1) * kper < KS ? (sp + 1) * kper : KS;
        for (int ks = sp * kper; ks < ks1; ++ks, ++n) {
          const int s = static_cast<int>(n % nst);
          const uint32_t ph = (n / nst) & 1u;
          if (!mbar_wait_warp(&empty[s], ph ^ 1u, budget, a.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * stride;
          mbar_arrive_expect_tx_el(&full[s], tx);
          tma_load_2d_el(st, &maps.x, &full[s], 64 * ks, 128 * mt, pol_x);
          tma_load_2d_el(st + atile, &maps.g, &full[s], 64 * ks, EN * nc, pol_g);
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA can exit
        const uint32_t first = n > static_cast<uint32_t>(nst) ? n - nst : 0u;
        for (uint32_t i = first; i < n; ++i)
          mbar_wait_warp(&full[i % nst], (i / nst) & 1u, 20000000ull, nullptr, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // the whole warp runs the loop converged; one elected lane issues
    {
      const uint32_t idesc = idesc_bf16(128, static_cast<uint32_t>(EN));
      const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(smem));
      const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(smem + atile));
      int s = 0;
      uint32_t ph = 0, li = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x, ++li) {
        int mt, nc, sp;
        decode(it, mt, nc, sp);
        const int nks = ((sp + 1) * kper < KS ? (sp + 1) * kper : KS) - sp * kper;
        const uint32_t acc = li & 1u;
        const uint32_t aph = (li >> 1) & 1u;
        if (!mbar_wait_warp(&acc_empty[acc], aph ^ 1u, budget, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * 256u;
        for (int ks = 0; ks < nks; ++ks) {
          if (!mbar_wait_warp(&full[s], ph, budget, a.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = static_cast<uint64_t>(s) * static_cast<uint64_t>(stride >> 4);
          mma_bf16_el(d, adesc0 + so, bdesc0 + so, idesc, ks != 0);
          mma_bf16_el(d, adesc0 + so + 2, bdesc0 + so + 2, idesc, 1u);
          mma_bf16_el(d, adesc0 + so + 4, bdesc0 + so + 4, idesc, 1u);
          mma_bf16_el(d, adesc0 + so + 6, bdesc0 + so + 6, idesc, 1u);
          tc_commit_el(&empty[s]);
          if (++s == nst) {
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
    __syncwarp();
  } else if (warp < kFirstRouteWarp) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter of this warp
    float* stg = reinterpret_cast<float*>(smem + kStgOff) + (warp - 2) * 1024;
    uint32_t li = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x, ++li) {
      const uint32_t acc = li & 1u;
      const uint32_t aph = (li >> 1) & 1u;
      bool ok = mbar_wait_bounded(&acc_full[acc], aph, budget, a.err, abort_flag);
      ok = named_barrier_and(1, 128, ok && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      int mt, nc, sp;
      decode(it, mt, nc, sp);
      const int t0 = 128 * mt + 32 * q;
      float* dst = S > 1 ? a.part + static_cast<size_t>(sp) * a.T * a.E : a.logits;
      store_logit_tile(tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * 256u, EN, stg, lane, t0, nc * EN, a.T,
                       a.E, dst);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      // publish: every writer's stores before a counter moves
      __threadfence();
      named_barrier(1, 128);
      if (S > 1) {
        // the last of the S splits of (mt, nc) sums the partial tiles in split order
        const int tid = threadIdx.x - 64;  // 0..127
        if (tid == 0) *last_flag = atomicAdd(split_done + mt * nch + nc, 1) == S - 1;
        named_barrier(1, 128);
        const bool last = *last_flag != 0;
        named_barrier(1, 128);  // the flag is read before the next item rewrites it
        if (!last) continue;
        __threadfence();
        const int rows = a.T - 128 * mt < 128 ? a.T - 128 * mt : 128;
        const int q4 = EN / 4;
        for (int idx = tid; idx < rows * q4; idx += 128) {
          const int r = idx / q4;
          const int e = nc * EN + 4 * (idx - r * q4);
          if (e >= a.E) continue;
          const size_t off = static_cast<size_t>(128 * mt + r) * a.E + e;
          float4 acc4 = __ldcg(reinterpret_cast<const float4*>(a.part + off));
          for (int p = 1; p < S; ++p) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(a.part + static_cast<size_t>(p) * a.T * a.E + off));
            acc4.x += v.x;
            acc4.y += v.y;
            acc4.z += v.z;
            acc4.w += v.w;
          }
          *reinterpret_cast<float4*>(a.logits + off) = acc4;
        }
        __threadfence();
        named_barrier(1, 128);
      }
      if (warp == 2 && lane == 0) atomicAdd(tile_done + mt, 1);
    }
  }
  route_pool<KPL>(a, s_b, bias_bar, s_idx + warp * 32, lane);

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The gate GEMM on CTA pairs (plan.pair): a cluster of two CTAs runs item
// (token-tile pair tp, expert chunk nc) as tcgen05.mma.cta_group::2 of M = 256
// tokens (CTA r: token tile 2tp + r) by N = EN experts (CTA r holds gate rows
// [EN nc + r EN/2, +EN/2)); each CTA's TMEM receives its own 128 x EN
// accumulator, which its epilogue writes as logits rows of its token tile.
// Both CTAs' loads complete on the even CTA's full barrier (TMA
// .cta_group::2); the even CTA's MMA commits arrive on both CTAs' empty and
// acc_full barriers; acc_empty of the even CTA counts both CTAs' epilogue
// warps.  Routing as in router_kernel.  No K split (pairs are used only when
// there are enough token tiles).
template <int KPL>
__global__ void __launch_bounds__(kThreads, 1) router_pair_kernel(const __grid_constant__ RouterMaps maps,
                                                                  const RouterArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kMaxStages;
  uint64_t* acc_full = empty + kMaxStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done = acc_empty + 2;
  uint64_t* bias_bar = done + 1;  // the routing warps' copy of the bias is in s_b
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bias_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* s_b = reinterpret_cast<float*>(smem + kBiasOff);
  int* s_idx = reinterpret_cast<int*>(smem + kIdxOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool lead = rank == 0;
  const int EN = a.plan.EN, nch = a.plan.nch, items = a.plan.items, tiles = a.plan.tiles;
  const int half = EN / 2;
  const int stride = (kATile + half * 128 + 1023) & ~1023;  // bytes per pipeline stage
  const int nst = kStageArea / stride < kMaxStages ? kStageArea / stride : kMaxStages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);   // the even CTA's producer (plus both CTAs' bytes)
      mbar_init(&empty[s], 1);  // the pair MMA's commit (multicast)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);  // the epilogue warps of both CTAs
    }
    mbar_init(done, 1);
    mbar_init(bias_bar, 32 * (kWarps - kFirstRouteWarp));
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.x);
    prefetch_tmap(&maps.g);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  load_bias(a, s_b, bias_bar, warp);
  const int KS = a.H / 64;
  const uint64_t budget = a.budget_ns;
  int* tile_done = a.sync + 2;
  const int pairi = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (warp == 0) {
    // ---------------------------------------------------------------- producers (both CTAs)
    // the whole warp runs the loop converged; one elected lane issues
    {
      const uint32_t tx2 = 2u * static_cast<uint32_t>(kATile + half * 128);
      const uint64_t pol_x = policy_evict_normal();
      const uint64_t pol_g = policy_evict_last();
      const uint32_t lead_full = cluster_map(full, 0);
      uint32_t n = 0;
      bool ok = true;
      for (int it = pairi; it < items && ok; it += npairs) {
        const int tp = it / nch, nc = it - tp * nch;
        const int mt = 2 * tp + static_cast<int>(rank);
        const int grow = EN * nc + static_cast<int>(rank) * half;
        for (int ks = 0; ks < KS; ++ks, ++n) {
          const int s = static_cast<int>(n % nst);
          const uint32_t ph = (n / nst) & 1u;
          if (!mbar_wait_warp(&empty[s], ph ^ 1u, budget, a.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * stride;
          const uint32_t bar = lead_full + 8u * static_cast<uint32_t>(s);
          if (lead) mbar_arrive_expect_tx_el(&full[s], tx2);
          tma_load_2d_pair_el(st, &maps.x, bar, 64 * ks, 128 * mt, pol_x);
          tma_load_2d_pair_el(st + kATile, &maps.g, bar, 64 * ks, grow, pol_g);
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA can exit
        if (lead) {
          const uint32_t first = n > static_cast<uint32_t>(nst) ? n - nst : 0u;
          for (uint32_t i = first; i < n; ++i)
            mbar_wait_warp(&full[i % nst], (i / nst) & 1u, 20000000ull, nullptr, nullptr);
        } else {
          spin_ns(100000ull);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    // the whole warp runs the loop converged; one elected lane issues
    if (lead) {
      const uint32_t idesc = idesc_bf16(256, static_cast<uint32_t>(EN));
      const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(smem));
      const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(smem + kATile));
      int s = 0;
      uint32_t ph = 0, li = 0;
      bool ok = true;
      for (int it = pairi; it < items && ok; it += npairs, ++li) {
        const uint32_t acc = li & 1u;
        if (!mbar_wait_warp<true>(&acc_empty[acc], ((li >> 1) & 1u) ^ 1u, budget, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * 256u;
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait_warp(&full[s], ph, budget, a.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = static_cast<uint64_t>(s) * static_cast<uint64_t>(stride >> 4);
          mma_bf16_pair_el(d, adesc0 + so, bdesc0 + so, idesc, ks != 0);
          mma_bf16_pair_el(d, adesc0 + so + 2, bdesc0 + so + 2, idesc, 1u);
          mma_bf16_pair_el(d, adesc0 + so + 4, bdesc0 + so + 4, idesc, 1u);
          mma_bf16_pair_el(d, adesc0 + so + 6, bdesc0 + so + 6, idesc, 1u);
          tc_commit_pair_el(&empty[s]);
          if (++s == nst) {
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
    __syncwarp();
  } else if (warp < kFirstRouteWarp) {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;
    float* stg = reinterpret_cast<float*>(smem + kStgOff) + (warp - 2) * 1024;
    const uint32_t lead_acc_empty = cluster_map(acc_empty, 0);
    uint32_t li = 0;
    for (int it = pairi; it < items; it += npairs, ++li) {
      const uint32_t acc = li & 1u;
      bool ok = mbar_wait_bounded(&acc_full[acc], (li >> 1) & 1u, budget, a.err, abort_flag);
      ok = named_barrier_and(1, 128, ok && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      const int tp = it / nch, nc = it - tp * nch;
      const int mt = 2 * tp + static_cast<int>(rank);
      store_logit_tile(tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * 256u, EN, stg, lane, 128 * mt + 32 * q,
                       nc * EN, a.T, a.E, a.logits);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (lead)
          mbar_arrive(&acc_empty[acc]);
        else
          mbar_arrive_remote(lead_acc_empty + 8u * acc);
      }
      // publish: every writer's stores before the tile's counter moves
      __threadfence();
      named_barrier(1, 128);
      if (warp == 2 && lane == 0 && mt < tiles) atomicAdd(tile_done + mt, 1);
    }
  }
  route_pool<KPL>(a, s_b, bias_bar, s_idx + warp * 32, lane);

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no MMA of the pair and no remote arrive is outstanding past here
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <int KPL>
cudaError_t launch_pair_kpl(const RouterMaps& maps, const RouterArgs& a, int sms, cudaStream_t st) {
  static int pairs_of[kMaxDevices] = {};  // co-resident clusters of two (per instantiation and device)
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  int& pairs = pairs_of[dev];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeCooperative;  // the routing warps wait on other CTAs' tiles
  at[1].val.cooperative = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  if (pairs == 0) {
    cudaError_t e =
        cudaFuncSetAttribute(router_pair_kernel<KPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (sms / 2)), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, router_pair_kernel<KPL>, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    pairs = n < sms / 2 ? n : sms / 2;
  }
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  return cudaLaunchKernelEx(&cfg, router_pair_kernel<KPL>, maps, a);
}

template <int KPL>
cudaError_t launch_kpl(const RouterMaps& maps, const RouterArgs& a, int sms, cudaStream_t st) {
  static int ready_on[kMaxDevices] = {};  // attribute set and occupancy checked (per instantiation and device)
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  int& ready = ready_on[dev];
  if (!ready) {
    cudaError_t e = cudaFuncSetAttribute(router_kernel<KPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, router_kernel<KPL>, kThreads, kSmem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    ready = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;  // the routing warps wait on other CTAs' tiles
  at[0].val.cooperative = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(sms), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, router_kernel<KPL>, maps, a);
}

}  // namespace

cudaError_t launch_router(const RouterMaps& maps, const RouterArgs& a, int sms, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (a.E % 4 != 0 || a.H % 64 != 0 || a.E > kMaxE || sms <= 0) return cudaErrorInvalidValue;
  if (a.xrows != 32 && a.xrows != 64 && a.xrows != 128) return cudaErrorInvalidValue;
  if (a.plan.S > 1 && a.part == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(a.sync, 0, router_sync_bytes(a.plan), st);
  if (e != cudaSuccess) return e;
  if (a.plan.pair) {
    if (a.xrows != 128 || a.plan.S != 1) return cudaErrorInvalidValue;
    if (a.E <= 64) return launch_pair_kpl<2>(maps, a, sms, st);
    if (a.E <= 256) return launch_pair_kpl<8>(maps, a, sms, st);
    return launch_pair_kpl<32>(maps, a, sms, st);
  }
  if (a.E <= 64) return launch_kpl<2>(maps, a, sms, st);
  if (a.E <= 256) return launch_kpl<8>(maps, a, sms, st);
  return launch_kpl<32>(maps, a, sms, st);
}

}  // namespace kmoe
