// The fused router: gate GEMM (bf16 hidden x bf16 gate weight -> fp32
// logits) and the top-k routing in one kernel (router.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace kmoe {

// Work decomposition of the gate GEMM: token tiles of 128 rows (the MMA's M)
// times expert chunks of EN columns (the MMA's N), one work item each, the
// whole K (= H) per item.  The plan depends on the shape only (never on the
// device), so the logits' rounding is the same on every GPU.
struct RouterPlan {
  int EN;       // experts per item, a multiple of 32 in [32, 256]
  int nch;      // expert chunks: ceil(E / EN)
  int tiles;    // token tiles: ceil(T / 128)
  int items;    // tiles * nch
};

// Picks EN to minimise (rounds of items over 152 SMs) x (MMA time per K step,
// proportional to EN above ~112 columns, flat below); ties go to the smaller
// EN (more SMs streaming the gate weight).
__host__ inline RouterPlan plan_router(int T, int E) {
  constexpr int kSlots = 152;
  RouterPlan best{};
  long long best_cost = -1;
  const int tiles = (T + 127) / 128;
  for (int en = 32; en <= 256; en += 32) {
    const int nch = (E + en - 1) / en;
    const long long items = static_cast<long long>(tiles) * nch;
    const long long rounds = (items + kSlots - 1) / kSlots;
    const long long cost = rounds * (en > 112 ? en : 112);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = RouterPlan{en, nch, tiles, static_cast<int>(items)};
    }
  }
  return best;
}

// Bytes of the router's synchronisation words: the token counter of the
// routing warps and one completion counter per token tile.
__host__ inline size_t router_sync_bytes(int T) { return static_cast<size_t>(2 + (T + 127) / 128) * 4; }

struct RouterMaps {
  CUtensorMap x;  // bf16 [T, H], box 64 x 128, 128-byte swizzle
  CUtensorMap g;  // bf16 [E, H], box 64 x EN, 128-byte swizzle
};

struct RouterArgs {
  int T, H, E, k;
  RouterPlan plan;
  const float* bias;   // [E]
  float* logits;       // [T, E] fp32 (written, then read back by the routing warps)
  int32_t* ids;        // [T, k]
  float* wts;          // [T, k]
  int* sync;           // router_sync_bytes(T), zeroed by the launch
  uint32_t* err;       // device error word
  unsigned long long budget_ns;
};

// Launches the fused router on `sms` CTAs (one per SM, co-resident: a
// cooperative launch).  Zeroes a.sync first.  Requires E % 4 == 0, H % 64 == 0.
cudaError_t launch_router(const RouterMaps& maps, const RouterArgs& a, int sms, cudaStream_t st);

}  // namespace kmoe
