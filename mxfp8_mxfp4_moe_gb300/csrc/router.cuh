// The fused router: gate GEMM (bf16 hidden x bf16 gate weight -> fp32
// logits) and the top-k routing in one kernel (router.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace kmoe {

struct RouterMaps {
  CUtensorMap x;  // bf16 [T, H], box 64 x xrows, 128-byte swizzle
  CUtensorMap g;  // bf16 [E, H], box 64 x EN, 128-byte swizzle
};

struct RouterArgs {
  int T, H, E, k;
  int xrows;           // rows of the x box: 32, 64 (T that small) or 128
  RouterPlan plan;
  const float* bias;   // [E]
  float* logits;       // [T, E] fp32 (written, then read back by the routing warps)
  float* part;         // [S, T, E] fp32 partial sums of the K splits (S > 1 only)
  int32_t* ids;        // [T, k]
  float* wts;          // [T, k]
  int* sync;           // router_sync_bytes(plan), zeroed by the launch
  uint32_t* err;       // device error word
  unsigned long long budget_ns;
};

// Launches the fused router on `sms` CTAs (one per SM, co-resident: a
// cooperative launch).  Zeroes a.sync first.  Requires E % 4 == 0, H % 64 == 0.
cudaError_t launch_router(const RouterMaps& maps, const RouterArgs& a, int sms, cudaStream_t st);

}  // namespace kmoe
