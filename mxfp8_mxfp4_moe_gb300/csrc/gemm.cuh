// Arguments and launcher of the grouped block-scaled expert GEMMs (gemm.cu).
#pragma once
#include "common.cuh"

namespace kmoe {

struct GemmArgs {
  const int32_t* counts;      // [E]
  const int32_t* seg_start;   // [E+1]
  const int32_t* tile_start;  // [E+1]
  const uint8_t* wsf;         // prepared weight scales [E][MT][KB][512]
  const uint8_t* bsf;         // token-tile-layout scales of the B rows
  int E, MT, KB, max_tiles;
  int H, I;
  // FC1 epilogue
  uint8_t* iq;   // [R, I] E4M3 codes of SiTU output
  uint8_t* isf;  // token-tile-layout scales (K = I)
  float beta, beta_lin;
  // FC2 epilogue
  float* y;                   // [T*k, H]
  const int32_t* slot_of_row;  // [R]
  uint32_t* err;
  unsigned long long budget_ns;
};

// fc1: FC1 with the SiTU + MXFP8 requantisation epilogue; otherwise FC2 with
// fp32 per-slot stores.  BN is the token-tile size of the layer (32, 64, 224).
cudaError_t launch_moe_gemm(bool fc1, int BN, const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmArgs& a,
                            int grid, cudaStream_t st);

}  // namespace kmoe
