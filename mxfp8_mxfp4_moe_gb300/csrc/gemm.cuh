// Arguments and launcher of the grouped block-scaled expert GEMMs (gemm.cu).
#pragma once
#include "common.cuh"

namespace kmoe {

// One prepared weight block: 128 tile rows x 64 code bytes + 512 scale bytes
// (codes of all blocks first, then the scales of all blocks).
constexpr int kWeightBlockBytes = 8192 + 512;

// Tensor maps of one grouped GEMM: the weight codes (box of kps K blocks)
// and the token rows in boxes of 32, 64, 128 rows, of one whole tile and of
// half a tile (the share of one CTA of a pair).
struct GemmMaps {
  CUtensorMap a;
  CUtensorMap b[5];
  CUtensorMap asf;  // weight scales as rows of 128 B, box of 4 rows (one block)
  CUtensorMap bsf;  // token-tile scales as rows of 128 B, box of one K block of a tile
};

// K blocks (of 128) moved per pipeline stage for a token-tile size and a K
// of KB blocks: two for the 32-row tiles when KB is even, else one (the
// 64-row tiles run two CTAs per SM with single-K-block stages).
inline int gemm_kblocks_per_stage(int BN, int KB) { return (BN <= 32 && KB % 2 == 0) ? 2 : 1; }

struct GemmArgs {
  const int32_t* counts;      // [E]
  const int32_t* seg_start;   // [E+1]
  const int32_t* tile_start;  // [E+1]
  const uint8_t* wq;          // prepared weight codes: [E][MT][KB] blocks of 128 rows x 64 B
  const uint8_t* wsf;         // prepared weight scales: [E][MT][KB] blocks of 512 B
  const uint8_t* bsf;         // token-tile-layout scales of the B rows
  int E, MT, KB, max_tiles;
  int H, I;
  // FC1 epilogue
  uint8_t* iq;   // [R, I] E4M3 codes of SiTU output
  uint8_t* isf;  // token-tile-layout scales (K = I)
  float kg, ku, bb;            // SiTU: 2/situ_beta, 2/situ_linear_beta, situ_beta*situ_linear_beta
  // FC2 epilogue
  float* y;                   // [T*k, H]
  const int32_t* slot_of_row;  // [R]
  uint32_t* err;
  unsigned long long budget_ns;
  int* sched;  // work-item counter of this launch (zero before it; CTA-pair kernel)
  // FC1 activation: 0 = SiTU (kg, ku, bb above), 1 = the clamped SwiGLU control
  int act;
  float sw_alpha, sw_beta, sw_limit;
};

// Re-lays raw codes [E, rows, K/2] and scales [E, rows, K/32] into prepared blocks.
cudaError_t launch_prep_weights(const uint8_t* codes, const uint8_t* sf, uint8_t* out, int E, int MT, int KB,
                                int rows_per_expert, int K, int fc1, int I, cudaStream_t st);

// fc1: FC1 with the SiTU + MXFP8 requantisation epilogue; otherwise FC2 with
// fp32 per-slot stores.  BN is the token-tile size of the layer (32, 64, 224).
// kps must equal gemm_kblocks_per_stage(BN, a.KB) (the depth of maps.a's box).
// pdl: launched with programmatic stream serialization (its predecessor on
// the stream is a kernel of the same forward chain).
cudaError_t launch_moe_gemm(bool fc1, int BN, int kps, const GemmMaps& maps, const GemmArgs& a, int grid,
                            cudaStream_t st, bool pdl);

// The CTA-pair kernel for BN = 224 (gemm_pair.cu): weight tiles per expert
// (MT) and K blocks (KB) must both be even.  `sms` is the SM count; the grid
// is the number of co-resident pairs.
bool pair_gemm_supported(int MT, int KB);
cudaError_t launch_moe_gemm_pair(bool fc1, const GemmMaps& maps, const GemmArgs& a, int sms, cudaStream_t st,
                                 bool pdl);

}  // namespace kmoe
