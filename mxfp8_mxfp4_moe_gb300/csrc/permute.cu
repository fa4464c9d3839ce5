// Expert permutation: per-expert histogram, exclusive scans and a stable
// rank of every routed slot among the slots of its expert, so that the rows
// of each expert form one contiguous, token-ordered segment.  The grouped
// GEMMs walk those segments in token tiles of `BN` rows.
//
//   pass 1 (rank_kernel, one block per 1024 slots): stable rank of each slot
//          inside its block (warps in order, __match_any_sync inside a warp)
//          and the block's per-expert counts.
//   pass 2 (scan_kernel, one block): per-expert totals, prefix over blocks,
//          segment starts and the tile starts of the two tile classes:
//          experts with at most `thr` rows are cut into tiles of BN rows
//          (tile_start: prefix of ceil(count/BN) over those experts), the
//          others into tiles of kBigTileRows rows (tile_start_big).
// Batches of at most kRankChunk slots (decode) take both passes in one block
// (permute_small_kernel): one launch, the counts staying in shared memory.
// The final row of slot s is seg_start[e] + chunk_prefix[block][e] + rank[s];
// it is computed where the row is written (the quantise-scatter kernel).
#include "common.cuh"

namespace kmoe {

__global__ void __launch_bounds__(kRankChunk) rank_kernel(const int32_t* __restrict__ ids, int R, int E,
                                                          int32_t* __restrict__ rank,
                                                          int32_t* __restrict__ chunk_counts,
                                                          uint32_t* __restrict__ err) {
  chain_wait();
  extern __shared__ int cnt[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int s = blockIdx.x * kRankChunk + threadIdx.x;
  int id = s < R ? ids[s] : -1;
  if (id >= E) {
    atomicOr(err, 2u);  // KMOE_DEVERR_BOUNDS: an expert id out of range (treated as masked)
    id = -1;
  }
  const bool valid = id >= 0;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const unsigned peers = __match_any_sync(0xffffffffu, valid ? id : -1);
  const unsigned lower = peers & ((1u << lane) - 1u);
  const int nwarps = blockDim.x >> 5;
  int my = -1;
  for (int w = 0; w < nwarps; ++w) {
    int base = 0;
    if (warp == w && valid) base = cnt[id];
    __syncwarp();
    if (warp == w && valid) {
      my = base + __popc(lower);
      if (lower == 0) cnt[id] = base + __popc(peers);
    }
    __syncthreads();
  }
  if (s < R) rank[s] = my;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[static_cast<size_t>(blockIdx.x) * E + e] = cnt[e];
}

// Single block.  chunk_counts [nchunk][E] becomes its exclusive prefix over
// chunks; counts/seg_start/tile_start are written.
__device__ __forceinline__ int small_tiles(int c, int BN, int thr) { return c <= thr ? (c + BN - 1) / BN : 0; }
__device__ __forceinline__ int big_tiles(int c, int thr) {
  return c > thr ? (c + kBigTileRows - 1) / kBigTileRows : 0;
}

__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ chunk_counts, int nchunk, int E, int BN,
                                                    int thr, int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ seg_start, int32_t* __restrict__ tile_start,
                                                    int32_t* __restrict__ tile_start_big) {
  chain_wait();
  __shared__ int s_rows[1024];
  __shared__ int s_tiles[1024];
  __shared__ int s_big[1024];
  const int per = (E + blockDim.x - 1) / blockDim.x;  // experts per thread (contiguous)
  const int e0 = threadIdx.x * per;
  int rows = 0, tiles = 0, bigt = 0;
  for (int e = e0; e < e0 + per && e < E; ++e) {
    int run = 0;
    // batches of independent loads, then the running prefix (keeps loads in flight)
    for (int c0 = 0; c0 < nchunk; c0 += 16) {
      int v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        v[i] = (c0 + i < nchunk) ? chunk_counts[static_cast<size_t>(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (c0 + i < nchunk) chunk_counts[static_cast<size_t>(c0 + i) * E + e] = run;
        run += v[i];
      }
    }
    counts[e] = run;
    rows += run;
    tiles += small_tiles(run, BN, thr);
    bigt += big_tiles(run, thr);
  }
  s_rows[threadIdx.x] = rows;
  s_tiles[threadIdx.x] = tiles;
  s_big[threadIdx.x] = bigt;
  __syncthreads();
  // inclusive Hillis-Steele scan over threads
  for (int off = 1; off < blockDim.x; off <<= 1) {
    int vr = threadIdx.x >= off ? s_rows[threadIdx.x - off] : 0;
    int vt = threadIdx.x >= off ? s_tiles[threadIdx.x - off] : 0;
    int vb = threadIdx.x >= off ? s_big[threadIdx.x - off] : 0;
    __syncthreads();
    s_rows[threadIdx.x] += vr;
    s_tiles[threadIdx.x] += vt;
    s_big[threadIdx.x] += vb;
    __syncthreads();
  }
  int r = threadIdx.x > 0 ? s_rows[threadIdx.x - 1] : 0;
  int t = threadIdx.x > 0 ? s_tiles[threadIdx.x - 1] : 0;
  int b = threadIdx.x > 0 ? s_big[threadIdx.x - 1] : 0;
  for (int e = e0; e < e0 + per && e < E; ++e) {
    seg_start[e] = r;
    tile_start[e] = t;
    tile_start_big[e] = b;
    const int c = counts[e];
    r += c;
    t += small_tiles(c, BN, thr);
    b += big_tiles(c, thr);
  }
  if (threadIdx.x == blockDim.x - 1) {
    seg_start[E] = s_rows[blockDim.x - 1];
    tile_start[E] = s_tiles[blockDim.x - 1];
    tile_start_big[E] = s_big[blockDim.x - 1];
  }
}

// Single block of kRankChunk threads for R <= kRankChunk and E <= kMaxE: the
// ranks of rank_kernel's first block (slot s on thread s) and the scans of
// scan_kernel (expert e on thread e) over the counts in shared memory.  The
// one chunk's exclusive prefix is 0.
__global__ void __launch_bounds__(kRankChunk) permute_small_kernel(const int32_t* __restrict__ ids, int R, int E,
                                                                   int BN, int thr, int32_t* __restrict__ rank,
                                                                   int32_t* __restrict__ chunk_prefix,
                                                                   int32_t* __restrict__ counts,
                                                                   int32_t* __restrict__ seg_start,
                                                                   int32_t* __restrict__ tile_start,
                                                                   int32_t* __restrict__ tile_start_big,
                                                                   uint32_t* __restrict__ err) {
  static_assert(kRankChunk == 1024 && kMaxE <= kRankChunk, "one slot and one expert per thread, 32 warps");
  chain_wait();
  __shared__ int cnt[kMaxE];
  __shared__ int w_rows[32], w_tiles[32], w_big[32];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  // stable ranks: warps in order, lanes in order inside a warp
  const int s = threadIdx.x;
  int id = s < R ? ids[s] : -1;
  if (id >= E) {
    atomicOr(err, 2u);  // KMOE_DEVERR_BOUNDS: an expert id out of range (treated as masked)
    id = -1;
  }
  const bool valid = id >= 0;
  const unsigned peers = __match_any_sync(0xffffffffu, valid ? id : -1);
  const unsigned lower = peers & ((1u << lane) - 1u);
  int my = -1;
  const int nw = (R + 31) >> 5;  // warps that hold slots (the same bound for every thread)
  for (int w = 0; w < nw; ++w) {
    int base = 0;
    if (warp == w && valid) base = cnt[id];
    __syncwarp();
    if (warp == w && valid) {
      my = base + __popc(lower);
      if (lower == 0) cnt[id] = base + __popc(peers);
    }
    __syncthreads();
  }
  if (s < R) rank[s] = my;
  // exclusive prefixes of rows and tiles in expert order
  const int e = threadIdx.x;
  const int c = e < E ? cnt[e] : 0;
  const int t = small_tiles(c, BN, thr);
  const int tb = big_tiles(c, thr);
  if (e < E) {
    counts[e] = c;
    chunk_prefix[e] = 0;
  }
  int ir = c, it = t, ib = tb;  // inclusive within the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int vr = __shfl_up_sync(0xffffffffu, ir, off);
    const int vt = __shfl_up_sync(0xffffffffu, it, off);
    const int vb = __shfl_up_sync(0xffffffffu, ib, off);
    if (lane >= off) {
      ir += vr;
      it += vt;
      ib += vb;
    }
  }
  if (lane == 31) {
    w_rows[warp] = ir;
    w_tiles[warp] = it;
    w_big[warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    int wr = w_rows[lane], wt = w_tiles[lane], wb = w_big[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int vr = __shfl_up_sync(0xffffffffu, wr, off);
      const int vt = __shfl_up_sync(0xffffffffu, wt, off);
      const int vb = __shfl_up_sync(0xffffffffu, wb, off);
      if (lane >= off) {
        wr += vr;
        wt += vt;
        wb += vb;
      }
    }
    w_rows[lane] = wr;  // inclusive over warps
    w_tiles[lane] = wt;
    w_big[lane] = wb;
  }
  __syncthreads();
  if (e < E) {
    seg_start[e] = (warp > 0 ? w_rows[warp - 1] : 0) + ir - c;
    tile_start[e] = (warp > 0 ? w_tiles[warp - 1] : 0) + it - t;
    tile_start_big[e] = (warp > 0 ? w_big[warp - 1] : 0) + ib - tb;
  }
  if (threadIdx.x == 0) {
    seg_start[E] = w_rows[31];
    tile_start[E] = w_tiles[31];
    tile_start_big[E] = w_big[31];
  }
}

cudaError_t launch_permute(const int32_t* ids, int R, int E, int BN, int thr, int32_t* rank, int32_t* chunk_prefix,
                           int32_t* counts, int32_t* seg_start, int32_t* tile_start, int32_t* tile_start_big,
                           uint32_t* err, cudaStream_t st, bool pdl) {
  const int nchunk = (R + kRankChunk - 1) / kRankChunk;
  if (nchunk <= 1)
    return launch_chained(permute_small_kernel, dim3(1), dim3(kRankChunk), 0, st, pdl, ids, R, E, BN, thr, rank,
                          chunk_prefix, counts, seg_start, tile_start, tile_start_big, err);
  const cudaError_t e = launch_chained(rank_kernel, dim3(nchunk), dim3(kRankChunk), E * sizeof(int), st, pdl, ids, R,
                                       E, rank, chunk_prefix, err);
  if (e != cudaSuccess) return e;
  return launch_chained(scan_kernel, dim3(1), dim3(1024), 0, st, pdl, chunk_prefix, nchunk, E, BN, thr, counts,
                        seg_start, tile_start, tile_start_big);
}

}  // namespace kmoe
