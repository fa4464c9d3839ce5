// Shared definitions of the kmoe kernels: status handling, the workspace
// layout, the token-tile scale layout and small numeric helpers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/kmoe.h"
#include "ptx.cuh"

namespace kmoe {

constexpr int kRankChunk = 1024;  // slots per block in the stable rank pass
constexpr int kMaxE = 1024;       // experts supported by the routing kernel
constexpr int kMaxK = 32;
constexpr int kMaxDevices = 64;   // devices whose per-device launch state the library keeps

// The current device's ordinal, or -1 if it cannot be read or is not below
// kMaxDevices (launch state such as a kernel's shared-memory attribute or its
// co-resident cluster count is kept per device).
__host__ inline int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

// ---------------------------------------------------------------- launch chaining
// The forward's kernels run back to back on one stream.  Each is launched
// with programmatic stream serialization (pdl): it may start launching while
// its predecessor still runs, so its CTAs are resident when the predecessor
// ends.  Every kernel of the chain first waits until its predecessor grid has
// completed and its memory is visible (griddepcontrol.wait returns at once
// for a launch without that dependency), and only then lets its own
// successor begin launching.  Nothing a kernel does precedes the wait, so the
// stream order of every memory access is unchanged, and each grid completes
// only after its predecessor: the order is transitive through the chain.
__device__ __forceinline__ void chain_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
__host__ inline cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                           cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------- tile layout
// Scales of the B operand (token rows) are stored per token tile so that a
// tile's scales for one 128-wide K block form whole 512-byte blocks that
// tcgen05.cp copies into TMEM at a 4-aligned column, and the blocks of
// consecutive K blocks of one tile are contiguous (one copy per stage):
//   block (tile, kb, chunk) = 512 bytes, chunk = local_row / 128,
//   byte j*16 + c*4 + g%4 holds row 32c + j (of the chunk) for K group g.
__host__ __device__ __forceinline__ size_t tile_sf_offset(int tile, int local_row, int g, int nch, int KB) {
  const int kb = g >> 2;
  const int chunk = local_row >> 7;
  const int r = local_row & 127;
  return ((static_cast<size_t>(tile) * KB + kb) * nch + chunk) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (g & 3);
}

// ---------------------------------------------------------------- fused router plan
// Work decomposition of the gate GEMM (router.cu): token tiles of 128 rows
// (the MMA's M) times expert chunks of EN columns (the MMA's N), optionally
// times S splits of K (= H) when there are too few items to occupy the SMs;
// the last split of a (tile, chunk) to finish sums the S partial tiles in
// split order.  The plan depends on the shape only (never on the device), so
// the logits' rounding is the same on every GPU.
struct RouterPlan {
  int EN;     // experts per item, a multiple of 32 in [32, 256]
  int nch;    // expert chunks: ceil(E / EN)
  int tiles;  // token tiles: ceil(T / 128)
  int S;      // K splits
  int kper;   // 64-wide K steps per split (the last split may have fewer)
  int items;  // tiles * nch * S; CTA pairs: ceil(tiles / 2) * nch
  int pair;   // 1: items run on CTA pairs (two token tiles, M = 256, EN / 2 gate rows per CTA)
};

// Estimated cycles of one 64-wide K step of an item: the larger of its loads
// (bytes per SM at ~49 B per cycle, the bytes in flight over the load latency)
// and its 4 MMAs (EN / 2 cycles each, at least ~54).
__host__ inline long long router_step_cycles(int EN, bool pair) {
  const long long bytes = 16384 + (pair ? 64LL : 128LL) * EN;
  const long long load = bytes / 49;
  const long long mma = 4LL * (EN / 2 > 54 ? EN / 2 : 54);
  return load > mma ? load : mma;
}

// One CTA per item: EN minimises (rounds of items over 152 SMs) x (MMA time
// per K step, proportional to EN above ~112 columns, flat below); ties go to
// the smaller EN (more SMs streaming the gate weight).  Fewer than 76 items:
// K is split so that about 152 items run, each with at least 8 K steps.
// Enough token tiles: CTA pairs if the step estimate favours them.
__host__ inline RouterPlan plan_router(int T, int H, int E) {
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
      best = RouterPlan{en, nch, tiles, 1, 0, static_cast<int>(items), 0};
    }
  }
  const int KS = H / 64;
  // CTA pairs: each SM moves its 128 token rows and half of the EN gate rows
  // per K step for the same MMA work; taken when the estimate is 10 % better
  if (tiles >= 2 && best.items >= kSlots / 2) {
    const long long single = ((best.items + kSlots - 1) / kSlots) * router_step_cycles(best.EN, false);
    const int tpairs = (tiles + 1) / 2;
    RouterPlan pb{};
    long long pcost = -1;
    for (int en = 32; en <= 256; en += 32) {
      const int nch = (E + en - 1) / en;
      const long long items = static_cast<long long>(tpairs) * nch;
      const long long cost = ((items + kSlots / 2 - 1) / (kSlots / 2)) * router_step_cycles(en, true);
      if (pcost < 0 || cost < pcost) {
        pcost = cost;
        pb = RouterPlan{en, nch, tiles, 1, KS, static_cast<int>(items), 1};
      }
    }
    if (10 * pcost < 9 * single) return pb;
  }
  const int base = best.items;
  int S = 1;
  if (base > 0 && base < kSlots / 2) {
    S = kSlots / base;
    const int smax = KS / 8 > 1 ? KS / 8 : 1;
    if (S > smax) S = smax;
  }
  best.kper = (KS + S - 1) / S;
  best.S = (KS + best.kper - 1) / best.kper;  // no empty split
  best.items = base * best.S;
  return best;
}

// Router counters: the routing warps' token counter, one completion counter
// per token tile, one split counter per (tile, chunk).
__host__ inline size_t router_sync_bytes(const RouterPlan& r) {
  return static_cast<size_t>(2 + r.tiles + r.tiles * r.nch) * 4;
}
__host__ inline size_t router_part_bytes(const RouterPlan& r, int T, int E) {
  return r.S > 1 ? static_cast<size_t>(r.S) * T * E * 4 : 0;
}

// ---------------------------------------------------------------- workspace
// Token tiles come in two classes, chosen per expert from its row count:
// experts with at most kBigRows rows are cut into small tiles of BN (32 or
// 64) rows, run by the one-CTA kernel (two CTAs per SM) that streams their
// weights at HBM speed; experts with more rows are cut into 224-row tiles,
// run by the CTA-pair kernel, where the tensor pipe is the limit.  Each class
// has its own tile numbering (tile_start / tile_start_big, prefixes over the
// experts in order) and its own token-tile scale arrays.
constexpr int kBigRows = 64;
constexpr int kBigTileRows = 224;

struct Layout {
  size_t err, topk_ids, topk_w, counts, seg_start, tile_start, chunk_prefix, rank, row_of_slot, slot_of_row;
  size_t xq, xsf, iq, isf, y, logits, router_sync, router_part, total;
  size_t tile_start_big, xsf_big, isf_big;
  int R, BN, nch, max_tiles, nchunk;
  int big;        // 1 if an expert can exceed kBigRows rows (T > kBigRows), else no big tiles
  int max_tiles_big;
};

// Small-tile size for a layer: 32 rows when few rows reach each expert on
// average (decode), else 64.
__host__ inline int choose_tile_rows(long long R, int E) {
  const double avg = static_cast<double>(R) / E;
  return avg <= 20.0 ? 32 : 64;
}

__host__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ inline bool make_layout(const kmoe_params& p, Layout& L) {
  if (p.T < 0 || p.H <= 0 || p.I <= 0 || p.E <= 0 || p.k <= 0) return false;
  const size_t R = static_cast<size_t>(p.T) * p.k;
  L.R = static_cast<int>(R);
  L.BN = choose_tile_rows(static_cast<long long>(R), p.E);
  L.nch = 1;
  // an expert has at most T rows (one per token)
  L.big = p.T > kBigRows ? 1 : 0;
  const size_t nE = static_cast<size_t>(p.E);
  const size_t small_cap = L.big ? nE * ((kBigRows + L.BN - 1) / L.BN) : (R + L.BN - 1) / L.BN + (R < nE ? R : nE);
  const size_t small_all = (R + L.BN - 1) / L.BN + (R < nE ? R : nE);
  L.max_tiles = static_cast<int>(small_cap < small_all ? small_cap : small_all);
  if (L.max_tiles < 1) L.max_tiles = 1;
  const size_t nbig = R / (kBigRows + 1) < nE ? R / (kBigRows + 1) : nE;  // experts with > kBigRows rows
  L.max_tiles_big = L.big ? static_cast<int>((R + kBigTileRows - 1) / kBigTileRows + nbig) : 0;
  L.nchunk = static_cast<int>((R + kRankChunk - 1) / kRankChunk);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + (bytes ? bytes : 1), 256);
    return o;
  };
  L.err = take(16);
  L.topk_ids = take(R * 4);
  L.topk_w = take(R * 4);
  L.counts = take(static_cast<size_t>(p.E) * 4);
  L.seg_start = take(static_cast<size_t>(p.E + 1) * 4);
  L.tile_start = take(static_cast<size_t>(p.E + 1) * 4);
  L.chunk_prefix = take(static_cast<size_t>(L.nchunk) * p.E * 4);
  L.rank = take(R * 4);
  L.row_of_slot = take(R * 4);
  L.slot_of_row = take(R * 4);
  L.xq = take(R * p.H);
  L.xsf = take(static_cast<size_t>(p.H / 128) * L.max_tiles * L.nch * 512);
  L.iq = take(R * p.I);
  L.isf = take(static_cast<size_t>(p.I / 128) * L.max_tiles * L.nch * 512);
  L.tile_start_big = take(static_cast<size_t>(p.E + 1) * 4);
  L.xsf_big = take(static_cast<size_t>(p.H / 128) * L.max_tiles_big * 2 * 512);
  L.isf_big = take(static_cast<size_t>(p.I / 128) * L.max_tiles_big * 2 * 512);
  L.y = take(R * p.H * 4);
  // the fused router's outputs and counters (token counter, one per 128-token tile)
  L.logits = take(static_cast<size_t>(p.T) * p.E * 4);
  const RouterPlan rp = plan_router(p.T, p.H, p.E);
  L.router_sync = take(router_sync_bytes(rp));
  L.router_part = take(router_part_bytes(rp, p.T, p.E));
  L.total = off;
  return true;
}

// ---------------------------------------------------------------- numerics
// 2^n as a float for n in [-127, 127] (exact).
__device__ __forceinline__ float exp2i(int n) {
  return n >= -126 ? __int_as_float((n + 127) << 23) : __int_as_float(0x00200000);
}

// Scale exponent of the microscaling rule: smallest e with amax <= qmax*2^e,
// clamped to [-127, 127], where qmax = 1.75 * 2^8 (E4M3) or 1.5 * 2^2 (E2M1).
// amax must be >= 0 (NaN already dropped).  Works on the fp32 bit pattern:
// amax = (1 + M/2^23) * 2^Ea, and the bound needs e = Ea - qexp (+1 when the
// significand exceeds qmax's).
template <int QEXP, uint32_t QMANT>
__device__ __forceinline__ int mx_scale_exp(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int ef = static_cast<int>((b >> 23) & 0xFF);
  if (ef == 0) return -127;             // zero or subnormal: far below any bound
  if (ef == 0xFF) return 127;           // inf
  const int ea = ef - 127;
  int e = ea - QEXP + ((b & 0x7FFFFF) > QMANT ? 1 : 0);
  e = e < -127 ? -127 : (e > 127 ? 127 : e);
  return e;
}
__device__ __forceinline__ int e4m3_scale_exp(float amax) { return mx_scale_exp<8, 0x600000u>(amax); }
__device__ __forceinline__ int e2m1_scale_exp(float amax) { return mx_scale_exp<2, 0x400000u>(amax); }

}  // namespace kmoe
