// C-ABI entry points of libkmoe (declared and documented in include/kmoe.h):
// argument checks, the workspace layout, TMA tensor-map construction and the
// stream-ordered launch sequence of the forward.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "gemm.cuh"
#include "router.cuh"

namespace kmoe {
cudaError_t launch_route(const float*, const float*, int, int, int, int32_t*, float*, cudaStream_t);
cudaError_t launch_permute(const int32_t*, int, int, int, int, int32_t*, int32_t*, int32_t*, int32_t*, int32_t*,
                           int32_t*, uint32_t*, cudaStream_t, bool);
cudaError_t launch_quant_rows(const void*, int, int, int, uint8_t*, uint8_t*, cudaStream_t);
cudaError_t launch_quant_scatter(const void*, int, int, int, int, int, int, const int32_t*, const int32_t*,
                                 const int32_t*, const int32_t*, const int32_t*, const int32_t*, const int32_t*,
                                 int32_t*, int32_t*, uint8_t*, uint8_t*, uint8_t*, cudaStream_t, bool);
cudaError_t launch_combine(const float*, const int32_t*, const float*, int, int, int, int, float, void*,
                           cudaStream_t, bool);
cudaError_t launch_wait_selftest(uint32_t* err, uint64_t budget_ns, cudaStream_t st);
cudaError_t launch_activation_selftest(const float*, const float*, int, int, float, float, float, float, float, float,
                                       float*, cudaStream_t);
cudaError_t launch_mma_peak(int iters, int N, int grid, uint32_t* err, cudaStream_t st);
__global__ void kmoe_probe_kernel();
}  // namespace kmoe

using namespace kmoe;

namespace {

constexpr unsigned long long kWaitBudgetNs = 2000000000ull;  // 2 s per device-side wait

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D tensor map over [rows, cols] elements with row stride `stride_bytes`.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
              uint64_t stride_bytes, uint32_t box_cols, uint32_t box_rows, bool swizzle128 = true) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[2] = {cols, rows};
  cuuint64_t gstr[1] = {stride_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), gdim, gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over the code region of prepared weights: [nblk][128 rows][128
// E2M1 codes] (64 bytes per row, 8192 per block); a box holds `depth`
// consecutive blocks (K blocks of one weight tile).
bool make_weight_map(CUtensorMap* m, const void* base, uint64_t nblk, uint32_t depth) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3] = {128, 128, nblk};
  cuuint64_t gstr[2] = {64, 8192};
  cuuint32_t box[3] = {128, 128, depth};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), gdim, gstr, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t weight_blocks(const kmoe_params* p, int which) {
  if (which == 0) return static_cast<size_t>(p->E) * (p->I / 64) * (p->H / 128);
  return static_cast<size_t>(p->E) * (p->H / 128) * (p->I / 128);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_params(const kmoe_params* p) {
  if (!p) return KMOE_ERR_ARG;
  if (p->T < 0 || p->H <= 0 || p->I <= 0 || p->E <= 0 || p->k <= 0) return KMOE_ERR_ARG;
  if ((p->flags & ~KMOE_FLAG_SWIGLU) != 0u) return KMOE_ERR_ARG;
  if (p->flags & KMOE_FLAG_SWIGLU) {
    // finite parameters and a positive clamp
    if (!std::isfinite(p->swiglu_alpha) || !std::isfinite(p->swiglu_beta) || !std::isfinite(p->swiglu_limit) ||
        !(p->swiglu_limit > 0.f))
      return KMOE_ERR_ARG;
  } else if (!(p->situ_beta > 0.f) || !(p->situ_linear_beta > 0.f) || !std::isfinite(p->situ_beta) ||
             !std::isfinite(p->situ_linear_beta)) {
    return KMOE_ERR_ARG;
  }
  if (p->E > kMaxE || p->k > p->E || p->k > kMaxK) return KMOE_ERR_ARG;
  if (p->H % 128 != 0 || p->I % 128 != 0) return KMOE_ERR_SHAPE;
  // row indices of the weight tensor maps stay within int range
  if (static_cast<long long>(p->E) * 2 * p->I >= (1LL << 31) || static_cast<long long>(p->E) * p->H >= (1LL << 31))
    return KMOE_ERR_SHAPE;
  if (static_cast<long long>(p->T) * p->k >= (1LL << 31)) return KMOE_ERR_SHAPE;
  return KMOE_OK;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Tensor maps and launch of the fused router (router.cu) over caller memory.
int run_router(const void* x_bf16, const void* w_gate_bf16, const float* bias, int T, int H, int E, int k,
               float* logits, float* part, int32_t* ids, float* wts, int* sync, uint32_t* err, cudaStream_t stream) {
  RouterArgs a{};
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = k;
  a.xrows = T <= 32 ? 32 : (T <= 64 ? 64 : 128);
  a.plan = plan_router(T, H, E);
  a.bias = bias;
  a.logits = logits;
  a.part = part;
  a.ids = ids;
  a.wts = wts;
  a.sync = sync;
  a.err = err;
  a.budget_ns = kWaitBudgetNs;
  RouterMaps m;
  if (!make_map(&m.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x_bf16, H, T, static_cast<uint64_t>(H) * 2, 64,
                static_cast<uint32_t>(a.xrows)) ||
      !make_map(&m.g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_gate_bf16, H, E, static_cast<uint64_t>(H) * 2, 64,
                static_cast<uint32_t>(a.plan.pair ? a.plan.EN / 2 : a.plan.EN)))
    return KMOE_ERR_CUDA;
  const int sms = num_sms();
  if (sms <= 0) return KMOE_ERR_CUDA;
  return launch_router(m, a, sms, stream) == cudaSuccess ? KMOE_OK : KMOE_ERR_CUDA;
}

// Shape and pointer checks of the fused router's inputs.
int check_router_args(const void* x_bf16, const void* w_gate_bf16, const float* bias, int T, int H, int E, int k) {
  if (T < 0 || H <= 0 || E <= 0 || E > kMaxE || k <= 0 || k > E || k > kMaxK) return KMOE_ERR_ARG;
  if (H % 64 != 0 || E % 4 != 0) return KMOE_ERR_SHAPE;
  if (T > 0 && (!x_bf16 || !w_gate_bf16 || !bias)) return KMOE_ERR_ARG;
  if (T > 0 && (!aligned(x_bf16, 16) || !aligned(w_gate_bf16, 16))) return KMOE_ERR_ALIGN;
  return KMOE_OK;
}

#define KMOE_CK(call)                           \
  do {                                          \
    if ((call) != cudaSuccess) return KMOE_ERR_CUDA; \
  } while (0)

}  // namespace

extern "C" {

const char* kmoe_status_string(int s) {
  switch (s) {
    case KMOE_OK: return "ok";
    case KMOE_ERR_ARG: return "invalid argument";
    case KMOE_ERR_SHAPE: return "unsupported shape (H and I must be multiples of 128; FC1 rows = 2 x FC2 K)";
    case KMOE_ERR_ALIGN: return "misaligned pointer";
    case KMOE_ERR_ARCH: return "device is not compute capability 10.3 (GB300) or the kernels do not load";
    case KMOE_ERR_WORKSPACE: return "workspace missing or too small";
    case KMOE_ERR_CUDA: return "CUDA call failed";
    case KMOE_ERR_TIMEOUT: return "a device-side wait timed out";
    case KMOE_ERR_DEVICE: return "device-side error (expert id out of range)";
    default: return "unknown status";
  }
}

int kmoe_check_device(int device) {
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return KMOE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return KMOE_ERR_ARCH;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return KMOE_ERR_CUDA;
  if (cur != device && cudaSetDevice(device) != cudaSuccess) return KMOE_ERR_CUDA;
  cudaFuncAttributes fa;
  const cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kmoe_probe_kernel));
  if (cur != device) cudaSetDevice(cur);
  if (e != cudaSuccess) return KMOE_ERR_ARCH;
  if (!encode_fn()) return KMOE_ERR_CUDA;
  return KMOE_OK;
}

size_t kmoe_workspace_size(const kmoe_params* p) {
  if (check_params(p) != KMOE_OK) return 0;
  Layout L;
  if (!make_layout(*p, L)) return 0;
  return L.total;
}

int kmoe_workspace_layout(const kmoe_params* p, kmoe_ws_layout* out) {
  int st = check_params(p);
  if (st != KMOE_OK) return st;
  if (!out) return KMOE_ERR_ARG;
  Layout L;
  if (!make_layout(*p, L)) return KMOE_ERR_ARG;
  out->err = L.err;
  out->topk_ids = L.topk_ids;
  out->topk_w = L.topk_w;
  out->counts = L.counts;
  out->seg_start = L.seg_start;
  out->tile_start = L.tile_start;
  out->row_of_slot = L.row_of_slot;
  out->slot_of_row = L.slot_of_row;
  out->xq = L.xq;
  out->xsf = L.xsf;
  out->iq = L.iq;
  out->isf = L.isf;
  out->y = L.y;
  out->tile_rows = L.BN;
  out->max_tiles = L.max_tiles;
  out->total = L.total;
  out->logits = L.logits;
  out->tile_start_big = L.tile_start_big;
  out->xsf_big = L.xsf_big;
  out->isf_big = L.isf_big;
  out->tile_rows_big = L.big ? kBigTileRows : 0;
  out->max_tiles_big = L.max_tiles_big;
  out->big_rows = kBigRows;
  return KMOE_OK;
}

size_t kmoe_tile_sf_offset(int tile, int local_row, int g, int tile_rows, int K, int max_tiles) {
  (void)max_tiles;
  return tile_sf_offset(tile, local_row, g, (tile_rows + 127) / 128, K / 128);
}

int kmoe_route(const float* logits, const float* bias, int T, int E, int k, int32_t* topk_ids, float* topk_w,
               cudaStream_t stream) {
  if (T < 0 || E <= 0 || E > kMaxE || k <= 0 || k > E || k > kMaxK) return KMOE_ERR_ARG;
  if (T > 0 && (!logits || !bias || !topk_ids || !topk_w)) return KMOE_ERR_ARG;
  KMOE_CK(launch_route(logits, bias, T, E, k, topk_ids, topk_w, stream));
  return KMOE_OK;
}

int kmoe_quantize_mx(const void* x_bf16, int rows, int cols, int fmt, uint8_t* codes, uint8_t* scales,
                     cudaStream_t stream) {
  if (rows < 0 || cols <= 0) return KMOE_ERR_ARG;
  if (fmt != KMOE_MXFP8_E4M3 && fmt != KMOE_MXFP4_E2M1) return KMOE_ERR_ARG;
  if (cols % 128 != 0) return KMOE_ERR_SHAPE;
  if (rows == 0) return KMOE_OK;
  if (!x_bf16 || !codes || !scales) return KMOE_ERR_ARG;
  if (!aligned(x_bf16, 16) || !aligned(codes, 16)) return KMOE_ERR_ALIGN;
  KMOE_CK(launch_quant_rows(x_bf16, rows, cols, fmt, codes, scales, stream));
  return KMOE_OK;
}

size_t kmoe_prepared_weight_bytes(const kmoe_params* p, int which) {
  if (check_params(p) != KMOE_OK || (which != 0 && which != 1)) return 0;
  return weight_blocks(p, which) * kWeightBlockBytes;
}

int kmoe_prepare_weights(const kmoe_params* p, const uint8_t* w13, const uint8_t* w13_sf, const uint8_t* w2,
                         const uint8_t* w2_sf, uint8_t* w13_k, uint8_t* w2_k, cudaStream_t stream) {
  int st = check_params(p);
  if (st != KMOE_OK) return st;
  if (!w13 || !w13_sf || !w2 || !w2_sf || !w13_k || !w2_k) return KMOE_ERR_ARG;
  if (!aligned(w13, 16) || !aligned(w2, 16) || !aligned(w13_k, 256) || !aligned(w2_k, 256)) return KMOE_ERR_ALIGN;
  KMOE_CK(launch_prep_weights(w13, w13_sf, w13_k, p->E, p->I / 64, p->H / 128, 2 * p->I, p->H, 1, p->I, stream));
  KMOE_CK(launch_prep_weights(w2, w2_sf, w2_k, p->E, p->H / 128, p->I / 128, p->H, p->I, 0, p->I, stream));
  return KMOE_OK;
}

int kmoe_forward(const kmoe_params* p, const void* x_bf16, const float* logits, const float* bias,
                 const uint8_t* w13_k, const uint8_t* w2_k, const int32_t* topk_ids, const float* topk_w,
                 void* out_bf16, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return kmoe_forward_ex(p, x_bf16, logits, bias, w13_k, w2_k, topk_ids, topk_w, out_bf16, workspace, ws_bytes,
                         stream, nullptr);
}

// The forward; routing from given ids/weights, from logits, or (w_gate set)
// by the fused router from x and the gate weight.
static int forward_impl(const kmoe_params* p, const void* x_bf16, const float* logits, const void* w_gate,
                        const float* bias, const uint8_t* w13_k, const uint8_t* w2_k, const int32_t* topk_ids,
                        const float* topk_w, void* out_bf16, void* workspace, size_t ws_bytes, cudaStream_t stream,
                        const kmoe_stage_events* ev) {
  int st = check_params(p);
  if (st != KMOE_OK) return st;
  Layout L;
  if (!make_layout(*p, L)) return KMOE_ERR_ARG;
  if (w_gate) {
    st = check_router_args(x_bf16, w_gate, bias, p->T, p->H, p->E, p->k);
    if (st != KMOE_OK) return st;
  }
  if (!workspace || ws_bytes < L.total) return KMOE_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KMOE_ERR_ALIGN;
  if (p->T == 0) return KMOE_OK;
  const bool given = topk_ids != nullptr;
  if ((topk_ids == nullptr) != (topk_w == nullptr)) return KMOE_ERR_ARG;
  if (!x_bf16 || !w13_k || !w2_k || !out_bf16) return KMOE_ERR_ARG;
  if (!given && !w_gate && (!logits || !bias)) return KMOE_ERR_ARG;
  if (!aligned(x_bf16, 16) || !aligned(out_bf16, 16) || !aligned(w13_k, 256) || !aligned(w2_k, 256))
    return KMOE_ERR_ALIGN;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws + L.err);
  int32_t* ids = reinterpret_cast<int32_t*>(ws + L.topk_ids);
  float* wts = reinterpret_cast<float*>(ws + L.topk_w);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  int32_t* seg_start = reinterpret_cast<int32_t*>(ws + L.seg_start);
  int32_t* tile_start = reinterpret_cast<int32_t*>(ws + L.tile_start);
  int32_t* chunk_prefix = reinterpret_cast<int32_t*>(ws + L.chunk_prefix);
  int32_t* rank = reinterpret_cast<int32_t*>(ws + L.rank);
  int32_t* row_of_slot = reinterpret_cast<int32_t*>(ws + L.row_of_slot);
  int32_t* slot_of_row = reinterpret_cast<int32_t*>(ws + L.slot_of_row);
  uint8_t* xq = ws + L.xq;
  uint8_t* xsf = ws + L.xsf;
  uint8_t* iq = ws + L.iq;
  uint8_t* isf = ws + L.isf;
  float* y = reinterpret_cast<float*>(ws + L.y);
  const int T = p->T, H = p->H, I = p->I, E = p->E, k = p->k, R = L.R;

  int32_t* tile_start_big = reinterpret_cast<int32_t*>(ws + L.tile_start_big);
  uint8_t* xsf_big = ws + L.xsf_big;
  uint8_t* isf_big = ws + L.isf_big;
  // experts with more rows than `thr` take the big tiles (none when no expert can)
  const int thr = L.big ? kBigRows : 0x7fffffff;

  // Tensor maps of one tile class: weights as E2M1 (unpacked to 16-byte
  // aligned groups in smem), token rows as bytes in boxes of 32, 64, 128, a
  // tile and half a tile of rows, and (CTA-pair kernel) the weight and token
  // scale regions as rows of 128 bytes.
  auto class_maps = [&](GemmMaps& m, const uint8_t* w_k, int which, int kps, const uint8_t* act, int K,
                        const uint8_t* sf, int bn, int max_tiles) -> bool {
    const int nch = (bn + 127) / 128;
    const uint64_t nblk = weight_blocks(p, which);
    if (!make_weight_map(&m.a, w_k, nblk, kps)) return false;
    if (!make_map(&m.asf, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_k + nblk * 8192, 128, nblk * 4, 128, 128, 4, false))
      return false;
    const uint64_t sf_rows = static_cast<uint64_t>(K / 128) * (max_tiles > 0 ? max_tiles : 1) * nch * 4;
    if (!make_map(&m.bsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, sf, 128, sf_rows, 128, 128, 4 * nch, false)) return false;
    for (int i = 0; i < 5; ++i) {
      const uint32_t rows = i < 3 ? (32u << i) : static_cast<uint32_t>(i == 3 ? bn : bn / 2);
      if (!make_map(&m.b[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, act, K, R, K, 128, rows)) return false;
    }
    return true;
  };
  const int kps1 = gemm_kblocks_per_stage(L.BN, H / 128);
  const int kps2 = gemm_kblocks_per_stage(L.BN, I / 128);
  const int kpsb1 = gemm_kblocks_per_stage(kBigTileRows, H / 128);
  const int kpsb2 = gemm_kblocks_per_stage(kBigTileRows, I / 128);
  GemmMaps m1, m2, mb1, mb2;
  if (!class_maps(m1, w13_k, 0, kps1, xq, H, xsf, L.BN, L.max_tiles) ||
      !class_maps(m2, w2_k, 1, kps2, iq, I, isf, L.BN, L.max_tiles))
    return KMOE_ERR_CUDA;
  if (L.big && (!class_maps(mb1, w13_k, 0, kpsb1, xq, H, xsf_big, kBigTileRows, L.max_tiles_big) ||
                !class_maps(mb2, w2_k, 1, kpsb2, iq, I, isf_big, kBigTileRows, L.max_tiles_big)))
    return KMOE_ERR_CUDA;

  auto mark = [&](cudaEvent_t e) { return (ev && e) ? cudaEventRecord(e, stream) : cudaSuccess; };
  KMOE_CK(mark(ev ? ev->start : nullptr));
  // the error word reports this call only; words 2 and 3 are the FC1 / FC2 work-item counters
  KMOE_CK(cudaMemsetAsync(err, 0, 16, stream));
  if (given) {
    KMOE_CK(cudaMemcpyAsync(ids, topk_ids, static_cast<size_t>(R) * 4, cudaMemcpyDeviceToDevice, stream));
    KMOE_CK(cudaMemcpyAsync(wts, topk_w, static_cast<size_t>(R) * 4, cudaMemcpyDeviceToDevice, stream));
  } else if (w_gate) {
    st = run_router(x_bf16, w_gate, bias, T, H, E, k, reinterpret_cast<float*>(ws + L.logits),
                    reinterpret_cast<float*>(ws + L.router_part), ids, wts,
                    reinterpret_cast<int*>(ws + L.router_sync), err, stream);
    if (st != KMOE_OK) return st;
  } else {
    KMOE_CK(launch_route(logits, bias, T, E, k, ids, wts, stream));
  }
  KMOE_CK(mark(ev ? ev->routed : nullptr));
  // Kernels after the first are chained (launch_chained): each may begin
  // launching while its predecessor runs (also inside a captured graph,
  // where the T=16 layer replays in 857 us chained, 860 us not).  Not across
  // stage events (their records sit between the kernels), nor after the copy
  // of given ids.
  const bool pdl = ev == nullptr;
  KMOE_CK(launch_permute(ids, R, E, L.BN, thr, rank, chunk_prefix, counts, seg_start, tile_start, tile_start_big, err,
                         stream, pdl && !given));
  KMOE_CK(mark(ev ? ev->permuted : nullptr));
  KMOE_CK(launch_quant_scatter(x_bf16, T, H, k, E, L.BN, thr, ids, rank, chunk_prefix, counts, seg_start, tile_start,
                               tile_start_big, row_of_slot, slot_of_row, xq, xsf, xsf_big, stream, pdl));
  KMOE_CK(mark(ev ? ev->quantized : nullptr));
  const int grid = num_sms();
  if (grid <= 0) return KMOE_ERR_CUDA;
  // FC1 and FC2 each run the big-tile experts (CTA pairs) and then the
  // small-tile experts; the two launches cover disjoint experts and rows
  GemmArgs a1{counts, seg_start, tile_start, w13_k, w13_k + weight_blocks(p, 0) * 8192, xsf, E, I / 64, H / 128,
              L.max_tiles, H, I, iq, isf, static_cast<float>(2.0 / p->situ_beta),
              static_cast<float>(2.0 / p->situ_linear_beta),
              static_cast<float>(static_cast<double>(p->situ_beta) * p->situ_linear_beta), nullptr, slot_of_row,
              err, kWaitBudgetNs, reinterpret_cast<int*>(err) + 2,
              (p->flags & KMOE_FLAG_SWIGLU) ? 1 : 0, p->swiglu_alpha, p->swiglu_beta, p->swiglu_limit};
  if (L.big) {
    GemmArgs ab1 = a1;
    ab1.tile_start = tile_start_big;
    ab1.bsf = xsf_big;
    ab1.isf = isf_big;
    ab1.max_tiles = L.max_tiles_big;
    KMOE_CK(launch_moe_gemm(true, kBigTileRows, kpsb1, mb1, ab1, grid, stream, pdl));
  }
  KMOE_CK(launch_moe_gemm(true, L.BN, kps1, m1, a1, grid, stream, pdl));
  KMOE_CK(mark(ev ? ev->fc1 : nullptr));
  GemmArgs a2{counts, seg_start, tile_start, w2_k, w2_k + weight_blocks(p, 1) * 8192, isf, E, H / 128, I / 128,
              L.max_tiles, H, I, nullptr, nullptr, 0.f, 0.f, 0.f, y, slot_of_row, err, kWaitBudgetNs,
              reinterpret_cast<int*>(err) + 3, 0, 0.f, 0.f, 0.f};
  if (L.big) {
    GemmArgs ab2 = a2;
    ab2.tile_start = tile_start_big;
    ab2.bsf = isf_big;
    ab2.max_tiles = L.max_tiles_big;
    KMOE_CK(launch_moe_gemm(false, kBigTileRows, kpsb2, mb2, ab2, grid, stream, pdl));
  }
  KMOE_CK(launch_moe_gemm(false, L.BN, kps2, m2, a2, grid, stream, pdl));
  KMOE_CK(mark(ev ? ev->fc2 : nullptr));
  KMOE_CK(launch_combine(y, ids, wts, T, H, k, E, p->routed_scaling_factor, out_bf16, stream, pdl));
  KMOE_CK(mark(ev ? ev->combined : nullptr));
  return KMOE_OK;
}

int kmoe_forward_ex(const kmoe_params* p, const void* x_bf16, const float* logits, const float* bias,
                    const uint8_t* w13_k, const uint8_t* w2_k, const int32_t* topk_ids, const float* topk_w,
                    void* out_bf16, void* workspace, size_t ws_bytes, cudaStream_t stream,
                    const kmoe_stage_events* ev) {
  return forward_impl(p, x_bf16, logits, nullptr, bias, w13_k, w2_k, topk_ids, topk_w, out_bf16, workspace, ws_bytes,
                      stream, ev);
}

int kmoe_forward_router(const kmoe_params* p, const void* x_bf16, const void* w_gate_bf16, const float* bias,
                        const uint8_t* w13_k, const uint8_t* w2_k, void* out_bf16, void* workspace, size_t ws_bytes,
                        cudaStream_t stream, const kmoe_stage_events* ev) {
  if (!w_gate_bf16) return KMOE_ERR_ARG;
  return forward_impl(p, x_bf16, nullptr, w_gate_bf16, bias, w13_k, w2_k, nullptr, nullptr, out_bf16, workspace,
                      ws_bytes, stream, ev);
}

size_t kmoe_router_workspace_size(int T, int H, int E) {
  if (T < 0 || H <= 0 || H % 64 != 0 || E <= 0 || E > kMaxE) return 0;
  const RouterPlan rp = plan_router(T, H, E);
  return 256 + align_up(router_sync_bytes(rp), 256) + align_up(router_part_bytes(rp, T, E), 256);
}

int kmoe_router(const void* x_bf16, const void* w_gate_bf16, const float* bias, int T, int H, int E, int k,
                float* logits, int32_t* topk_ids, float* topk_w, void* workspace, size_t ws_bytes,
                cudaStream_t stream) {
  int st = check_router_args(x_bf16, w_gate_bf16, bias, T, H, E, k);
  if (st != KMOE_OK) return st;
  if (!workspace || ws_bytes < kmoe_router_workspace_size(T, H, E)) return KMOE_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KMOE_ERR_ALIGN;
  if (T == 0) return KMOE_OK;
  if (!logits || !topk_ids || !topk_w) return KMOE_ERR_ARG;
  if (!aligned(logits, 16)) return KMOE_ERR_ALIGN;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  KMOE_CK(cudaMemsetAsync(err, 0, 16, stream));
  const RouterPlan rp = plan_router(T, H, E);
  float* part = reinterpret_cast<float*>(ws + 256 + align_up(router_sync_bytes(rp), 256));
  return run_router(x_bf16, w_gate_bf16, bias, T, H, E, k, logits, part, topk_ids, topk_w,
                    reinterpret_cast<int*>(ws + 256), err, stream);
}

int kmoe_device_error(void* workspace, uint32_t* word, cudaStream_t stream) {
  if (!workspace) return KMOE_ERR_ARG;
  uint32_t v = 0;
  uint32_t* dev = static_cast<uint32_t*>(workspace);  // the error word is at offset 0
  KMOE_CK(cudaMemcpyAsync(&v, dev, 4, cudaMemcpyDeviceToHost, stream));
  KMOE_CK(cudaStreamSynchronize(stream));
  KMOE_CK(cudaMemsetAsync(dev, 0, 4, stream));
  KMOE_CK(cudaStreamSynchronize(stream));
  if (word) *word = v;
  if (v & KMOE_DEVERR_TIMEOUT) return KMOE_ERR_TIMEOUT;
  if (v) return KMOE_ERR_DEVICE;
  return KMOE_OK;
}

int kmoe_mma_peak_run(int iters, int N, void* workspace, cudaStream_t stream) {
  if (!workspace || iters < 1 || iters > (1 << 24) || N < 16 || N > 256 || N % 16 != 0) return KMOE_ERR_ARG;
  const int grid = num_sms();
  if (grid <= 0) return KMOE_ERR_CUDA;
  KMOE_CK(launch_mma_peak(iters, N, grid, static_cast<uint32_t*>(workspace), stream));
  return KMOE_OK;
}

int kmoe_selftest_wait_timeout(void* workspace, int budget_us, cudaStream_t stream) {
  if (!workspace || budget_us <= 0 || budget_us > 1000000) return KMOE_ERR_ARG;
  KMOE_CK(launch_wait_selftest(static_cast<uint32_t*>(workspace), static_cast<uint64_t>(budget_us) * 1000ull,
                               stream));
  return KMOE_OK;
}

int kmoe_selftest_activation(const kmoe_params* p, const float* gate, const float* up, int n, float* out,
                             cudaStream_t stream) {
  if (!p) return KMOE_ERR_ARG;
  kmoe_params q = *p;  // only the activation fields matter here
  q.T = 0;
  q.H = q.I = 128;
  q.E = q.k = 1;
  const int st = check_params(&q);
  if (st != KMOE_OK) return st;
  if (n < 0) return KMOE_ERR_ARG;
  if (n > 0 && (!gate || !up || !out)) return KMOE_ERR_ARG;
  const bool swiglu = (p->flags & KMOE_FLAG_SWIGLU) != 0u;
  KMOE_CK(launch_activation_selftest(gate, up, n, swiglu ? 1 : 0, static_cast<float>(2.0 / p->situ_beta),
                                     static_cast<float>(2.0 / p->situ_linear_beta),
                                     static_cast<float>(static_cast<double>(p->situ_beta) * p->situ_linear_beta),
                                     p->swiglu_alpha, p->swiglu_beta, p->swiglu_limit, out, stream));
  return KMOE_OK;
}

}  // extern "C"
