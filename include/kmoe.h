/*
 * kmoe -- Kimi-K3 routed-expert MoE forward (MXFP8 activations x MXFP4
 * weights, SiTU gated activation) for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument is a DEVICE pointer owned by the caller
 * unless its comment says "host".  The library never allocates device
 * memory and never synchronises the host inside these calls: work is
 * enqueued on the given stream and errors that only the device can see
 * (a bounded wait that gave up) are recorded in the workspace and read
 * back with kmoe_device_error().  Argument errors are reported before
 * anything is enqueued.  All calls are safe to capture in a CUDA graph
 * (fixed grids, device-side counts, no host reads of device data).
 * An empty batch (T = 0, or rows = 0 for kmoe_quantize_mx) is valid
 * everywhere: after the size checks the call returns KMOE_OK having
 * enqueued nothing, so the outputs and the workspace (its error word
 * included) keep their contents, and null data pointers are accepted.
 *
 * Layout conventions (all row-major, contiguous, no strides):
 *   bf16 activations x      [T, H]
 *   router logits           [T, E] float
 *   router (gate) weight    [E, H] bf16 (kmoe_router, kmoe_forward_router)
 *   correction bias         [E] float
 *   w13 codes               [E, 2I, H/2] uint8, two E2M1 codes per byte
 *                           (element 2j in the low nibble); rows [0, I) are
 *                           the gate projection, rows [I, 2I) the up
 *                           projection ("[gate; up]" halves)
 *   w13 scales (raw)        [E, 2I, H/32] uint8 UE8M0 (value 2^(b-127))
 *   w2 codes                [E, H, I/2] uint8
 *   w2 scales (raw)         [E, H, I/32] uint8
 *   output                  [T, H] bf16
 * Sources (web pages this library follows):
 *   - Kimi-K3 SM120 FlashInfer MXFP4 page: serving call chain (sigmoid +
 *     correction-bias top-16 with renormalised weights), real checkpoint
 *     contract (packed MXFP4, group-32 E8M0 scales, [gate; up] halves),
 *     the SiTU formula with situ_beta = 4 and situ_linear_beta = 25, the
 *     gated width rule (FC1 = 2 x FC2 K), the NaN/Inf decision record
 *     (saturating-finite MXFP8, no 0xFF scale), and the non-fused,
 *     deterministic finalize; the gate's logits that TopK consumes (the
 *     fused router) and the SwiGLU control group's parameters.
 *   - Kimi-K3 MoE path analysis page (SM100 section): MXFP8 pre-dispatch
 *     quantisation (per-32 absmax -> UE8M0 -> E4M3, four scale bytes per
 *     int32), weight/scale re-layout at load time for TMEM-staged scales,
 *     routed_scaling_factor.
 */
#ifndef KMOE_H_
#define KMOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (the only definition of these values). */
enum kmoe_status {
  KMOE_OK = 0,
  KMOE_ERR_ARG = 1,        /* null pointer, k > E, non-positive size, bad enum */
  KMOE_ERR_SHAPE = 2,      /* H or I not a multiple of 128, FC1 width != 2 x FC2 K, ... */
  KMOE_ERR_ALIGN = 3,      /* a pointer is not aligned as documented */
  KMOE_ERR_ARCH = 4,       /* device is not sm_103 (GB300) or the kernels do not load */
  KMOE_ERR_WORKSPACE = 5,  /* workspace null or smaller than kmoe_workspace_size() */
  KMOE_ERR_CUDA = 6,       /* a CUDA runtime/driver call failed */
  KMOE_ERR_TIMEOUT = 7,    /* a device-side bounded wait gave up (see kmoe_device_error) */
  KMOE_ERR_DEVICE = 8      /* other device-side error (e.g. an expert id >= E in the input) */
};

/* Quantisation formats for kmoe_quantize_mx. */
enum kmoe_mx_format {
  KMOE_MXFP8_E4M3 = 0,  /* one E4M3 code per byte */
  KMOE_MXFP4_E2M1 = 1   /* two E2M1 codes per byte, element 2j in the low nibble */
};

/* kmoe_params.flags: the FC1 activation is the clamped SwiGLU control
 * (SM120 page, activation table: the kernel the pages compare SiTU against)
 *   out = g' * sigmoid(alpha * g') * (u' + beta),  g' = min(g, limit),
 *   u' = clamp(u, -limit, limit),
 * with alpha, beta, limit = swiglu_alpha, swiglu_beta, swiglu_limit; without
 * the flag it is SiTU (situ_beta, situ_linear_beta). */
#define KMOE_FLAG_SWIGLU 1u

/* Layer parameters (host struct). */
typedef struct kmoe_params {
  int T;                        /* tokens, >= 0 */
  int H;                        /* hidden size, multiple of 128 */
  int I;                        /* expert intermediate size, multiple of 128 */
  int E;                        /* experts, 1..1024 */
  int k;                        /* experts per token, 1..min(E, 32) */
  float situ_beta;              /* SiTU gate beta (Kimi-K3: 4.0), > 0 */
  float situ_linear_beta;       /* SiTU linear beta (Kimi-K3: 25.0), > 0 */
  float routed_scaling_factor;  /* applied in the combine (1.0 in the workloads) */
  uint32_t flags;               /* 0 or KMOE_FLAG_SWIGLU */
  float swiglu_alpha;           /* SwiGLU control (1.702); used with KMOE_FLAG_SWIGLU */
  float swiglu_beta;            /* (1.0) */
  float swiglu_limit;           /* (7.0), > 0 */
} kmoe_params;

/* Human-readable name of a status code (static string). */
const char* kmoe_status_string(int status);

/* Checks that `device` is a GB300-class GPU (compute capability 10.3) and
 * that this library's kernels load on it.  Call once at initialisation;
 * returns KMOE_ERR_ARCH otherwise (fail at init, never at the first layer). */
int kmoe_check_device(int device);

/* Bytes of device workspace kmoe_forward needs for these parameters (0 on
 * invalid parameters). */
size_t kmoe_workspace_size(const kmoe_params* p);

/* Offsets (bytes from the workspace base) of the stage tensors kmoe_forward
 * leaves in the workspace, for inspection and tests.  Host struct. */
typedef struct kmoe_ws_layout {
  size_t err;          /* uint32 device error word (KMOE_DEVERR_* bits) */
  size_t topk_ids;     /* int32 [T, k] expert ids used (routed or given) */
  size_t topk_w;       /* float [T, k] routing weights used */
  size_t counts;       /* int32 [E] rows per expert */
  size_t seg_start;    /* int32 [E+1] first expert-sorted row of each expert */
  size_t tile_start;   /* int32 [E+1] first small tile of each expert (prefix over the small-tile experts) */
  size_t row_of_slot;  /* int32 [T*k] expert-sorted row of slot t*k+j (-1 if masked) */
  size_t slot_of_row;  /* int32 [R] slot t*k+j of each expert-sorted row */
  size_t xq;           /* uint8 [R, H] E4M3 codes of x, expert-sorted */
  size_t xsf;          /* uint8 tile-layout UE8M0 scales of xq (see kmoe_tile_sf_offset) */
  size_t iq;           /* uint8 [R, I] E4M3 codes of the FC1 activation, expert-sorted */
  size_t isf;          /* uint8 tile-layout UE8M0 scales of iq */
  size_t y;            /* float [T*k, H] per-slot FC2 outputs (slot order) */
  int tile_rows;       /* rows per small token tile (32 or 64) chosen for these parameters */
  int max_tiles;       /* capacity of the small-tile scale arrays (xsf, isf), in tiles */
  size_t total;        /* == kmoe_workspace_size(p) */
  size_t logits;       /* float [T, E] router logits (written by kmoe_forward_router) */
  /* Experts with more than big_rows rows are cut into tiles of tile_rows_big
   * rows with their own numbering and scale arrays; the others into small
   * tiles.  tile_rows_big is 0 when no expert can have more than big_rows
   * rows (T <= big_rows): every tile is then small. */
  size_t tile_start_big; /* int32 [E+1] first big tile of each expert (prefix over the big-tile experts) */
  size_t xsf_big;      /* uint8 tile-layout scales of xq rows in big tiles */
  size_t isf_big;      /* uint8 tile-layout scales of iq rows in big tiles */
  int tile_rows_big;   /* 224, or 0 (see above) */
  int max_tiles_big;   /* capacity of xsf_big / isf_big, in tiles */
  int big_rows;        /* row-count threshold of the big tiles */
} kmoe_ws_layout;
int kmoe_workspace_layout(const kmoe_params* p, kmoe_ws_layout* out /* host */);

/* Routing (Kimi-K3 TopK: sigmoid scores, e_score_correction_bias used only
 * to choose, weights gathered from the un-biased scores and renormalised).
 * key[e] = fp32(sigmoid(logit[e])) + bias[e] (one fp32 add; the sigmoid is
 * evaluated in double and rounded once); the k largest keys are chosen,
 * equal keys going to the lower expert index; slot j holds the j-th largest
 * key.  topk_w[t, j] = s_j / sum_j' s_j' (float, sums to 1).
 *   logits [T, E] float, bias [E] float, topk_ids [T, k] int32 (out),
 *   topk_w [T, k] float (out).  E <= 1024, k <= min(E, 32). */
int kmoe_route(const float* logits, const float* bias, int T, int E, int k, int32_t* topk_ids, float* topk_w,
               cudaStream_t stream);

/* The router (Kimi-K3 SM120 FlashInfer MXFP4 page, "Phase 1: serving call
 * chain": TopK consumes the gate's logits), fused: the gate GEMM
 *   logits[t, e] = sum_h x[t, h] * w_gate[e, h]
 * on the tensor cores (bf16 x bf16, fp32 accumulation; the summation order,
 * split K included, depends only on (T, H, E)), followed in the same kernel by the routing of
 * kmoe_route on those logits; tokens of finished 128-token tiles are routed
 * while the gate GEMM of later tiles runs.
 *   x [T, H] bf16 and w_gate [E, H] bf16 (both row-major, 16-byte aligned),
 *   bias [E] float; logits [T, E] float (out, 16-byte aligned), topk_ids
 *   [T, k] int32 (out), topk_w [T, k] float (out).  H a multiple of 64, E a
 *   multiple of 4 and <= 1024, k <= min(E, 32).
 *   workspace: device memory of kmoe_router_workspace_size(T, H, E) bytes
 *   (0 for invalid sizes), 256-byte aligned, caller-owned: counters and, when
 *   few token tiles leave SMs idle (decode), the partial sums of a split K;
 *   its first word is the device error word (read it with
 *   kmoe_device_error).  The call launches one CTA per SM (in clusters of
 *   two, M = 256 tensor-core pairs, when there are enough 128-token tiles) as
 *   a cooperative launch (all co-resident), so it fails with KMOE_ERR_CUDA if
 *   the device cannot host them all at once.  Every device wait is bounded;
 *   a token whose logits did not arrive in time is left masked (ids -1,
 *   weights 0) and the timeout bit is set. */
size_t kmoe_router_workspace_size(int T, int H, int E);
int kmoe_router(const void* x_bf16, const void* w_gate_bf16, const float* bias, int T, int H, int E, int k,
                float* logits, int32_t* topk_ids, float* topk_w, void* workspace, size_t ws_bytes,
                cudaStream_t stream);

/* Microscaling quantisation of bf16 rows, one UE8M0 scale per 32 columns
 * (Kimi-K3 MoE path analysis page, SM100 section, mega_moe_pre_dispatch:
 * bf16 -> per-32 absmax -> UE8M0 scale -> FP8 E4M3 codes, four scale bytes
 * per int32; the NaN/Inf handling follows the SM120 FlashInfer MXFP4 page's
 * NaN/Inf decision record: saturating-finite payload, no 0xFF scale byte).
 * Scale byte = e + 127 with e the smallest integer such that
 * amax <= qmax * 2^e (qmax = 448 for E4M3, 6 for E2M1), clamped to
 * [-127, 127]; NaN is ignored by the absmax; codes are round-to-nearest-even
 * of x * 2^-e, saturating to +-qmax; NaN elements become +0.  The scale row
 * is cols/32 bytes, i.e. cols/128 little-endian int32 words (four scale
 * bytes per int32).
 *   x [rows, cols] bf16, cols a multiple of 128;
 *   codes [rows, cols] (E4M3) or [rows, cols/2] (E2M1) uint8 (out);
 *   scales [rows, cols/32] uint8 (out).  x and codes 16-byte aligned. */
int kmoe_quantize_mx(const void* x_bf16, int rows, int cols, int fmt, uint8_t* codes, uint8_t* scales,
                     cudaStream_t stream);

/* Bytes of the prepared weights (which = 0: FC1 / w13, 1: FC2 / w2):
 * blocks of KMOE_WEIGHT_BLOCK_BYTES, one per (expert, 128-row weight tile,
 * 128-wide K block): E*(I/64)*(H/128) blocks for w13 and E*(H/128)*(I/128)
 * for w2 (the raw code + scale bytes, re-ordered). */
#define KMOE_WEIGHT_BLOCK_BYTES (8192 + 512)
size_t kmoe_prepared_weight_bytes(const kmoe_params* p, int which);

/* One-time weight preparation (load time, not per forward; cf. the pages'
 * process_weights_after_loading re-layout for the SM100 path).  Re-lays the
 * raw checkpoint tensors into the order the GEMMs stream them: for each
 * expert, each 128-row weight tile (FC1: gate rows 64m..64m+63 followed by
 * the matching up rows I+64m..; FC2: rows 128m..128m+127) and each 128-wide K
 * block, one contiguous block of 128 rows x 64 code bytes followed by the 512
 * scale bytes of those rows (32 lanes x 4 rows x 4 K groups, the order in
 * which tcgen05.cp copies scales into tensor memory).
 *   w13 [E, 2I, H/2], w13_sf [E, 2I, H/32], w2 [E, H, I/2], w2_sf [E, H, I/32]
 *   (raw, in; codes 16-byte aligned);
 *   w13_k, w2_k (out, kmoe_prepared_weight_bytes each, 256-byte aligned). */
int kmoe_prepare_weights(const kmoe_params* p, const uint8_t* w13, const uint8_t* w13_sf, const uint8_t* w2,
                         const uint8_t* w2_sf, uint8_t* w13_k, uint8_t* w2_k, cudaStream_t stream);

/* The routed-expert MoE forward:
 *   route (unless topk_ids/topk_w are given) -> MXFP8-quantise x ->
 *   expert-sorted permutation -> FC1 (x . w13^T, gate and up) -> SiTU (or
 *   the SwiGLU control with KMOE_FLAG_SWIGLU) -> MXFP8 requantise -> FC2
 *   (. w2^T) -> out[t] = bf16(rsf * sum_j w_j y_j)
 *   with slots summed in order j = 0..k-1 in fp32 (deterministic).
 * x [T, H] bf16 (16-byte aligned); logits/bias as kmoe_route (ignored when
 * topk_ids is given); w13_k/w2_k from kmoe_prepare_weights (256-byte
 * aligned); topk_ids [T, k] int32 and topk_w [T, k] float optional (both or
 * neither; an id < 0 marks a masked slot that adds 0; an id >= E raises
 * KMOE_ERR_DEVICE via kmoe_device_error and is masked); out [T, H] bf16
 * (16-byte aligned); workspace of kmoe_workspace_size(p) bytes, 256-byte
 * aligned, reused by every call (not thread-safe per workspace). */
int kmoe_forward(const kmoe_params* p, const void* x_bf16, const float* logits, const float* bias,
                 const uint8_t* w13_k, const uint8_t* w2_k, const int32_t* topk_ids, const float* topk_w,
                 void* out_bf16, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Events recorded on `stream` between the stages of kmoe_forward_ex (host
 * struct of caller-created events; a null field is skipped).  Recorded in
 * order: start, after routing (or the copy of the given routing), after the
 * permutation, after the quantise-scatter, after FC1, after FC2, after the
 * combine.  For profiling; the kernels launched are the same. */
typedef struct kmoe_stage_events {
  cudaEvent_t start, routed, permuted, quantized, fc1, fc2, combined;
} kmoe_stage_events;

/* kmoe_forward with optional stage events (ev may be null). */
int kmoe_forward_ex(const kmoe_params* p, const void* x_bf16, const float* logits, const float* bias,
                    const uint8_t* w13_k, const uint8_t* w2_k, const int32_t* topk_ids, const float* topk_w,
                    void* out_bf16, void* workspace, size_t ws_bytes, cudaStream_t stream,
                    const kmoe_stage_events* ev /* host */);

/* kmoe_forward with the fused router (kmoe_router) in place of the routing
 * kernel: the routing comes from x and the gate weight w_gate [E, H] bf16
 * (16-byte aligned; H a multiple of 64, E a multiple of 4) instead of given
 * logits.  The logits are left in the workspace (kmoe_ws_layout.logits).
 * Other arguments, the workspace and the error behaviour are those of
 * kmoe_forward_ex (ev may be null; its `routed` event follows the router). */
int kmoe_forward_router(const kmoe_params* p, const void* x_bf16, const void* w_gate_bf16, const float* bias,
                        const uint8_t* w13_k, const uint8_t* w2_k, void* out_bf16, void* workspace, size_t ws_bytes,
                        cudaStream_t stream, const kmoe_stage_events* ev /* host */);

/* Reads the device error word of `workspace` (synchronises `stream`), clears
 * it, and returns KMOE_OK, KMOE_ERR_TIMEOUT or KMOE_ERR_DEVICE.  *word (host,
 * may be null) receives the raw bits (1: a bounded wait timed out, 2: an
 * expert id >= E was seen).  kmoe_forward clears the word when it starts, so
 * it reports the most recent forward on that workspace. */
int kmoe_device_error(void* workspace, uint32_t* word, cudaStream_t stream);

/* Byte offset, inside a tile-layout scale array (xsf/isf, or xsf_big/isf_big,
 * of the workspace), of the scale of row `local_row` of token tile `tile` for
 * 32-group `g` (K index 32g..32g+31), given the array's tile size (tile_rows
 * or tile_rows_big), the K width in elements and the tile capacity of the
 * array.  Host helper for inspection. */
size_t kmoe_tile_sf_offset(int tile, int local_row, int g, int tile_rows, int K, int max_tiles);

/* Measurement aid: the tensor-pipe roof of the instruction the expert GEMMs
 * issue (tcgen05.mma .kind::mxf8f6f4 block-scaled, E2M1 A of 128 rows x E4M3
 * B of N rows, K = 32 per instruction).  Launches one CTA per SM, each issuing
 * 4 * iters such instructions on operands resident in shared memory; the
 * caller times the stream.  FLOPs of the launch:
 * num_SMs * iters * 4 * 2 * 128 * N * 32.  N a multiple of 16 in [16, 256],
 * iters in [1, 2^24].  A wait that gives up sets the timeout bit of
 * workspace's error word (read with kmoe_device_error). */
int kmoe_mma_peak_run(int iters, int N, void* workspace, cudaStream_t stream);

/* Self-test of the bounded device wait: launches one block that waits on a
 * barrier nobody arrives at, for at most `budget_us` microseconds, and
 * reports the outcome in workspace's error word (read it with
 * kmoe_device_error, which must then return KMOE_ERR_TIMEOUT). */
int kmoe_selftest_wait_timeout(void* workspace, int budget_us, cudaStream_t stream);

/* Self-test of the FC1 epilogue's activation: out[i] = the activation that
 * the forward applies to (gate[i], up[i]), evaluated by the same device
 * functions in fp32 (SiTU with p->situ_beta and p->situ_linear_beta, or the
 * SwiGLU control with KMOE_FLAG_SWIGLU and its parameters; SM120 page, SiTU
 * reference formula and activation table).  It lets a test bound the fp32
 * evaluation's error against an exact reference.  Only the activation fields
 * of *p are read (and checked as kmoe_forward checks them); gate, up and out
 * are device arrays of n floats. */
int kmoe_selftest_activation(const kmoe_params* p, const float* gate, const float* up, int n, float* out,
                             cudaStream_t stream);

/* Size of the scratch array built into the library for kmoe_forward_noalloc
 * (32 MiB, reserved on every GPU that loads the library until the process
 * exits). */
#define KMOE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/* kmoe_forward for callers that cannot allocate device memory -- for example
 * a runtime that plans all GPU memory up front, or a plug-in that receives a
 * stream but no allocator -- and so cannot pass a workspace.  The pages this
 * library follows have no counterpart of this call; it is an integration aid.
 * Arguments are those of kmoe_forward without the workspace; the caller still
 * owns every input and output.  The workspace is a fixed array inside the
 * library of KMOE_NOALLOC_SCRATCH_BYTES; layers whose kmoe_workspace_size()
 * exceeds it are rejected with KMOE_ERR_WORKSPACE (small decode batches fit:
 * T = 16 at H = 7168, I = 3584, E = 896, k = 16 needs about 21 MiB).  Nothing
 * is allocated or freed.  The first call on a device looks up the array's
 * device address with that device current; make that first call before any
 * stream capture.  A device reset (cudaDeviceReset) ends the context that
 * address belongs to; the first call after it looks the address up again.
 * Every call uses the same array, which keeps the previous call's contents,
 * so calls that can overlap on the GPU race: order them.
 * device_error (device pointer, optional) receives the call's device error
 * word (the bits kmoe_device_error reports) when the stream reaches it; an
 * empty batch (T = 0) writes 0 there. */
int kmoe_forward_noalloc(const kmoe_params* p, const void* x_bf16, const float* logits, const float* bias,
                         const uint8_t* w13_k, const uint8_t* w2_k, const int32_t* topk_ids, const float* topk_w,
                         void* out_bf16, uint32_t* device_error, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* KMOE_H_ */
