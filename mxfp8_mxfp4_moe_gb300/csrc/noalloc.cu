// kmoe_forward_noalloc: the forward for callers that cannot allocate device
// memory.  Some hosts of this library own every byte of GPU memory themselves
// (a serving runtime with a fixed memory plan, a plugin that is handed a
// stream but no allocator, code that must not add allocations after start-up)
// and so cannot provide the workspace kmoe_forward needs.  This entry point
// keeps that workspace in one fixed array inside the library instead.
//
// The array below is reserved on every GPU that loads the library, for the
// life of the process.  Its device address is looked up once per device
// context, on the first call made with that device current
// (cudaGetSymbolAddress); make that first call before capturing any stream.
// A device reset (cudaDeviceReset) ends the context and the module with it:
// the next call sees a new context and looks the address up again.  All
// calls share the array and find the previous call's data in it: calls that
// may overlap on the GPU (on different streams, or from several host threads)
// race and must be ordered by the caller.  The stage kernels are the ones
// kmoe_forward uses.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = KMOE_NOALLOC_SCRATCH_BYTES;
using kmoe::kMaxDevices;

static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
unsigned long long g_ctx[kMaxDevices] = {};  // id of the context each cached address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Id of the driver's current context, 0 if none is current: the device's
// primary context once cudaSetDevice has run, a new one (with a new id,
// unique within the process) after cudaDeviceReset.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_cur == nullptr || get_id == nullptr || get_cur(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_scratch on the current device (set-up on first use in
// each context of the device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long ctx = current_context_id();
  if (ctx == 0) {
    e = cudaSetDevice(dev);  // makes the device's primary context current
    if (e != cudaSuccess) return e;
    ctx = current_context_id();
    if (ctx == 0) return cudaErrorInitializationError;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr || g_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
    g_ctx[dev] = ctx;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int kmoe_forward_noalloc(const kmoe_params* p, const void* x_bf16, const float* logits,
                                    const float* bias, const uint8_t* w13_k, const uint8_t* w2_k,
                                    const int32_t* topk_ids, const float* topk_w, void* out_bf16,
                                    uint32_t* device_error, cudaStream_t stream) {
  const size_t need = kmoe_workspace_size(p);
  if (need == 0) return KMOE_ERR_ARG;
  if (need > kScratchBytes) return KMOE_ERR_WORKSPACE;  // layer too large for the built-in scratch
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return KMOE_ERR_CUDA;
  const int st = kmoe_forward(p, x_bf16, logits, bias, w13_k, w2_k, topk_ids, topk_w, out_bf16, ws, kScratchBytes,
                              stream);
  if (st != KMOE_OK) return st;
  if (device_error != nullptr && p->T == 0) {
    // an empty batch enqueues no stage, so the array's error word still holds
    // an earlier call's bits: report this call's (none)
    if (cudaMemsetAsync(device_error, 0, sizeof(uint32_t), stream) != cudaSuccess) return KMOE_ERR_CUDA;
  } else if (device_error != nullptr) {
    // the error word sits at the start of the workspace
    if (cudaMemcpyAsync(device_error, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
      return KMOE_ERR_CUDA;
  }
  return KMOE_OK;
}
