// kmoe_forward_noalloc: the forward for callers that cannot allocate device
// memory.  Some hosts of this library own every byte of GPU memory themselves
// (a serving runtime with a fixed memory plan, a plugin that is handed a
// stream but no allocator, code that must not add allocations after start-up)
// and so cannot provide the workspace kmoe_forward needs.  This entry point
// keeps that workspace in one fixed array inside the library instead.
//
// The array below is reserved on every GPU that loads the library, for the
// life of the process.  Its device address is looked up once per device, on
// the first call made with that device current (cudaGetSymbolAddress); make
// that first call before capturing any stream.  All calls share the array and
// find the previous call's data in it: calls that may overlap on the GPU (on
// different streams, or from several host threads) race and must be ordered
// by the caller.  The stage kernels are the ones kmoe_forward uses.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = KMOE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (set-up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
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
  if (device_error != nullptr) {
    // the error word sits at the start of the workspace
    if (cudaMemcpyAsync(device_error, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
      return KMOE_ERR_CUDA;
  }
  return KMOE_OK;
}
