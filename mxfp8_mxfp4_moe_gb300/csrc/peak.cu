// Tensor-pipe roof for the exact instruction the expert GEMMs issue:
// tcgen05.mma .kind::mxf8f6f4 block-scaled, E2M1 A (128 rows, unpacked smem
// format) x E4M3 B (N rows), fp32 accumulate in TMEM, one CTA per SM.  The
// operands stay resident in shared memory (zeros, smallest UE8M0 scales), so
// the kernel measures issue and tensor throughput only; the caller times it.
#include "common.cuh"

namespace kmoe {

__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int N, uint32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                 // 16 KB
  uint8_t* sB = smem + 16384;         // 32 KB (up to 256 rows)
  uint8_t* sSF = smem + 16384 + 32768;  // 1 KB: A scales, then B scales (two blocks)
  uint64_t* bar = reinterpret_cast<uint64_t*>(sSF + 1536);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (16384 + 32768 + 1536) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) {
    const uint32_t sf = tmem + 256;
    tc_cp_32x128b_warpx4(sf, sdesc_sf_32x16(smem_u32(sSF)));
    tc_cp_32x128b_warpx4(sf + 4, sdesc_sf_32x16(smem_u32(sSF + 512)));
    tc_cp_32x128b_warpx4(sf + 8, sdesc_sf_32x16(smem_u32(sSF + 1024)));
    const uint32_t aaddr = smem_u32(sA), baddr = smem_u32(sB);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_mxf8f6f4(tmem, sdesc_kmajor_sw128(aaddr + 32 * kk), sdesc_kmajor_sw128(baddr + 32 * kk),
                     idesc_mxf8f6f4(128, static_cast<uint32_t>(N), MX_E2M1, MX_E4M3, kk, kk), sf, sf + 4,
                     (it | kk) != 0);
    }
    tc_commit(bar);
    mbar_wait_bounded(bar, 0, 2000000000ull, err, nullptr);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_mma_peak(int iters, int N, int grid, uint32_t* err, cudaStream_t st) {
  const int smem = 1024 + 16384 + 32768 + 1536 + 64;
  static bool attr_set[kMaxDevices] = {};  // per device (idempotent)
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  mma_peak_kernel<<<grid, 128, smem, st>>>(iters, N, err);
  return cudaGetLastError();
}

}  // namespace kmoe
