// Measured FP8 tensor-core ceiling of this GPU: every SM runs one CTA whose single thread
// issues block-scaled tcgen05.mma (E4M3 x E4M3, UE8M0 scales, FP32 accumulation in TMEM)
// of shape 128 x 256 x 32 back to back from shared memory; the grid is timed with CUDA
// events. This bounds what any GEMM kernel of this library can reach on the same part
// (same instruction, no data movement). Not an operation of the method: a diagnostic for
// the roofline.
#include <cuda_runtime.h>

#include <cstdint>

#include "dg.h"
#include "ptx.cuh"

namespace {

constexpr int kN = 256;                       // MMA N (one 128 x 256 accumulator)
constexpr int kSmemBytes = 200 * 1024;        // keeps one CTA per SM
constexpr uint32_t kStatusTimeout = 1u;

__global__ void __launch_bounds__(128, 1) mma_ceiling_kernel(int iters, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a = base;                          // 128 rows x 128 bytes (one K-group of A)
  uint8_t* b = base + 128 * 128;              // 256 rows x 128 bytes
  uint8_t* sf = b + kN * 128;                 // scale chunks (UE8M0 code 127 = 1.0)
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t done_bar;
  // finite E4M3 bytes (exponent field <= 14, so never the NaN code), varying per element
  for (int i = threadIdx.x; i < 128 * 128 + kN * 128; i += blockDim.x) {
    const uint32_t h = (static_cast<uint32_t>(i) * 2654435761u) ^ (blockIdx.x * 40503u);
    base[i] = static_cast<uint8_t>((h >> 13) & 0x77u);
  }
  for (int i = threadIdx.x; i < 2048; i += blockDim.x) sf[i] = 127;
  if (threadIdx.x == 0) {
    dg::mbar_init(&done_bar, 1);
    dg::fence_mbarrier_init();
  }
  dg::fence_proxy_async_smem();
  __syncthreads();
  if (threadIdx.x / 32 == 0) {
    dg::tmem_alloc(&tmem_slot, 512);
    dg::tmem_relinquish();
  }
  dg::tc_fence_before();
  __syncthreads();
  dg::tc_fence_after();
  const uint32_t t = tmem_slot;
  if (threadIdx.x == 0) {
    const uint64_t ad = dg::make_smem_desc(dg::smem_addr(a), 16, 1024, dg::kLayoutSwizzle128B);
    const uint64_t bd = dg::make_smem_desc(dg::smem_addr(b), 16, 1024, dg::kLayoutSwizzle128B);
    const uint64_t sd = dg::make_smem_desc(dg::smem_addr(sf), 0, 128, dg::kLayoutNone);
    dg::tmem_copy_32x128b_warpx4(t + kN, sd);             // SFA: 4 columns
    dg::tmem_copy_32x128b_warpx4(t + kN + 8, sd);         // SFB: 8 columns
    dg::tmem_copy_32x128b_warpx4(t + kN + 12, sd);
    const uint32_t idesc = dg::make_idesc_mxf8_e4m3(128, kN);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        dg::mma_mxf8_block_scale(t, ad + 2 * k, bd + 2 * k, idesc, t + kN, t + kN + 8, (i | k) != 0);
    }
    dg::tc_commit(&done_bar);
    if (!dg::mbar_wait(&done_bar, 0, 2000000000ull)) atomicOr(status, kStatusTimeout);
  }
  dg::tc_fence_before();
  __syncthreads();
  if (threadIdx.x / 32 == 0) {
    dg::tc_fence_after();
    dg::tmem_dealloc(t, 512);
  }
}

}  // namespace

extern "C" dg_status dg_measure_fp8_mma_tflops(int iters_per_sm, double* tflops, double* ms) {
  if (iters_per_sm <= 0 || iters_per_sm > (1 << 20) || !tflops) return DG_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DG_ERR_CUDA;
  if (cudaFuncSetAttribute(mma_ceiling_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return DG_ERR_CUDA;
  uint32_t* status = nullptr;
  if (cudaMalloc(&status, sizeof(uint32_t)) != cudaSuccess) return DG_ERR_CUDA;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  dg_status result = DG_ERR_CUDA;
  float elapsed = 0.0f;
  uint32_t h_status = 0;
  if (cudaMemset(status, 0, sizeof(uint32_t)) == cudaSuccess && cudaEventCreate(&e0) == cudaSuccess &&
      cudaEventCreate(&e1) == cudaSuccess) {
    mma_ceiling_kernel<<<sms, 128, kSmemBytes>>>(iters_per_sm / 4 + 1, status);   // warm-up
    cudaEventRecord(e0);
    mma_ceiling_kernel<<<sms, 128, kSmemBytes>>>(iters_per_sm, status);
    cudaEventRecord(e1);
    if (cudaEventSynchronize(e1) == cudaSuccess && cudaEventElapsedTime(&elapsed, e0, e1) == cudaSuccess &&
        cudaMemcpy(&h_status, status, sizeof(uint32_t), cudaMemcpyDeviceToHost) == cudaSuccess) {
      if (h_status != 0) {
        result = DG_ERR_TIMEOUT;
      } else {
        const double flop = 2.0 * 128 * kN * 32 * 4.0 * iters_per_sm * sms;
        *tflops = flop / (static_cast<double>(elapsed) * 1e-3) / 1e12;
        if (ms) *ms = elapsed;
        result = DG_OK;
      }
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(status);
  cudaGetLastError();
  return result;
}
