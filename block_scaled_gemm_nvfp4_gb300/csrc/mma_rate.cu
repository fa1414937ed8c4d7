// Isolated tensor-core instruction rate: the ceiling the GEMM is measured
// against.  One CTA per SM (a CTA pair per two SMs for the cta_group::2
// forms); one thread per CTA (the pair's leader) issues back-to-back MMAs on
// fixed shared-memory operands into one TMEM accumulator, commits once and
// waits (bounded).  Operand and scale contents are whatever shared and
// tensor memory hold: the rate does not depend on them enough to matter
// (all-zero and random operands differ by about 2 % in the full GEMM), and
// nothing reads the accumulator.  The pages have no counterpart: this is a
// measurement tool for the block-scaled GEMM's roofline, not part of the
// method.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kRateThreads = 128;
// 120 KB of dynamic shared memory keeps one CTA per SM, so no two CTAs
// compete for an SM's tensor memory.
constexpr size_t kRateSmem = 120 * 1024 + 1024;

template <bool PAIR, bool F16>
__global__ void __launch_bounds__(kRateThreads, 1)
    mma_rate_kernel(unsigned long long* cycles, int iters, uint32_t idesc, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint32_t tmem_base;
  __shared__ __align__(8) uint64_t done;
  __shared__ int never;
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&done, 1);
    never = 0;
    ptx::fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    if (PAIR) {
      ptx::tmem_alloc_pair(&tmem_base, 512);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&tmem_base, 512);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (threadIdx.x == 0) {
    const unsigned long long t0 = clock64();
    if (rank == 0) {
      // A at offset 0 (16 KB), B at 32 KB (up to 32 KB): 128-byte swizzled
      // K-major tiles as in the GEMM; K steps advance 32 bytes in the rows
      const uint64_t ad = ptx::smem_desc(ptx::smem_u32(smem), 16, 1024, ptx::kSwizzle128B);
      const uint64_t bd = ptx::smem_desc(ptx::smem_u32(smem + 32768), 16, 1024, ptx::kSwizzle128B);
      for (int i = 0; i < iters; ++i) {
        const uint64_t o = static_cast<uint64_t>(2 * (i & 3));
        if (F16) {
          if (PAIR)
            ptx::tc_mma_f16_pair(tmem, ad + o, bd + o, idesc, 1u);
          else
            ptx::tc_mma_f16(tmem, ad + o, bd + o, idesc, 1u);
        } else {
          if (PAIR)
            ptx::tc_mma_nvf4_pair(tmem, ad + o, bd + o, idesc, tmem + 256, tmem + 336, 1u);
          else
            ptx::tc_mma_nvf4(tmem, ad + o, bd + o, idesc, tmem + 256, tmem + 336, 1u);
        }
      }
      if (PAIR)
        ptx::tc_commit_pair_multicast(&done, static_cast<uint16_t>(0x3));
      else
        ptx::tc_commit(&done);
    }
    if (!ptx::mbar_wait(&done, 0, &never)) ptx::set_status(status, kDevTimeout);
    cycles[blockIdx.x] = clock64() - t0;
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();
  if (threadIdx.x < 32) {
    ptx::tc_fence_after();
    if (PAIR)
      ptx::tmem_dealloc_pair(tmem, 512);
    else
      ptx::tmem_dealloc(tmem, 512);
  }
}

template <bool PAIR, bool F16>
cudaError_t launch_rate(int grid, unsigned long long* cycles, int iters, uint32_t idesc, uint32_t* status,
                        cudaStream_t stream) {
  auto k = mma_rate_kernel<PAIR, F16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kRateSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRateThreads);
  cfg.dynamicSmemBytes = kRateSmem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = PAIR ? 2 : 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, cycles, iters, idesc, status);
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_debug_mma_rate(int32_t kind, int32_t iters, double* tflops, double* cycles_per_mma) {
  using namespace nvfp4;
  if (kind < 0 || kind > 3 || iters < 16 || iters > (1 << 20) || !tflops || !cycles_per_mma)
    return NVFP4_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 2)
    return NVFP4_ERR_CUDA;
  const bool pair = kind == 0 || kind == 2;
  const bool f16 = kind >= 2;
  const int grid = pair ? sms & ~1 : sms;
  const int M = pair ? 256 : 128, N = 256, K = f16 ? 16 : 64;
  // instruction descriptor: A and B formats (E2M1 with E4M3 block scales, or
  // BF16 with an FP32 accumulator), N / 8, M / 16
  uint32_t idesc = f16 ? ((1u << 4) | (1u << 7) | (1u << 10)) : ((1u << 7) | (1u << 10));
  idesc |= static_cast<uint32_t>(N >> 3) << 17;
  idesc |= static_cast<uint32_t>(M >> 4) << 24;
  unsigned long long* cycles = nullptr;
  uint32_t* status = nullptr;
  if (cudaMalloc(&cycles, grid * sizeof(unsigned long long)) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaMalloc(&status, sizeof(uint32_t)) != cudaSuccess) {
    cudaFree(cycles);
    return NVFP4_ERR_CUDA;
  }
  cudaStream_t s = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  nvfp4_status rc = NVFP4_OK;
  auto launch = [&]() {
    if (pair) return f16 ? launch_rate<true, true>(grid, cycles, iters, idesc, status, s)
                         : launch_rate<true, false>(grid, cycles, iters, idesc, status, s);
    return f16 ? launch_rate<false, true>(grid, cycles, iters, idesc, status, s)
               : launch_rate<false, false>(grid, cycles, iters, idesc, status, s);
  };
  const int reps = 5;
  float ms = 0.0f;
  uint32_t st = 0;
  std::vector<unsigned long long> h(grid);
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess || cudaEventCreate(&e0) != cudaSuccess ||
      cudaEventCreate(&e1) != cudaSuccess || cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) {
    rc = NVFP4_ERR_CUDA;
  } else {
    bool ok = launch() == cudaSuccess && launch() == cudaSuccess && cudaEventRecord(e0, s) == cudaSuccess;
    for (int r = 0; ok && r < reps; ++r) ok = launch() == cudaSuccess;
    ok = ok && cudaEventRecord(e1, s) == cudaSuccess && cudaStreamSynchronize(s) == cudaSuccess &&
         cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess &&
         cudaMemcpy(&st, status, sizeof(uint32_t), cudaMemcpyDeviceToHost) == cudaSuccess &&
         cudaMemcpy(h.data(), cycles, grid * sizeof(unsigned long long), cudaMemcpyDeviceToHost) == cudaSuccess;
    if (!ok)
      rc = NVFP4_ERR_CUDA;
    else if (st != 0)
      rc = static_cast<nvfp4_status>(st);
  }
  if (rc == NVFP4_OK) {
    // issuing CTAs: every CTA in single mode, the leaders in pair mode
    double sum = 0.0;
    int n = 0;
    for (int i = 0; i < grid; i += pair ? 2 : 1, ++n) sum += static_cast<double>(h[i]);
    *cycles_per_mma = sum / n / iters;
    const double flops = 2.0 * M * N * K * static_cast<double>(iters) * (pair ? grid / 2 : grid);
    *tflops = flops / (ms / reps * 1e-3) / 1e12;
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (s) cudaStreamDestroy(s);
  cudaFree(status);
  cudaFree(cycles);
  return rc;
}
