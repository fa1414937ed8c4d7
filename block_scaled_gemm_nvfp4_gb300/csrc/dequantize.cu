// NVFP4 dequantisation: y = e2m1(code) * e4m3(scale) * s.
//
// The product of an E2M1 element and an E4M3 scale is exact in FP32, so the
// only rounding is the final multiply by the tensor scale; BF16 output is
// that FP32 value rounded to nearest even.  One thread per run of 16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

template <bool OUT_F32>
__global__ void __launch_bounds__(256) dequant_kernel(const DequantArgs a) {
  const int64_t kb_count = a.k / 16;
  const int64_t katoms = (kb_count + 3) / 4;
  const int64_t total = a.rows * kb_count;
  const float s = *a.tensor_scale;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / kb_count, kb = i - r * kb_count;
    int64_t si;
    if (a.sf_mma) {
      const int rr = static_cast<int>(r & 127);
      si = ((r >> 7) * katoms + (kb >> 2)) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + static_cast<int>(kb & 3);
    } else {
      si = r * kb_count + kb;
    }
    const float sfv = ptx::e4m3_to_float(a.sf[si]);
    const uint2 c = *reinterpret_cast<const uint2*>(a.codes + r * (a.k / 2) + kb * 8);
    float y[16];
    uint32_t h[4];
    ptx::cvt_e2m1x8_to_f16x2(c.x, h);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
      y[2 * j] = f.x;
      y[2 * j + 1] = f.y;
    }
    ptx::cvt_e2m1x8_to_f16x2(c.y, h);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
      y[8 + 2 * j] = f.x;
      y[8 + 2 * j + 1] = f.y;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) y[j] = __fmul_rn(__fmul_rn(y[j], sfv), s);
    if (OUT_F32) {
      float* out = static_cast<float*>(a.out) + r * a.ldo + kb * 16;
#pragma unroll
      for (int j = 0; j < 16; ++j) out[j] = y[j];
    } else {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + r * a.ldo + kb * 16;
#pragma unroll
      for (int j = 0; j < 16; ++j) out[j] = __float2bfloat16_rn(y[j]);
    }
  }
}

}  // namespace

cudaError_t launch_dequantize(const DequantArgs& a, cudaStream_t stream) {
  const int64_t total = a.rows * (a.k / 16);
  if (total == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 8 * device_sm_count());
  if (a.out_f32)
    dequant_kernel<true><<<static_cast<int>(blocks), 256, 0, stream>>>(a);
  else
    dequant_kernel<false><<<static_cast<int>(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace nvfp4
