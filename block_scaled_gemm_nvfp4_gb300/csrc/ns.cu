// Newton-Schulz step of the Root optimizer with NVFP4 products (sm_103a).
//
// "Full-Stack FP4: Stable LLM Pretraining with Quantized Projections,
// Optimizers, and Attention", section 2.3 (Q-Root): the Newton-Schulz matrix
// products run directly in NVFP4, stabilised by shape-dependent coefficients
// a, b, c and clipping of p99 outliers.  The pages print neither the
// coefficients nor the step; the step built here is the quintic one on an
// iterate X [m, n]:
//     A = X X^T,   B = b A + c A A^T,   X' = a X + B X,
// every product L R^T the NVFP4 GEMM of its operands, each clipped to
// [-q, q] with q its own p-th percentile magnitude (nearest rank) and then
// quantised along its K (1x16 blocks, round to nearest even), results in BF16.
//
// Kernels in this file (the rest of the step is nvfp4_quantize_dual,
// nvfp4_quantize and nvfp4_gemm):
//   * the p-th percentile of |x| over a BF16 tensor, exactly: a two-level
//     radix selection on the 15-bit magnitude pattern (for non-negative
//     floats the bit order is the value order), one pass for a histogram of
//     the top 8 bits, one for the low 7 bits inside the selected bin, and a
//     one-block selection that writes q;
//   * clipping to [-q, q] (on the bit patterns: a magnitude above q's becomes
//     q's, with the element's sign), BF16 in and out, exact; inside the step
//     the clip kernel also does the selection, so each percentile-and-clip
//     is two histogram passes and one clip pass;
//   * out = BF16(RN(RN(a x) + RN(b y))), elementwise in FP32.
// All three are HBM-bound streaming kernels: 16-byte vector loads and stores,
// grids of a few CTAs per SM.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kHiBins = 256;  // magnitude bits 14..7
constexpr int kLoBins = 128;  // magnitude bits 6..0

__device__ __forceinline__ uint32_t bf16_lo(uint32_t w) { return w & 0xFFFFu; }
__device__ __forceinline__ uint32_t bf16_hi(uint32_t w) { return w >> 16; }

// Visit every BF16 element of x [n] (16-byte aligned) as its bit pattern:
// whole 8-element vectors first, then the tail.
template <typename F>
__device__ __forceinline__ void for_each_bf16(const uint16_t* x, int64_t n, F&& f) {
  const int64_t nvec = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    const uint4 w = __ldcs(xv + i);
    f(bf16_lo(w.x)); f(bf16_hi(w.x)); f(bf16_lo(w.y)); f(bf16_hi(w.y));
    f(bf16_lo(w.z)); f(bf16_hi(w.z)); f(bf16_lo(w.w)); f(bf16_hi(w.w));
  }
  for (int64_t i = nvec * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    f(static_cast<uint32_t>(x[i]));
}

// Histogram of the top 8 magnitude bits.  Per-warp private histograms in
// shared memory keep the atomics on a few hot bins (values of one scale)
// from serialising across the block.  A NaN (magnitude above 0x7F80) is
// reported as non-finite; the percentile is then unspecified.
__global__ void __launch_bounds__(kThreads) hist_hi_kernel(const uint16_t* x, int64_t n, uint32_t* hist,
                                                            uint32_t* status) {
  __shared__ uint32_t h[kWarps][kHiBins];
  for (int i = threadIdx.x; i < kWarps * kHiBins; i += kThreads) (&h[0][0])[i] = 0;
  __syncthreads();
  uint32_t* mine = h[threadIdx.x >> 5];
  bool bad = false;
  for_each_bf16(x, n, [&](uint32_t b) {
    const uint32_t m = b & 0x7FFFu;
    bad |= m > 0x7F80u;
    atomicAdd(&mine[m >> 7], 1u);
  });
  if (__syncthreads_or(bad) && threadIdx.x == 0) ptx::set_status(status, kDevNonFinite);
  for (int bin = threadIdx.x; bin < kHiBins; bin += kThreads) {
    uint32_t s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += h[w][bin];
    if (s) atomicAdd(&hist[bin], s);
  }
}

// The bin holding the k-th smallest value (1-based) of a histogram, and the
// rank inside it.  One warp, sequential over the bins in chunks of 32.
__device__ __forceinline__ void select_bin(const uint32_t* hist, int bins, uint64_t k, int& bin, uint64_t& k_in) {
  const int lane = threadIdx.x & 31;
  uint64_t before = 0;
  bin = bins - 1;
  k_in = 1;
  for (int base = 0; base < bins; base += 32) {
    const uint64_t c = (base + lane < bins) ? hist[base + lane] : 0u;
    // inclusive prefix sum over the warp
    uint64_t inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
      if (lane >= o) inc += t;
    }
    const bool hit = before + inc >= k && before + inc - c < k;
    const uint32_t mask = __ballot_sync(0xFFFFFFFFu, hit);
    if (mask) {
      const int src = __ffs(mask) - 1;
      const uint64_t exc = __shfl_sync(0xFFFFFFFFu, before + inc - c, src);
      bin = base + src;
      k_in = k - exc;
      return;
    }
    before += __shfl_sync(0xFFFFFFFFu, inc, 31);
  }
}

// Histogram of the low 7 magnitude bits of the elements whose top 8 bits
// are the selected bin (each block finds that bin itself).
__global__ void __launch_bounds__(kThreads) hist_lo_kernel(const uint16_t* x, int64_t n, uint64_t k,
                                                            const uint32_t* hist_hi, uint32_t* hist_lo) {
  __shared__ uint32_t h[kWarps][kLoBins];
  __shared__ int sel;
  for (int i = threadIdx.x; i < kWarps * kLoBins; i += kThreads) (&h[0][0])[i] = 0;
  if (threadIdx.x < 32) {
    int bin;
    uint64_t k_in;
    select_bin(hist_hi, kHiBins, k, bin, k_in);
    if (threadIdx.x == 0) sel = bin;
  }
  __syncthreads();
  const uint32_t want = static_cast<uint32_t>(sel);
  uint32_t* mine = h[threadIdx.x >> 5];
  for_each_bf16(x, n, [&](uint32_t b) {
    const uint32_t m = b & 0x7FFFu;
    if ((m >> 7) == want) atomicAdd(&mine[m & 127u], 1u);
  });
  __syncthreads();
  for (int bin = threadIdx.x; bin < kLoBins; bin += kThreads) {
    uint32_t s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += h[w][bin];
    if (s) atomicAdd(&hist_lo[bin], s);
  }
}

// The selected magnitude's bit pattern from the two histograms (one warp).
__device__ __forceinline__ uint32_t select_bits(uint64_t k, const uint32_t* hist_hi, const uint32_t* hist_lo) {
  int hi, lo;
  uint64_t k_in, k_lo;
  select_bin(hist_hi, kHiBins, k, hi, k_in);
  select_bin(hist_lo, kLoBins, k_in, lo, k_lo);
  return (static_cast<uint32_t>(hi) << 7) | static_cast<uint32_t>(lo);
}

// q = the k-th smallest magnitude, as the FP32 value of its BF16 pattern.
__global__ void select_kernel(uint64_t k, const uint32_t* hist_hi, const uint32_t* hist_lo, float* q) {
  const uint32_t bits = select_bits(k, hist_hi, hist_lo);
  if (threadIdx.x == 0) *q = __uint_as_float(bits << 16);
}

__device__ __forceinline__ uint32_t clip_bits(uint32_t b, uint32_t qm) {
  const uint32_t m = b & 0x7FFFu;
  return (m > qm && m <= 0x7F80u) ? ((b & 0x8000u) | qm) : b;  // NaN passes through
}

// SELECT: the block's first warp selects the percentile from the histograms
// itself (block 0 also stores it in q), which saves the one-block selection
// launch inside the Newton-Schulz step; otherwise q is read.
template <bool SELECT>
__global__ void __launch_bounds__(kThreads) clip_kernel(const uint16_t* x, int64_t n, uint64_t k, const uint32_t* hist,
                                                        float* q, uint16_t* out) {
  __shared__ uint32_t sel;
  uint32_t qm;
  if (SELECT) {
    if (threadIdx.x < 32) {
      const uint32_t bits = select_bits(k, hist, hist + kHiBins);
      if (threadIdx.x == 0) {
        sel = bits;
        if (blockIdx.x == 0) *q = __uint_as_float(bits << 16);
      }
    }
    __syncthreads();
    qm = sel;
  } else {
    qm = (__float_as_uint(*q) >> 16) & 0x7FFFu;
  }
  const int64_t nvec = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint4* ov = reinterpret_cast<uint4*>(out);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    uint4 w = __ldcs(xv + i);
    uint32_t* e = &w.x;
#pragma unroll
    for (int j = 0; j < 4; ++j) e[j] = clip_bits(e[j] & 0xFFFFu, qm) | (clip_bits(e[j] >> 16, qm) << 16);
    ov[i] = w;
  }
  for (int64_t i = nvec * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = static_cast<uint16_t>(clip_bits(x[i], qm));
}

__device__ __forceinline__ uint32_t axpby1(uint32_t xb, uint32_t yb, float a, float b) {
  const float s = __fadd_rn(__fmul_rn(a, __uint_as_float(xb << 16)), __fmul_rn(b, __uint_as_float(yb << 16)));
  // BF16 round to nearest even of a finite FP32 value (NaN kept a NaN)
  const uint32_t u = __float_as_uint(s);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__global__ void __launch_bounds__(kThreads) axpby_kernel(const uint16_t* x, const uint16_t* y, int64_t n, float a,
                                                         float b, uint16_t* out) {
  const int64_t nvec = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const uint4* yv = reinterpret_cast<const uint4*>(y);
  uint4* ov = reinterpret_cast<uint4*>(out);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    const uint4 wx = __ldcs(xv + i), wy = __ldcs(yv + i);
    const uint32_t* ex = &wx.x;
    const uint32_t* ey = &wy.x;
    uint4 r;
    uint32_t* er = &r.x;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      er[j] = axpby1(ex[j] & 0xFFFFu, ey[j] & 0xFFFFu, a, b) | (axpby1(ex[j] >> 16, ey[j] >> 16, a, b) << 16);
    ov[i] = r;
  }
  for (int64_t i = nvec * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = static_cast<uint16_t>(axpby1(x[i], y[i], a, b));
}

int stream_grid(int64_t n) {
  const int64_t per_cta = static_cast<int64_t>(kThreads) * 8 * 4;  // four vectors per thread at least
  int64_t g = (n + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 4;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_abs_percentile(const uint16_t* x, int64_t n, uint64_t k, uint32_t* hist, float* q,
                                  uint32_t* status, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(hist, 0, (kHiBins + kLoBins) * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  const int g = stream_grid(n);
  hist_hi_kernel<<<g, kThreads, 0, stream>>>(x, n, hist, status);
  hist_lo_kernel<<<g, kThreads, 0, stream>>>(x, n, k, hist, hist + kHiBins);
  select_kernel<<<1, 32, 0, stream>>>(k, hist, hist + kHiBins, q);
  return cudaGetLastError();
}

cudaError_t launch_clip(const uint16_t* x, int64_t n, const float* q, uint16_t* out, cudaStream_t stream) {
  clip_kernel<false><<<stream_grid(n), kThreads, 0, stream>>>(x, n, 0, nullptr, const_cast<float*>(q), out);
  return cudaGetLastError();
}

cudaError_t launch_percentile_clip(const uint16_t* x, int64_t n, uint64_t k, uint32_t* hist, float* q, uint16_t* out,
                                   uint32_t* status, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(hist, 0, (kHiBins + kLoBins) * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  const int g = stream_grid(n);
  hist_hi_kernel<<<g, kThreads, 0, stream>>>(x, n, hist, status);
  hist_lo_kernel<<<g, kThreads, 0, stream>>>(x, n, k, hist, hist + kHiBins);
  clip_kernel<true><<<g, kThreads, 0, stream>>>(x, n, k, hist, q, out);
  return cudaGetLastError();
}

cudaError_t launch_axpby(const uint16_t* x, const uint16_t* y, int64_t n, float a, float b, uint16_t* out,
                         cudaStream_t stream) {
  axpby_kernel<<<stream_grid(n), kThreads, 0, stream>>>(x, y, n, a, b, out);
  return cudaGetLastError();
}

}  // namespace nvfp4
