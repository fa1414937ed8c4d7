// Quantised AdamW state codec on sm_103a ("Full-Stack FP4: Stable LLM
// Pretraining with Quantized Projections, Optimizers, and Attention",
// section 2.2, Q-AdamW).
//
// First moment m [rows, cols] (FP32):
//   x = 1/4 H16 diag(sigma) m per run of 16 along a row (Hadamard mixing);
//   s = amax(x) / 2688 (1 if zero);
//   per run, adaptive 4/6: the block-scale bytes E4M3((bamax/6)/s) and
//   E4M3((bamax/4)/s) are both tried and the one with the smaller
//   round-to-nearest squared error (left-to-right FP32 sum) is kept, the
//   6-mapping on a tie; the run is then rounded stochastically with it
//   (Philox4x32-10 word per element, as the quantiser).
// Second moment v [rows, cols] (FP32 >= 0, rows and cols multiples of 16):
//   r = sqrt(v); per 16x16 tile mu = BF16(RN(T * 2^-8)) with T the row sums
//   (left to right) added in row order; residual e = r - mu; x = 1/4 H16
//   diag(sigma) e per run; s = amax(x) / 2688; round-to-nearest NVFP4 (1x16).
// Decoding inverts each step (inverse transform diag(sigma) 1/4 H16, plus mu,
// squared for v).
//
// One thread per run of 16: a 256-thread CTA covers 16 rows x 16 column
// blocks, thread t taking row t & 15 of column block t >> 4, so the 16 runs of
// a 16x16 tile are 16 adjacent lanes (the tile mean is a shuffle sum in row
// order).  Two passes for the encoders: the transformed amax (one atomicMax
// of FP32 bits per CTA), then the encode with s from it.  Every FP32 step is
// an explicit round-to-nearest operation, so the codes equal the plain
// statement of the codec bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "encode.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerCta = 16;
constexpr int kBlocksPerCta = kThreads / kRowsPerCta;  // column blocks of 16
constexpr size_t kAmaxWordOffset = 64;                 // in the workspace header

struct CodecParams {
  const float* in;        // m or v (encode)
  float* out;             // m_hat or v_hat (decode)
  uint8_t* codes;         // [rows, cols/2]
  uint8_t* sf;            // [rows, cols/16], row-major
  float* tensor_scale;    // device
  const float* tensor_scale_in;
  uint16_t* mean;         // [rows/16, cols/16] BF16 bits (v only)
  const uint16_t* mean_in;
  uint32_t* amax;         // FP32 bits, workspace
  uint32_t* status;
  int64_t rows, cols, kb;
  uint64_t sr_offset;
  uint32_t sgn[16];       // transform signs as FP32 sign bits
  uint32_t rk0[10], rk1[10];  // Philox round keys of sr_seed
};

__device__ __forceinline__ void load16(const float* p, float (&v)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 f = reinterpret_cast<const float4*>(p)[q];
    v[4 * q] = f.x;
    v[4 * q + 1] = f.y;
    v[4 * q + 2] = f.z;
    v[4 * q + 3] = f.w;
  }
}

__device__ __forceinline__ void store16(float* p, const float (&v)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    reinterpret_cast<float4*>(p)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// x' = 1/4 H16 diag(sigma) x (sigma as sign bits; flipping the sign bit is the
// exact product by -1).
__device__ __forceinline__ void forward16(float (&v)[16], const uint32_t (&sgn)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(__float_as_uint(v[j]) ^ sgn[j]);
#pragma unroll
  for (int st = 1; st < 16; st <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & st) continue;
      const float a = v[i], b = v[i + st];
      v[i] = __fadd_rn(a, b);
      v[i + st] = __fsub_rn(a, b);
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], 0.25f);
}

// x = diag(sigma) 1/4 H16 x' (H16 H16 = 16 I).
__device__ __forceinline__ void inverse16(float (&v)[16], const uint32_t (&sgn)[16]) {
#pragma unroll
  for (int st = 1; st < 16; st <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & st) continue;
      const float a = v[i], b = v[i + st];
      v[i] = __fadd_rn(a, b);
      v[i + st] = __fsub_rn(a, b);
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(__float_as_uint(__fmul_rn(v[j], 0.25f)) ^ sgn[j]);
}

// The values of sixteen E2M1 codes (two words, element j in nibble j & 7 of
// word j >> 3), exact, by the hardware conversion to f16.
__device__ __forceinline__ void e2m1_values(uint32_t w0, uint32_t w1, float (&val)[16]) {
  uint32_t h[8];
  ptx::cvt_e2m1x8_to_f16x2(w0, *reinterpret_cast<uint32_t(*)[4]>(&h[0]));
  ptx::cvt_e2m1x8_to_f16x2(w1, *reinterpret_cast<uint32_t(*)[4]>(&h[4]));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 p2 = *reinterpret_cast<const __half2*>(&h[i]);
    val[2 * i] = __low2float(p2);
    val[2 * i + 1] = __high2float(p2);
  }
}

// Round-to-nearest squared error of a run under scale byte sfb (left-to-right FP32 sum).
__device__ __forceinline__ float rne_error(const float (&x)[16], uint32_t sfb, float s) {
  float deq[16];
  if (sfb != 0) {
    const float d = __fmul_rn(ptx::e4m3_to_float(sfb), s);
    float q[16];
    divide_run<false>(x, d, q);  // the IEEE quotients (residual-corrected where that is exact)
    e2m1_values(ptx::cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]),
                ptx::cvt_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]), deq);
#pragma unroll
    for (int j = 0; j < 16; ++j) deq[j] = __fmul_rn(deq[j], d);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) deq[j] = 0.0f;
  }
  float err = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float e = __fsub_rn(x[j], deq[j]);
    err = __fadd_rn(err, __fmul_rn(e, e));
  }
  return err;
}

// The second moment's run, ready to quantise: sqrt, minus the tile mean,
// transformed.  All 32 lanes take part in the shuffles; lanes of column
// blocks past the tensor carry zeros.
__device__ __forceinline__ uint16_t v_residual(const CodecParams& p, int64_t row, int64_t cb, bool valid,
                                               float (&x)[16]) {
  float rowsum = 0.0f;
  if (valid) {
    load16(p.in + row * p.cols + cb * 16, x);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      x[j] = __fsqrt_rn(x[j]);
      rowsum = __fadd_rn(rowsum, x[j]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = 0.0f;
  }
  const int base = threadIdx.x & 16;  // first lane of this tile's 16
  float total = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) total = __fadd_rn(total, __shfl_sync(0xFFFFFFFFu, rowsum, base + i));
  const __nv_bfloat16 mu = __float2bfloat16_rn(__fmul_rn(total, 0.00390625f));
  const float muf = __bfloat162float(mu);
#pragma unroll
  for (int j = 0; j < 16; ++j) x[j] = __fsub_rn(x[j], muf);
  forward16(x, p.sgn);
  return *reinterpret_cast<const uint16_t*>(&mu);
}

__device__ __forceinline__ void amax_reduce(uint32_t m, uint32_t* out) {
  __shared__ uint32_t red[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) t = max(t, red[w]);
    atomicMax(out, t);
  }
}

// CTA b covers rows 16 (b / groups) .. + 15 and column blocks 16 (b % groups)
// .. + 15, groups = ceil(kb / 16).
__device__ __forceinline__ void run_coords(const CodecParams& p, int64_t& row, int64_t& cb, bool& valid) {
  const int64_t groups = (p.kb + kBlocksPerCta - 1) / kBlocksPerCta;
  const int64_t band = static_cast<int64_t>(blockIdx.x) / groups, grp = static_cast<int64_t>(blockIdx.x) % groups;
  row = band * kRowsPerCta + (threadIdx.x & 15);
  cb = grp * kBlocksPerCta + (threadIdx.x >> 4);
  valid = row < p.rows && cb < p.kb;
}

// Tensor scale from the amax word; false (and the status / NaN scale set) if
// the amax is not finite.
__device__ __forceinline__ bool scale_from_amax(const CodecParams& p, float& s) {
  const uint32_t m = *p.amax;
  if (m >= 0x7F800000u) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      ptx::set_status(p.status, kDevNonFinite);
      *p.tensor_scale = __uint_as_float(0x7FC00000u);
    }
    return false;
  }
  s = __fdiv_rn(__uint_as_float(m), 2688.0f);
  if (s == 0.0f) s = 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.tensor_scale = s;
  return true;
}

// ------------------------------------------------------------ first moment
__global__ void __launch_bounds__(kThreads) m_amax(const CodecParams p) {
  int64_t row, cb;
  bool valid;
  run_coords(p, row, cb, valid);
  uint32_t m = 0;
  if (valid) {
    float x[16];
    load16(p.in + row * p.cols + cb * 16, x);
    forward16(x, p.sgn);
    m = run_absmax_nan(x);
  }
  amax_reduce(m, p.amax);
}

__global__ void __launch_bounds__(kThreads) m_encode(const CodecParams p) {
  float s;
  if (!scale_from_amax(p, s)) return;
  int64_t row, cb;
  bool valid;
  run_coords(p, row, cb, valid);
  if (!valid) return;
  float x[16];
  load16(p.in + row * p.cols + cb * 16, x);
  forward16(x, p.sgn);
  const float bamax = __uint_as_float(run_absmax_nan(x));
  const uint32_t sf6 = ptx::cvt_e4m3(__fdiv_rn(__fdiv_rn(bamax, 6.0f), s));
  const uint32_t sf4 = ptx::cvt_e4m3(__fdiv_rn(__fdiv_rn(bamax, 4.0f), s));
  const uint32_t sfb = rne_error(x, sf4, s) < rne_error(x, sf6, s) ? sf4 : sf6;
  uint32_t w[2] = {0u, 0u};
  if (sfb != 0) {
    const float d = __fmul_rn(ptx::e4m3_to_float(sfb), s);
    float q[16];
    divide_run<true>(x, d, q);
    const uint64_t e0 = static_cast<uint64_t>(row * p.cols + cb * 16);
    const uint32_t o0 = static_cast<uint32_t>(p.sr_offset), o1 = static_cast<uint32_t>(p.sr_offset >> 32);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint64_t c = (e0 >> 2) + g;
      const uint4 r = philox4x32_10_rk(make_uint4(static_cast<uint32_t>(c), static_cast<uint32_t>(c >> 32), o0, o1),
                                       p.rk0, p.rk1);
      const float q0 = sr_round(q[4 * g], r.x), q1 = sr_round(q[4 * g + 1], r.y);
      const float q2 = sr_round(q[4 * g + 2], r.z), q3 = sr_round(q[4 * g + 3], r.w);
      // the rounded values are grid points: RNE conversion is exact
      const uint32_t c4 = ptx::cvt_e2m1x8(q0, q1, q2, q3, 0.f, 0.f, 0.f, 0.f) & 0xFFFFu;
      w[g >> 1] |= c4 << (16 * (g & 1));
    }
  }
  *reinterpret_cast<uint2*>(p.codes + row * (p.cols / 2) + cb * 8) = make_uint2(w[0], w[1]);
  p.sf[row * p.kb + cb] = static_cast<uint8_t>(sfb);
}

// Dequantised run: e2m1(code) * (e4m3(sf) * s).
__device__ __forceinline__ void dequant_run(const CodecParams& p, int64_t row, int64_t cb, float (&x)[16]) {
  const uint2 w = *reinterpret_cast<const uint2*>(p.codes + row * (p.cols / 2) + cb * 8);
  const float d = __fmul_rn(ptx::e4m3_to_float(p.sf[row * p.kb + cb]), *p.tensor_scale_in);
  e2m1_values(w.x, w.y, x);
#pragma unroll
  for (int j = 0; j < 16; ++j) x[j] = __fmul_rn(x[j], d);
}

__global__ void __launch_bounds__(kThreads) m_decode(const CodecParams p) {
  int64_t row, cb;
  bool valid;
  run_coords(p, row, cb, valid);
  if (!valid) return;
  float x[16];
  dequant_run(p, row, cb, x);
  inverse16(x, p.sgn);
  store16(p.out + row * p.cols + cb * 16, x);
}

// ----------------------------------------------------------- second moment
__global__ void __launch_bounds__(kThreads) v_amax(const CodecParams p) {
  int64_t row, cb;
  bool valid;
  run_coords(p, row, cb, valid);
  float x[16];
  v_residual(p, row, cb, valid, x);
  uint32_t m = valid ? run_absmax_nan(x) : 0u;
  if (valid) {
    // a negative or non-finite v shows as a NaN or infinite square root
    const float* in = p.in + row * p.cols + cb * 16;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (!(in[j] >= 0.0f) || in[j] == __uint_as_float(0x7F800000u)) m = 0x7FC00000u;
  }
  amax_reduce(m, p.amax);
}

__global__ void __launch_bounds__(kThreads) v_encode(const CodecParams p) {
  float s;
  if (!scale_from_amax(p, s)) return;
  int64_t row, cb;
  bool valid;
  run_coords(p, row, cb, valid);
  float x[16];
  const uint16_t mu = v_residual(p, row, cb, valid, x);
  if (!valid) return;
  if ((threadIdx.x & 15) == 0) p.mean[(row / 16) * p.kb + cb] = mu;
  const uint32_t sfb = block_scale_byte(run_absmax_nan(x), s);
  uint32_t w[2] = {0u, 0u};
  if (sfb != 0) {
    const float d = __fmul_rn(ptx::e4m3_to_float(sfb), s);
    float q[16];
    divide_run<false>(x, d, q);
    w[0] = ptx::cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
    w[1] = ptx::cvt_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]);
  }
  *reinterpret_cast<uint2*>(p.codes + row * (p.cols / 2) + cb * 8) = make_uint2(w[0], w[1]);
  p.sf[row * p.kb + cb] = static_cast<uint8_t>(sfb);
}

__global__ void __launch_bounds__(kThreads) v_decode(const CodecParams p) {
  int64_t row, cb;
  bool valid;
  run_coords(p, row, cb, valid);
  if (!valid) return;
  float x[16];
  dequant_run(p, row, cb, x);
  inverse16(x, p.sgn);
  const uint16_t mb = p.mean_in[(row / 16) * p.kb + cb];
  const float muf = __uint_as_float(static_cast<uint32_t>(mb) << 16);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float r = __fadd_rn(muf, x[j]);
    x[j] = __fmul_rn(r, r);
  }
  store16(p.out + row * p.cols + cb * 16, x);
}

dim3 codec_grid(int64_t rows, int64_t kb) {
  return dim3(static_cast<unsigned>(((kb + kBlocksPerCta - 1) / kBlocksPerCta) *
                                    ((rows + kRowsPerCta - 1) / kRowsPerCta)));
}

}  // namespace

cudaError_t launch_qadamw(const QadamwArgs& a, cudaStream_t stream) {
  CodecParams p{};
  p.in = a.in;
  p.out = a.out;
  p.codes = a.codes;
  p.sf = a.sf;
  p.tensor_scale = a.tensor_scale;
  p.tensor_scale_in = a.tensor_scale_in;
  p.mean = a.mean;
  p.mean_in = a.mean_in;
  p.rows = a.rows;
  p.cols = a.cols;
  p.kb = a.cols / 16;
  p.sr_offset = a.sr_offset;
  rht_sign_words(a.rht_seed, true, p.sgn);
  philox_round_keys(a.sr_seed, p.rk0, p.rk1);
  if (a.rows == 0 || a.cols == 0) return cudaSuccess;
  if (((p.kb + kBlocksPerCta - 1) / kBlocksPerCta) * ((a.rows + kRowsPerCta - 1) / kRowsPerCta) > 0x7FFFFFFFLL)
    return cudaErrorInvalidValue;
  const dim3 grid = codec_grid(a.rows, p.kb);
  if (a.op == QadamwArgs::kMDecode) {
    m_decode<<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
  }
  if (a.op == QadamwArgs::kVDecode) {
    v_decode<<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
  }
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.amax = reinterpret_cast<uint32_t*>(ws + kAmaxWordOffset);
  cudaError_t e = cudaMemsetAsync(p.amax, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  if (a.op == QadamwArgs::kMEncode) {
    m_amax<<<grid, kThreads, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    m_encode<<<grid, kThreads, 0, stream>>>(p);
  } else {
    v_amax<<<grid, kThreads, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    v_encode<<<grid, kThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace nvfp4
