// NVFP4 quantisation of BF16 tensors (sm_103a).
//
// Two passes over the input, both persistent grid-stride loops over tiles:
//   pass 0: tensor amax (after the optional random Hadamard transform), one
//           partial per CTA written to the workspace;
//   pass 1: every CTA reduces the partials, derives the FP32 tensor scale
//           s = amax / 2688 and encodes its tiles into E2M1 codes and E4M3
//           block scales.  Pass 1 walks the tiles in reverse order so that
//           its first reads hit the part of the input pass 0 left in L2.
//
// Format and rounding sequence (per run of 16 along K; the pages' NVFP4
// elements on a sparse 4-bit grid with custom scaling, "NVIDIA acelera o
// pre-treinamento de LLM: NVFP4 no Blackwell...", section "Por que cada
// porcento e importante"; Hadamard mixing and stochastic rounding from
// "Full-Stack FP4...", section 2.2):
//   t = (bamax / 6) / s -> E4M3 (RNE, saturating), d = e4m3(t) * s,
//   v = x / d -> E2M1 by RNE or by stochastic rounding with a Philox4x32-10
//   word per element.  All FP32 steps are IEEE round-to-nearest operations
//   (explicit _rn intrinsics; the file is built without FMA contraction).
//
// Thread layouts (one thread owns whole runs of 16, so the transform and the
// block maximum stay in registers):
//   row mode (Q = x):   a warp covers 16 rows x 32 columns; lane -> row
//                       (lane & 15), run (lane >> 4).  CTA tile 16 x 256.
//   col mode (Q = x^T): a warp covers 16 rows x 64 columns of x; lane ->
//                       columns 2*lane, 2*lane + 1 (two runs).  CTA tile
//                       128 rows x 64 columns of x.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

struct QParams {
  const uint16_t* x;
  int64_t rows, cols, ldx;
  int64_t qr, qk, kb_count;
  uint8_t* codes;
  uint8_t* sf;
  float* tensor_scale;
  uint32_t* status;
  uint32_t* partials;
  uint64_t rht_seed, sr_seed, sr_offset;
  int64_t tiles_c, num_tiles;
  int64_t sf_katoms;
  int sf_mma;
  int num_partials;
};

// Philox4x32-10 (Salmon et al., SC'11): ten rounds, Weyl key schedule.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ int64_t sf_index(const QParams& p, int64_t r, int64_t kb) {
  if (!p.sf_mma) return r * p.kb_count + kb;
  const int64_t atom = (r >> 7) * p.sf_katoms + (kb >> 2);
  const int rr = static_cast<int>(r & 127);
  return atom * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + static_cast<int>(kb & 3);
}

__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

// x' = 1/4 * H16 * diag(sigma) * x; butterflies of stride 1, 2, 4, 8.
__device__ __forceinline__ void rht16(float (&v)[16], uint32_t sign_mask) {
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(__float_as_uint(v[j]) ^ (((sign_mask >> j) & 1u) << 31));
#pragma unroll
  for (int s = 1; s < 16; s <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & s) continue;
      const float a = v[i], b = v[i + s];
      v[i] = __fadd_rn(a, b);
      v[i + s] = __fsub_rn(a, b);
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], 0.25f);
}

__device__ __forceinline__ uint32_t run_absmax_bits(const float (&v)[16]) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) m = max(m, abs_bits(v[j]));
  return m;
}

// Stochastic rounding of q onto the E2M1 grid: lo, hi the grid points around
// |q|, f = (|q| - lo) / (hi - lo), up iff (r >> 8) * 2^-24 < f; |q| >= 6 -> 6.
__device__ __forceinline__ float sr_round(float q, uint32_t r) {
  const float mag = fabsf(q);
  float g;
  if (mag >= 6.0f) {
    g = 6.0f;
  } else {
    const float step = mag < 2.0f ? 0.5f : (mag < 4.0f ? 1.0f : 2.0f);
    const float inv = mag < 2.0f ? 2.0f : (mag < 4.0f ? 1.0f : 0.5f);
    const float lo = __fmul_rn(floorf(__fmul_rn(mag, inv)), step);
    const float f = __fmul_rn(__fsub_rn(mag, lo), inv);
    const float u = __fmul_rn(static_cast<float>(r >> 8), 5.9604644775390625e-08f);
    g = (u < f) ? __fadd_rn(lo, step) : lo;
  }
  return copysignf(g, q);
}

// Encode one run of 16 values with block maximum `bamax`; e0 is the linear
// index of the run's first element in Q (for the Philox counter).
template <bool SR>
__device__ __forceinline__ uint2 encode_run(const float (&v)[16], float bamax, float s_dec, uint64_t e0,
                                            const QParams& p, uint32_t& sfb) {
  const float t = __fdiv_rn(__fdiv_rn(bamax, 6.0f), s_dec);
  sfb = ptx::cvt_e4m3(t);
  if (sfb == 0) return make_uint2(0u, 0u);
  const float d = __fmul_rn(ptx::e4m3_to_float(sfb), s_dec);
  float q[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) q[j] = __fdiv_rn(v[j], d);
  if (SR) {
    const uint32_t k0 = static_cast<uint32_t>(p.sr_seed), k1 = static_cast<uint32_t>(p.sr_seed >> 32);
    const uint32_t o0 = static_cast<uint32_t>(p.sr_offset), o1 = static_cast<uint32_t>(p.sr_offset >> 32);
    const uint64_t c = e0 >> 2;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint64_t cg = c + g;
      const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(cg), static_cast<uint32_t>(cg >> 32), o0, o1),
                                    k0, k1);
      q[4 * g + 0] = sr_round(q[4 * g + 0], w.x);
      q[4 * g + 1] = sr_round(q[4 * g + 1], w.y);
      q[4 * g + 2] = sr_round(q[4 * g + 2], w.z);
      q[4 * g + 3] = sr_round(q[4 * g + 3], w.w);
    }
  }
  return make_uint2(ptx::cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]),
                    ptx::cvt_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]));
}

__device__ __forceinline__ void unpack8(const uint4& w, float* v) {
  v[0] = __uint_as_float(w.x << 16);
  v[1] = __uint_as_float(w.x & 0xFFFF0000u);
  v[2] = __uint_as_float(w.y << 16);
  v[3] = __uint_as_float(w.y & 0xFFFF0000u);
  v[4] = __uint_as_float(w.z << 16);
  v[5] = __uint_as_float(w.z & 0xFFFF0000u);
  v[6] = __uint_as_float(w.w << 16);
  v[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

template <int PASS>
__device__ __forceinline__ uint4 load16(const uint4* ptr) {
  // The amax pass leaves the input in L2 for the encode pass; the encode
  // pass is the last reader.
  return PASS == 0 ? __ldg(ptr) : __ldcs(ptr);
}
template <int PASS>
__device__ __forceinline__ uint32_t load4(const uint32_t* ptr) {
  return PASS == 0 ? __ldg(ptr) : __ldcs(ptr);
}
template <int PASS>
__device__ __forceinline__ uint32_t load2(const uint16_t* ptr) {
  return PASS == 0 ? static_cast<uint32_t>(__ldg(ptr)) : static_cast<uint32_t>(__ldcs(ptr));
}

// ------------------------------------------------------------ row mode tile
template <bool BLOCK2D, bool RHT, bool SR, int PASS>
__device__ __forceinline__ void row_tile(const QParams& p, int64_t tile, uint32_t rht_mask, float s_dec,
                                         uint32_t& tmax) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tr = tile / p.tiles_c, tc = tile - tr * p.tiles_c;
  const int64_t row = tr * 16 + (lane & 15);
  const int64_t kb = tc * 16 + warp * 2 + (lane >> 4);
  const bool valid = row < p.qr && kb < p.kb_count;
  float v[16];
  if (valid) {
    const uint4* src = reinterpret_cast<const uint4*>(p.x + row * p.ldx + kb * 16);
    const uint4 a = load16<PASS>(src);
    const uint4 b = load16<PASS>(src + 1);
    unpack8(a, v);
    unpack8(b, v + 8);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = 0.0f;
  }
  if (RHT) rht16(v, rht_mask);
  uint32_t m = run_absmax_bits(v);
  if (PASS == 0) {
    tmax = max(tmax, m);
    return;
  }
  if (BLOCK2D) {
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  }
  if (!valid) return;
  uint32_t sfb;
  const uint2 c = encode_run<SR>(v, __uint_as_float(m), s_dec, static_cast<uint64_t>(row * p.qk + kb * 16), p, sfb);
  *reinterpret_cast<uint2*>(p.codes + row * (p.qk / 2) + kb * 8) = c;
  p.sf[sf_index(p, row, kb)] = static_cast<uint8_t>(sfb);
}

// ------------------------------------------------------------ col mode tile
template <bool BLOCK2D, bool RHT, bool SR, int PASS>
__device__ __forceinline__ void col_tile(const QParams& p, int64_t tile, uint32_t rht_mask, float s_dec,
                                         uint32_t& tmax) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tr = tile / p.tiles_c, tc = tile - tr * p.tiles_c;
  const int64_t kb = tr * 8 + warp;           // rows 16 kb .. 16 kb + 15 of x
  const int64_t c0 = tc * 64 + 2 * lane;      // columns c0, c0 + 1 of x = rows of Q
  const bool kvalid = kb < p.kb_count;
  const bool v0ok = kvalid && c0 < p.cols;
  const bool v1ok = kvalid && c0 + 1 < p.cols;
  float v0[16], v1[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    uint32_t w = 0;
    const uint16_t* src = p.x + (kb * 16 + j) * p.ldx + c0;
    if (v1ok)
      w = load4<PASS>(reinterpret_cast<const uint32_t*>(src));
    else if (v0ok)
      w = load2<PASS>(src);
    v0[j] = __uint_as_float(w << 16);
    v1[j] = __uint_as_float(w & 0xFFFF0000u);
  }
  if (RHT) {
    rht16(v0, rht_mask);
    rht16(v1, rht_mask);
  }
  uint32_t m0 = run_absmax_bits(v0), m1 = run_absmax_bits(v1);
  if (PASS == 0) {
    tmax = max(tmax, max(m0, m1));
    return;
  }
  if (BLOCK2D) {
    // a 16x16 tile is 16 columns of x = 8 lanes x 2 columns
    m0 = max(m0, m1);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) m0 = max(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, o));
    m1 = m0;
  }
  uint32_t sfb;
  if (v0ok) {
    const uint2 c = encode_run<SR>(v0, __uint_as_float(m0), s_dec, static_cast<uint64_t>(c0 * p.qk + kb * 16), p, sfb);
    *reinterpret_cast<uint2*>(p.codes + c0 * (p.qk / 2) + kb * 8) = c;
    p.sf[sf_index(p, c0, kb)] = static_cast<uint8_t>(sfb);
  }
  if (v1ok) {
    const uint2 c =
        encode_run<SR>(v1, __uint_as_float(m1), s_dec, static_cast<uint64_t>((c0 + 1) * p.qk + kb * 16), p, sfb);
    *reinterpret_cast<uint2*>(p.codes + (c0 + 1) * (p.qk / 2) + kb * 8) = c;
    p.sf[sf_index(p, c0 + 1, kb)] = static_cast<uint8_t>(sfb);
  }
}

__device__ __forceinline__ uint32_t block_max(uint32_t v, uint32_t* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) v = max(v, red[w]);
  return v;
}

template <bool COL, bool BLOCK2D, bool RHT, bool SR, int PASS>
__global__ void __launch_bounds__(kThreads) quant_kernel(const QParams p) {
  __shared__ uint32_t red[kThreads / 32];
  uint32_t rht_mask = 0;
  if (RHT) {
    const uint4 w = philox4x32_10(make_uint4(0u, 0u, 0u, 0u), static_cast<uint32_t>(p.rht_seed),
                                  static_cast<uint32_t>(p.rht_seed >> 32));
    rht_mask = w.x & 0xFFFFu;
  }
  float s_dec = 1.0f;
  if (PASS == 1) {
    uint32_t m = 0;
    for (int i = threadIdx.x; i < p.num_partials; i += kThreads) m = max(m, p.partials[i]);
    m = block_max(m, red);
    if (m >= 0x7F800000u) {  // inf or NaN somewhere in the input
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        ptx::set_status(p.status, kDevNonFinite);
        *p.tensor_scale = __uint_as_float(0x7FC00000u);
      }
      return;
    }
    s_dec = __fdiv_rn(__uint_as_float(m), 2688.0f);
    if (s_dec == 0.0f) s_dec = 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.tensor_scale = s_dec;
  }
  uint32_t tmax = 0;
  for (int64_t it = blockIdx.x; it < p.num_tiles; it += gridDim.x) {
    const int64_t tile = PASS == 1 ? p.num_tiles - 1 - it : it;
    if (COL)
      col_tile<BLOCK2D, RHT, SR, PASS>(p, tile, rht_mask, s_dec, tmax);
    else
      row_tile<BLOCK2D, RHT, SR, PASS>(p, tile, rht_mask, s_dec, tmax);
  }
  if (PASS == 0) {
    tmax = block_max(tmax, red);
    if (threadIdx.x == 0) p.partials[blockIdx.x] = tmax;
  }
}

// Zero the padding of the tensor-core scale layout: rows [qr, pad_r) and
// scale columns [kb_count, pad_kb).
__global__ void sf_pad_kernel(uint8_t* sf, int64_t qr, int64_t kb_count, int64_t pad_r, int64_t pad_kb,
                              int64_t katoms) {
  const int64_t n_rows_pad = (pad_r - qr) * pad_kb;
  const int64_t n_cols_pad = qr * (pad_kb - kb_count);
  const int64_t total = n_rows_pad + n_cols_pad;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int64_t r, kb;
    if (i < n_rows_pad) {
      r = qr + i / pad_kb;
      kb = i % pad_kb;
    } else {
      const int64_t j = i - n_rows_pad;
      const int64_t w = pad_kb - kb_count;
      r = j / w;
      kb = kb_count + j % w;
    }
    const int64_t atom = (r >> 7) * katoms + (kb >> 2);
    const int rr = static_cast<int>(r & 127);
    sf[atom * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + static_cast<int>(kb & 3)] = 0;
  }
}

template <bool COL, bool BLOCK2D, bool RHT, bool SR, int PASS>
int grid_for(int64_t num_tiles) {
  static int per_sm = -1;
  if (per_sm < 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, quant_kernel<COL, BLOCK2D, RHT, SR, PASS>, kThreads, 0) !=
            cudaSuccess ||
        b < 1)
      b = 1;
    per_sm = b;
  }
  int64_t g = static_cast<int64_t>(per_sm) * device_sm_count();
  g = std::min<int64_t>(g, kMaxAmaxPartials);
  g = std::min<int64_t>(g, std::max<int64_t>(num_tiles, 1));
  return static_cast<int>(std::max<int64_t>(g, 1));
}

template <bool COL, bool BLOCK2D, bool RHT, bool SR>
cudaError_t run_passes(QParams p, cudaStream_t stream) {
  const int g0 = grid_for<COL, false, RHT, false, 0>(p.num_tiles);
  p.num_partials = g0;
  quant_kernel<COL, false, RHT, false, 0><<<g0, kThreads, 0, stream>>>(p);
  const int g1 = grid_for<COL, BLOCK2D, RHT, SR, 1>(p.num_tiles);
  quant_kernel<COL, BLOCK2D, RHT, SR, 1><<<g1, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

template <bool COL, bool BLOCK2D, bool RHT>
cudaError_t dispatch_sr(const QParams& p, int sr, cudaStream_t s) {
  return sr ? run_passes<COL, BLOCK2D, RHT, true>(p, s) : run_passes<COL, BLOCK2D, RHT, false>(p, s);
}
template <bool COL, bool BLOCK2D>
cudaError_t dispatch_rht(const QParams& p, int rht, int sr, cudaStream_t s) {
  return rht ? dispatch_sr<COL, BLOCK2D, true>(p, sr, s) : dispatch_sr<COL, BLOCK2D, false>(p, sr, s);
}
template <bool COL>
cudaError_t dispatch_block(const QParams& p, int b2d, int rht, int sr, cudaStream_t s) {
  return b2d ? dispatch_rht<COL, true>(p, rht, sr, s) : dispatch_rht<COL, false>(p, rht, sr, s);
}

// Scratch for nvfp4_quantize_noalloc: the status word (first 256 bytes) and
// the partial-amax slots of the amax pass, in one file-scope device array.
// Every GPU that loads the library holds it until the process exits.  In
// host code `g_noalloc_scratch` only names the symbol; its device address
// comes from cudaGetSymbolAddress, once per device.
constexpr size_t kNoAllocScratchBytes = kWsHeaderBytes + kQuantScratchBytes;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

}  // namespace

cudaError_t noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return cudaSuccess;
}

cudaError_t launch_quantize_noalloc(QuantArgs a, cudaStream_t stream) {
  void* scratch = nullptr;
  cudaError_t e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) return e;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  // The status word must start at zero; the partial slots are fully written
  // by the amax pass before the encode pass reads them.
  e = cudaMemsetAsync(base, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  a.status = reinterpret_cast<uint32_t*>(base);
  a.partials = reinterpret_cast<uint32_t*>(base + kWsHeaderBytes);
  return launch_quantize(a, stream);
}

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t stream) {
  QParams p{};
  p.x = a.x;
  p.rows = a.rows;
  p.cols = a.cols;
  p.ldx = a.ldx;
  p.qr = a.qr;
  p.qk = a.qk;
  p.kb_count = a.qk / 16;
  p.codes = a.codes;
  p.sf = a.sf;
  p.tensor_scale = a.tensor_scale;
  p.status = a.status;
  p.partials = a.partials;
  p.rht_seed = a.rht_seed;
  p.sr_seed = a.sr_seed;
  p.sr_offset = a.sr_offset;
  p.sf_mma = a.sf_mma;
  p.sf_katoms = (p.kb_count + 3) / 4;
  int64_t tiles_r;
  if (!a.transpose) {
    tiles_r = (p.qr + 15) / 16;
    p.tiles_c = (p.kb_count + 15) / 16;
  } else {
    tiles_r = (p.kb_count + 7) / 8;
    p.tiles_c = (p.qr + 63) / 64;
  }
  p.num_tiles = tiles_r * p.tiles_c;
  cudaError_t err = a.transpose ? dispatch_block<true>(p, a.block2d, a.rht, a.sr, stream)
                                : dispatch_block<false>(p, a.block2d, a.rht, a.sr, stream);
  if (err != cudaSuccess) return err;
  if (a.sf_mma) {
    const int64_t pad_r = (p.qr + 127) / 128 * 128;
    const int64_t pad_kb = p.sf_katoms * 4;
    const int64_t total = (pad_r - p.qr) * pad_kb + p.qr * (pad_kb - p.kb_count);
    if (total > 0) {
      const int64_t blocks = std::min<int64_t>((total + 255) / 256, 4 * device_sm_count());
      sf_pad_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(p.sf, p.qr, p.kb_count, pad_r, pad_kb,
                                                                  p.sf_katoms);
      err = cudaGetLastError();
    }
  }
  return err;
}

}  // namespace nvfp4
