// NVFP4 encoding steps shared by the quantiser, the GEMM's quantising epilogue
// and the optimizer-state codec: the E4M3 block scale of a run of 16, the
// exact element division that precedes rounding onto the E2M1 grid, the
// Philox4x32-10 stream and the stochastic-rounding decision.
//
//   t = (bamax / 6) / s -> E4M3 (round to nearest even, saturating at 448),
//   d = e4m3(t) * s,  v = x / d (IEEE quotient).
//
// Every FP32 step is written as an explicit round-to-nearest intrinsic, so the
// results do not depend on the translation unit's contraction setting.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace nvfp4 {

// E4M3 block-scale byte of a run whose largest magnitude has FP32 bits
// `bamax_bits`, under the FP32 tensor scale s_dec.
__device__ __forceinline__ uint32_t block_scale_byte(uint32_t bamax_bits, float s_dec) {
  return ptx::cvt_e4m3(__fdiv_rn(__fdiv_rn(__uint_as_float(bamax_bits), 6.0f), s_dec));
}

// x / d for 2^-70 <= d < 2^126, given rd = RN(1/d): q0 = RN(x * rd) is
// within one ulp of x / d, and one residual correction q0 + RN(x - q0 d) * rd
// with an exact FMA residual rounds to the IEEE quotient (Markstein's
// division theorem; P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34, 1990), as long
// as nothing underflows: |x| >= 2^-96 and |q| >= 2^-100.  Outside that range
// the quotient is below 2^-25, where an RNE code is +-0 whatever its exact
// value and stochastic rounding only asks whether it is zero (divide_run
// keeps that answer exact by its choice of path).
__device__ __forceinline__ float div_fast(float x, float d, float rd) {
  const float q0 = __fmul_rn(x, rd);
  // (q0 d - x) is the negated residual; q0 - that * rd keeps the sign of a
  // zero x: for x = -0 both terms are -0, and the sum of two -0 is -0.
  return __fmaf_rn(-__fmaf_rn(q0, d, -x), rd, q0);
}

// The same block-scale byte with the two divisions done as residual-corrected
// divisions by constant reciprocals (RN(1/6) and rs = RN(1/s_dec), rs = 0 when
// s_dec is outside [2^-70, 2^126)): exact where div_fast is, which the
// condition bamax >= 2^-93 secures for both steps (then bamax / 6 >= 2^-96);
// a quotient below 2^-100 is below the smallest E4M3 step whatever its last
// bits, and one above 2^100 (or an overflow) is clamped there, where E4M3
// saturates at 448 anyway.  Elsewhere IEEE divisions.
__device__ __forceinline__ uint32_t block_scale_byte_rcp(uint32_t bamax_bits, float s_dec, float rs) {
  const float x = __uint_as_float(bamax_bits);
  float t;
  if (rs != 0.0f && x >= 0x1p-93f) {
    t = div_fast(div_fast(x, 6.0f, 0x1.555556p-3f), s_dec, rs);
    t = (t <= 0x1p100f) ? t : 0x1p100f;
  } else {
    t = __fdiv_rn(__fdiv_rn(x, 6.0f), s_dec);
  }
  return ptx::cvt_e4m3(t);
}

// q[j] = v[j] / d wherever the quotient can change a code.  Fast division
// where it is exact for every code (see div_fast): d in [2^-70, 2^126) for
// round-to-nearest.  Stochastic rounding (SR) also needs the zero-ness of
// quotients below 2^-25: every nonzero input (a BF16 value, or a transform of
// BF16 values) is at least 2^-135 in magnitude, so for d < 2^14 every such
// quotient and its fast approximation are nonzero.  Elsewhere IEEE division.
template <bool SR>
__device__ __forceinline__ void divide_run(const float (&v)[16], float d, float (&q)[16]) {
  const bool fast = d >= 0x1p-70f && d < (SR ? 0x1p14f : 0x1p126f);
  if (fast) {
    const float rd = __frcp_rn(d);
#pragma unroll
    for (int j = 0; j < 16; ++j) q[j] = div_fast(v[j], d, rd);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) q[j] = __fdiv_rn(v[j], d);
  }
}

// Largest |v| of a run as FP32 bits, with NaN propagated (max.NaN), so that
// a non-finite run shows as bits >= 0x7F800000.
__device__ __forceinline__ uint32_t run_absmax_nan(const float (&v)[16]) {
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) asm("max.NaN.f32 %0, %0, %1;" : "+f"(m) : "f"(fabsf(v[j])));
  return __float_as_uint(m);
}

__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

// Philox4x32-10 (Salmon et al., SC'11): ten rounds; the Weyl key schedule is
// precomputed on the host (sr_rk0 / sr_rk1).
__device__ __forceinline__ uint4 philox4x32_10_rk(uint4 c, const uint32_t (&rk0)[10], const uint32_t (&rk1)[10]) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c.z;
    c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ rk0[i], static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ c.w ^ rk1[i], static_cast<uint32_t>(p0));
  }
  return c;
}

// Stochastic rounding of q onto the E2M1 grid {0, .5, 1, 1.5, 2, 3, 4, 6}:
// lo, hi the grid points around |q|, f = (|q| - lo) / (hi - lo), round up iff
// k * 2^-24 < f with k = r >> 8; |q| >= 6 -> 6.  Branch-free, with b the
// magnitude bits of q and m its 23 mantissa bits:
//   |q| in [1, 6): the grid points are the values whose 22 mantissa bits
//     below the top one are zero and f * 2^24 = 4 * (those bits), so
//     k < f * 2^24 iff adding 2^22 - 1 - (r >> 10) to b carries into the
//     grid bit;
//   |q| in [1/2, 1): lo = 1/2, hi = 1 and f * 2^24 = 2 m, so k < 2 m iff
//     adding 2^23 - 1 - (r >> 9) to b carries into the exponent;
//   |q| in [0, 1/2): lo = 0, f * 2^24 = |q| * 2^25, exact in FP32, compared
//     with k (< 2^24, exact as a float).
// The shifts of r are taken as high halves of products (r * 2^(32-s)), and
// every |q| >= 6 (inf and NaN included) lands at or above the bits of 6, so
// one unsigned min saturates.  Returns the grid value with the sign of q.
__device__ __forceinline__ float sr_round(float q, uint32_t rnd) {
  const uint32_t qb = __float_as_uint(q);
  const uint32_t b = qb & 0x7FFFFFFFu;
  const uint32_t g_hi = (b + 0x3FFFFFu - __umulhi(rnd, 1u << 22)) & 0xFFC00000u;
  const uint32_t g_mid = (b + 0x7FFFFFu - __umulhi(rnd, 1u << 23)) & 0xFF800000u;
  const bool up0 = __uint2float_rn(__umulhi(rnd, 1u << 24)) < __fmul_rn(__uint_as_float(b), 33554432.0f);
  const uint32_t g_low = up0 ? 0x3F000000u : 0u;
  uint32_t g = b >= 0x3F800000u ? g_hi : (b >= 0x3F000000u ? g_mid : g_low);
  g = min(g, 0x40C00000u);
  return __uint_as_float(g | (qb & 0x80000000u));
}

}  // namespace nvfp4
