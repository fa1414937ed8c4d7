// NVFP4 quantisation of BF16 tensors (sm_103a).
//
// One call reads x [rows, cols] and writes one or two quantised outputs, each
// either Q = x (blocks of 16 along a row of x) or Q = x^T (blocks of 16 down a
// column of x), each with its own block shape, rounding, transform and tensor
// scale.  A linear layer needs both orientations of X and dY (fprop/dgrad use
// rows, wgrad uses columns) and of W (fprop, dgrad), so producing both from one
// read halves the quantiser's input traffic.
//
// The general form is two kernels, both persistent loops over 128 x 128 tiles
// of x that TMA copies into shared memory (two 64-column boxes, 128-byte
// swizzle; a ring of three stages in the amax pass, two in the encode pass):
//   pass 0: per-output tensor amax (after the optional random Hadamard
//           transform, in the output's orientation); one partial per CTA;
//   pass 1: every CTA reduces the partials, derives s = amax / 2688 and encodes
//           its tiles.  It walks the tiles in reverse order, so its first
//           reads hit the part of x that pass 0 left in L2.
// Under delayed scaling (a supplied amax for every output) pass 0 is not
// launched and pass 1 takes s from that amax: one read of x.  A single row
// output needs no tile at all: its encode pass is the streaming kernel
// quant_rows (except 16x16 blocks with round-to-nearest and no transform,
// which the staged tile serves faster).  Two outputs in
// 16x16 blocks with round-to-nearest, one per orientation (a weight's pair),
// hold the same codes transposed within each 16x16 tile: the transposed one
// is copied from the other's staged tile instead of encoded (mirror_tile).
// Where no tile is needed the passes stream runs of 16 straight from global
// memory instead, as many CTAs as are resident at once: quant_rows (the
// encode of a single row output), amax_rows (an amax of x itself) and
// amax_cols_pair (both amaxes of an activation's pair, down the columns).
// Out-of-range parts of a tile read as zero, so ragged tiles need no special
// case and the padding of the tensor-core scale layout comes out as zeros.
//
// Format and rounding sequence (per run of 16 along K; the pages' NVFP4
// elements on a sparse 4-bit grid with custom scaling, "NVIDIA acelera o
// pre-treinamento de LLM: NVFP4 no Blackwell...", section "Por que cada
// porcento e importante"; Hadamard mixing and stochastic rounding from
// "Full-Stack FP4...", section 2.2):
//   t = (bamax / 6) / s -> E4M3 (RNE, saturating), d = e4m3(t) * s,
//   v = x / d -> E2M1 by RNE or by stochastic rounding with a Philox4x32-10
//   word per element.  Every FP32 step is an IEEE round-to-nearest operation
//   (the file is built without FMA contraction).  The element division uses a
//   correctly rounded reciprocal (from a per-CTA table indexed by the scale
//   byte) and one FMA residual correction, which gives the IEEE quotient
//   wherever it can change a code (div_fast in encode.cuh); the block
//   scale's two divisions use the same scheme with the constant reciprocals
//   of 6 and of s (block_scale_byte_rcp).
//
// Thread layout: one thread owns whole runs of 16, so the transform and the
// block maximum stay in registers.  Thread t works on position p = t & 127
// (a tile row for Q = x, a tile column for Q = x^T) and runs j = (t >> 7) +
// 2i, i = 0..3; a warp's lanes are 32 consecutive positions of one run, so a
// 16 x 16 block is 16 adjacent lanes and the 128-byte swizzle keeps both read
// patterns free of bank conflicts.  Results are staged in shared memory and
// leave in whole 32-byte pieces.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "encode.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 128;                      // tile: 128 rows x 128 columns of x
constexpr int kBoxBytes = kTile * 128;          // one TMA box: 64 BF16 columns x 128 rows
constexpr int kStageBytes = 2 * kBoxBytes;      // 32 KB
// TMA ring depth: the encode pass keeps two stages (its staging buffers
// fill the rest of two CTAs' shared memory per SM); the amax pass has no
// staging and keeps three tiles in flight.
template <int PASS>
__host__ __device__ constexpr int stages_of() {
  return PASS == 0 ? 3 : 2;
}
// Per output, a tile's results are staged in shared memory before they go to
// global memory in whole 32-byte pieces: codes of position p, run j at
// p * 72 + 8 j (the 72-byte pitch spreads a warp's stores over the banks);
// scales as the two 128 x 4 atoms of the tensor-core layout.  Two staging
// buffers per output follow the ring.
constexpr int kStgPitch = 72;
constexpr int kStgCodes = kTile * kStgPitch;    // 9216
constexpr int kStgBytes = kStgCodes + 2 * 512;  // + scales
constexpr int kStgOffset = stages_of<1>() * kStageBytes;
template <int PASS>
constexpr int smem_bytes() {  // + slack to align to 1024 B
  return PASS == 0 ? stages_of<0>() * kStageBytes + 1024 : kStgOffset + 2 * kMaxQuantOutputs * kStgBytes + 1024;
}

struct OutParams {
  uint8_t* codes;
  uint8_t* sf;
  float* tensor_scale;
  uint32_t* partials;
  const float* amax_in;  // supplied amax (delayed scaling), or null: scan the operand
  int64_t qr, qk, code_ld, kb_count, katoms;
  uint64_t rht_seed, sr_seed, sr_offset;
  // Philox key schedule of sr_seed, one pair per round (parameter space, so
  // the round XORs read them as constant operands)
  uint32_t sr_rk0[10], sr_rk1[10];
  // transform signs: sigma_j = -1 as 0x80000000 (the FP32 sign bit), else 0
  uint32_t rht_sgn[16];
  int col, block2d, sr, rht, sf_mma, vec16;
};

struct TileParams {
  int64_t tiles_c, num_tiles;
  OutParams out[kMaxQuantOutputs];
  int n_out;
  int amax_shared;  // two outputs, neither transformed: output 1 reuses output 0's amax
  int mirror;       // -1, or the output copied from the other's staged tile (see mirror_tile)
  int amax_pair;    // -1, or the transformed column output whose sweep also gives the other's amax
  int num_partials;
  int skip_first_load;  // test hook: CTA 0 of this pass never loads its first tile
  uint32_t* status;
};


// x' = 1/4 * H16 * (diag(sigma) x) for a run whose signs were applied as it
// was loaded (load_run with SIGNED: flipping the sign bit is the exact product
// by -1, zeros included); butterflies of stride 1, 2, 4, 8, then the exact
// scaling by 1/4.
__device__ __forceinline__ void hadamard16(float (&v)[16]) {
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

// Largest |x'| of x' = 1/4 * H16 * v (v with the transform's signs already
// applied) as FP32 bits, for the amax passes, without forming x': the last
// butterfly's two outputs RN(a + b) and RN(a - b) have the larger magnitude
// RN(|a| + |b|) (rounding to nearest is monotonic and odd), and the exact
// scaling by 1/4 may follow the maximum because RN(m / 4) is monotonic in m.
// Equal to run_absmax_bits after hadamard16 bit for bit on finite runs; a run
// holding an infinity or NaN gives a value at or above the bits of infinity
// either way, which is all the amax pass tests.
__device__ __forceinline__ uint32_t hadamard16_absmax_bits(float (&v)[16]) {
#pragma unroll
  for (int s = 1; s < 8; s <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & s) continue;
      const float a = v[i], b = v[i + s];
      v[i] = __fadd_rn(a, b);
      v[i + s] = __fsub_rn(a, b);
    }
  }
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = max(m, abs_bits(__fadd_rn(fabsf(v[i]), fabsf(v[i + 8]))));
  return abs_bits(__fmul_rn(__uint_as_float(m), 0.25f));
}

// Largest |v| of a run as FP32 bits; inf and NaN sort above every finite
// value, which is how the amax pass detects them.
__device__ __forceinline__ uint32_t run_absmax_bits(const float (&v)[16]) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) m = max(m, abs_bits(v[j]));
  return m;
}

// Per-output divisor table, built once per CTA: for every nonzero finite
// scale byte b, d = e4m3(b) * s and rd = RN(1/d) where the fast division is
// exact for this rounding mode (rd = 0 elsewhere: IEEE division).
struct DivTable {
  float2 e[128];
};

// Encode one run of 16 values (already transformed) with block maximum
// `bamax_bits`; e0 is the linear index of the run's first element in Q, the
// Philox counter of element e being e >> 2 (word e & 3).
template <bool SR>
__device__ __forceinline__ uint2 encode_run(const float (&v)[16], uint32_t bamax_bits, float s_dec, float rs,
                                            const DivTable& dt, uint64_t e0, const OutParams& o, uint32_t& sfb) {
  sfb = block_scale_byte_rcp(bamax_bits, s_dec, rs);
  if (sfb == 0) return make_uint2(0u, 0u);
  const float2 dd = dt.e[sfb];
  float q[16];
  if (dd.y != 0.0f) {
#pragma unroll
    for (int j = 0; j < 16; ++j) q[j] = div_fast(v[j], dd.x, dd.y);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) q[j] = __fdiv_rn(v[j], dd.x);
  }
  if (SR) {
    const uint32_t o0 = static_cast<uint32_t>(o.sr_offset), o1 = static_cast<uint32_t>(o.sr_offset >> 32);
    const uint64_t c = e0 >> 2;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint64_t cg = c + g;
      const uint4 w =
          philox4x32_10_rk(make_uint4(static_cast<uint32_t>(cg), static_cast<uint32_t>(cg >> 32), o0, o1), o.sr_rk0,
                           o.sr_rk1);
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

// ----------------------------------------------------------- tile loaders
// Stage layout: box h (tile columns 64h .. 64h + 63) at h * 16 KB; tile row r
// at r * 128 bytes within the box; its 16-byte chunk c at ((c ^ (r & 7)) * 16).
//
// Run j (0..7) of position p (0..127): for Q = x, tile columns 16j .. 16j+15
// of tile row p; for Q = x^T, tile rows 16j .. 16j+15 of tile column p.
// SIGNED: element i also gets the sign bit sgn[i] (0 or 0x80000000) of the
// transform's sigma, folded into the widening as h * 2^16 + sgn (the low
// sixteen bits are zero, so the add is an exact sign flip).
template <bool COL, bool SIGNED = false>
__device__ __forceinline__ void load_run(const uint8_t* stage, int p, int j, float (&v)[16],
                                         const uint32_t* sgn = nullptr) {
  if (!COL) {
    const uint8_t* rowp = stage + (j >> 2) * kBoxBytes + p * 128;
    const int c = 2 * (j & 3), sw = p & 7;
    const uint4 a = *reinterpret_cast<const uint4*>(rowp + ((c ^ sw) << 4));
    const uint4 b = *reinterpret_cast<const uint4*>(rowp + (((c + 1) ^ sw) << 4));
    unpack8(a, v);
    unpack8(b, v + 8);
    if (SIGNED) {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(__float_as_uint(v[i]) ^ sgn[i]);
    }
  } else {
    const uint8_t* colp = stage + (p >> 6) * kBoxBytes + j * 16 * 128 + (p & 7) * 2;
    const int c = (p & 63) >> 3;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t h = *reinterpret_cast<const uint16_t*>(colp + i * 128 + ((c ^ (i & 7)) << 4));
      v[i] = __uint_as_float(SIGNED ? h * 65536u + sgn[i] : h << 16);
    }
  }
}

// ------------------------------------------------------------ amax pass
template <bool COL>
__device__ __forceinline__ uint32_t amax_tile(const uint8_t* stage, bool rht, const uint32_t* sgn) {
  const int p = threadIdx.x & 127, j0 = threadIdx.x >> 7;
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float v[16];
    if (rht) {
      load_run<COL, true>(stage, p, j0 + 2 * i, v, sgn);
      m = max(m, hadamard16_absmax_bits(v));
    } else {
      load_run<COL>(stage, p, j0 + 2 * i, v);
      m = max(m, run_absmax_bits(v));
    }
  }
  return m;
}

// Both amaxes of a pair whose output `rht` is transformed down the columns
// and whose other output is not transformed, from one sweep: the column runs
// are loaded with the transform's signs folded in, which leaves |x| as it is,
// so their maximum before the transform is the untransformed amax.
__device__ __forceinline__ void amax_tile_pair(const uint8_t* stage, const uint32_t* sgn, uint32_t& m_raw,
                                               uint32_t& m_rht) {
  const int p = threadIdx.x & 127, j0 = threadIdx.x >> 7;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float v[16];
    load_run<true, true>(stage, p, j0 + 2 * i, v, sgn);
    m_raw = max(m_raw, run_absmax_bits(v));
    m_rht = max(m_rht, hadamard16_absmax_bits(v));
  }
}

// ------------------------------------------------------------ encode pass
__device__ __forceinline__ int stg_sf_offset(int p, int j) {
  return kStgCodes + (j >> 2) * 512 + (p & 31) * 16 + (p >> 5) * 4 + (j & 3);
}

template <bool COL, bool SR>
__device__ __forceinline__ void encode_tile(const uint8_t* stage, uint8_t* stg, const OutParams& o, float s_dec,
                                            float rs, const DivTable& dt, int64_t tr,
                                            int64_t tc, uint32_t* status) {
  const int p = threadIdx.x & 127, j0 = threadIdx.x >> 7;
  const int64_t qrow = (COL ? tc : tr) * kTile + p;
  const int64_t kb0 = (COL ? tr : tc) * 8;
  // two runs per iteration for instruction-level parallelism, one on the
  // longer stochastic-rounding path
#pragma unroll(SR ? 1 : 2)
  for (int i = 0; i < 4; ++i) {
    const int j = j0 + 2 * i;
    float v[16];
    if (o.rht) {
      load_run<COL, true>(stage, p, j, v, o.rht_sgn);
      hadamard16(v);
    } else {
      load_run<COL>(stage, p, j, v);
    }
    // Inf and NaN were ruled out by the amax pass, except under a supplied
    // amax, where the operand is not scanned first: a non-finite run is
    // reported here (its codes are unspecified).
    uint32_t m = run_absmax_nan(v);
    if (o.block2d) {
#pragma unroll
      for (int x = 1; x < 16; x <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, x));
    }
    if (m >= 0x7F800000u) ptx::set_status(status, kDevNonFinite);
    uint32_t sfb;
    const uint2 c =
        encode_run<SR>(v, m, s_dec, rs, dt, static_cast<uint64_t>(qrow * o.qk + (kb0 + j) * 16), o, sfb);
    *reinterpret_cast<uint2*>(stg + p * kStgPitch + 8 * j) = c;
    stg[stg_sf_offset(p, j)] = static_cast<uint8_t>(sfb);
  }
}

// Output Q = x^T from the staged Q = x of the same tile when both use 16x16
// blocks and round-to-nearest under one tensor scale: element (r, c) then has
// the same block scale and the same code in both, so position p, run j of the
// transposed output is nibble p & 15 of run p >> 4 in the sixteen staged rows
// 16 j .. 16 j + 15 (element k of a run sits in nibble k), and its scale
// byte is that block's.  Rows and columns past the tensor carry what the
// zero fill gave the row output, as an encode of them would.
__device__ __forceinline__ void mirror_tile(const uint8_t* src, uint8_t* dst) {
  // Thread t: columns 4 cg .. 4 cg + 3 (cg = t & 31) of row group j = t >> 5,
  // which are nibbles 4 (cg & 3) .. + 3 of run cg >> 2 of each source row: one
  // 16-bit load per row gives all four (element k in nibble k, little-endian).
  const int cg = threadIdx.x & 31, j = threadIdx.x >> 5;
  const uint8_t* rows = src + 16 * j * kStgPitch + 8 * (cg >> 2) + 2 * (cg & 3);
  uint32_t w[4][2] = {{0u, 0u}, {0u, 0u}, {0u, 0u}, {0u, 0u}};
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint32_t h = *reinterpret_cast<const uint16_t*>(rows + e * kStgPitch);
#pragma unroll
    for (int c = 0; c < 4; ++c) w[c][e >> 3] |= ((h >> (4 * c)) & 0xFu) << (4 * (e & 7));
  }
  const uint32_t sf = src[stg_sf_offset(16 * j, cg >> 2)];  // the block's scale byte
  // stores staggered by cg, so a warp's stores spread over the banks: step i
  // writes column 4 cg + ((i + cg) & 3), its words picked by selects (a
  // runtime index into w would put it in local memory)
  const int r = cg & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = (i + r) & 3;
    uint2 v = make_uint2(w[0][0], w[0][1]);
    if (c == 1) v = make_uint2(w[1][0], w[1][1]);
    if (c == 2) v = make_uint2(w[2][0], w[2][1]);
    if (c == 3) v = make_uint2(w[3][0], w[3][1]);
    const int p = 4 * cg + c;
    *reinterpret_cast<uint2*>(dst + p * kStgPitch + 8 * j) = v;
    dst[stg_sf_offset(p, j)] = static_cast<uint8_t>(sf);
  }
}

// Staged tile -> global memory.  Thread t copies the codes of runs 4 (t & 1)
// .. + 3 of position t >> 1; the first 64 threads copy the two scale atoms.
// Rows of Q past qr and blocks past kb_count are not written, except that the
// tensor-core scale layout receives its zero padding.
__device__ __forceinline__ void copy_out(const uint8_t* stg, const OutParams& o, int64_t qrow0, int64_t kb0) {
  const int t = threadIdx.x;
  const int p = t >> 1, half = t & 1;
  const int64_t qrow = qrow0 + p;
  const int64_t kb = kb0 + 4 * half;
  if (qrow < o.qr && kb < o.kb_count) {
    const uint8_t* src = stg + p * kStgPitch + 32 * half;
    uint2 w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const uint2*>(src + 8 * i);
    uint8_t* dst = o.codes + qrow * o.code_ld + kb * 8;
    if (o.vec16 && kb + 4 <= o.kb_count) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0].x, w[0].y, w[1].x, w[1].y);
      *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[2].x, w[2].y, w[3].x, w[3].y);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (kb + i < o.kb_count) *reinterpret_cast<uint2*>(dst + 8 * i) = w[i];
    }
  }
  if (o.sf_mma) {
    if (t < 64) {
      const int64_t katom = (kb0 >> 2) + (t >> 5);
      if (katom < o.katoms)
        *reinterpret_cast<uint4*>(o.sf + ((qrow0 >> 7) * o.katoms + katom) * 512 + (t & 31) * 16) =
            *reinterpret_cast<const uint4*>(stg + kStgCodes + t * 16);
    }
  } else if (qrow < o.qr) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (kb + i < o.kb_count) o.sf[qrow * o.kb_count + kb + i] = stg[stg_sf_offset(p, 4 * half + i)];
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

// Encode pass for a single row output (Q = x).  Its runs share nothing
// across rows except the maximum of a 16x16 block, so no tile is staged:
// each thread streams whole runs of 16 straight from global memory (two
// 16-byte loads, the transform's signs folded in as the tiled loader does)
// and stores their codes and scale bytes directly, with the whole grid -- as
// many CTAs as are resident at once -- walking the runs backwards (the amax
// pass leaves the end of x in L2).  With 16x16 blocks the 16 lanes of a
// half-warp take the 16 rows of one block and share its maximum by shuffles.
// The walk covers the tensor-core scale layout's padding rows and blocks
// too, which receive zero scale bytes.  Same arithmetic, tensor scale and
// error reporting as the tiled encode pass.  (Two runs per iteration, or a
// grid of eight CTAs per SM, measured slower.)
template <bool SR, bool RHT, bool BLOCK2D>
__global__ void __launch_bounds__(kThreads) quant_rows(const uint16_t* __restrict__ x, int64_t ldx,
                                                      const TileParams p) {
  __shared__ uint32_t red[kThreads / 32];
  __shared__ DivTable dtab;
  const OutParams& o = p.out[0];
  const int tid = threadIdx.x;
  uint32_t m = 0;
  if (o.amax_in) {
    const float a = *o.amax_in;
    m = (a >= 0.0f) ? __float_as_uint(fabsf(a)) : 0x7FC00000u;
  } else {
    for (int i = tid; i < p.num_partials; i += kThreads) m = max(m, o.partials[i]);
    m = block_max(m, red);
  }
  if (m >= 0x7F800000u) {  // inf or NaN in the input (or a bad supplied amax)
    if (blockIdx.x == 0 && tid == 0) {
      ptx::set_status(p.status, kDevNonFinite);
      *o.tensor_scale = __uint_as_float(0x7FC00000u);
    }
    return;
  }
  float s = __fdiv_rn(__uint_as_float(m), 2688.0f);
  if (s == 0.0f) s = 1.0f;
  const float rs = (s >= 0x1p-70f && s < 0x1p126f) ? __frcp_rn(s) : 0.0f;
  if (blockIdx.x == 0 && tid == 0) *o.tensor_scale = s;
  if (tid >= 1 && tid < 127) {
    const float d = __fmul_rn(ptx::e4m3_to_float(static_cast<uint32_t>(tid)), s);
    const bool fast = d >= 0x1p-70f && d < (SR ? 0x1p14f : 0x1p126f);
    dtab.e[tid] = make_float2(d, fast ? __frcp_rn(d) : 0.0f);
  }
  __syncthreads();
  // Work items: runs (1x16), or 16-row groups of runs (16x16, the group's row
  // the thread's lane & 15, constant because the stride is a multiple of 16).
  constexpr int G = BLOCK2D ? 16 : 1;
  const int64_t rows_pad = o.sf_mma ? (o.qr + 127) / 128 * 128 : o.qr;
  const int64_t kb_pad = o.sf_mma ? o.katoms * 4 : o.kb_count;
  const int64_t total = rows_pad / G * kb_pad;
  if (total == 0) return;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (kThreads / G);
  const int rr = BLOCK2D ? (tid & 15) : 0;
  // Items are counted from the end: item i sits at r = total - 1 - i, row
  // group r / kb_pad, block r % kb_pad.  One division per thread; each step
  // back by the grid's stride then subtracts (stride / kb_pad, stride %
  // kb_pad) with a borrow.
  const int64_t step_rows = stride / kb_pad, step_kb = stride - step_rows * kb_pad;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * (kThreads / G) + tid / G;
  int64_t rg = (total - 1 - i0) / kb_pad;
  int64_t kb = (total - 1 - i0) - rg * kb_pad;
  const unsigned group_mask = BLOCK2D ? (0xFFFFu << (tid & 16)) : 0xFFFFFFFFu;
  for (int64_t i = i0; i < total; i += stride) {
    const int64_t row = rg * G + rr;
    const bool in = row < o.qr && kb < o.kb_count;  // uniform over a 16x16 block's lanes
    uint32_t sfb = 0u;
    if (in) {
      const uint4* src = reinterpret_cast<const uint4*>(x + row * ldx + kb * 16);
      float v[16];
      unpack8(__ldcs(src), v);
      unpack8(__ldcs(src + 1), v + 8);
      if (RHT) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(__float_as_uint(v[j]) ^ o.rht_sgn[j]);
        hadamard16(v);
      }
      uint32_t bm = run_absmax_nan(v);
      if (BLOCK2D) {
#pragma unroll
        for (int sh = 1; sh < 16; sh <<= 1) bm = max(bm, __shfl_xor_sync(group_mask, bm, sh));
      }
      if (bm >= 0x7F800000u) ptx::set_status(p.status, kDevNonFinite);  // codes unspecified
      const uint2 c =
          encode_run<SR>(v, bm, s, rs, dtab, static_cast<uint64_t>(row * o.qk + kb * 16), o, sfb);
      *reinterpret_cast<uint2*>(o.codes + row * o.code_ld + kb * 8) = c;
    }
    if (o.sf_mma)
      o.sf[((row >> 7) * o.katoms + (kb >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (kb & 3)] =
          static_cast<uint8_t>(sfb);
    else if (in)
      o.sf[row * o.kb_count + kb] = static_cast<uint8_t>(sfb);
    rg -= step_rows;
    kb -= step_kb;
    if (kb < 0) {
      kb += kb_pad;
      --rg;
    }
  }
}

// Amax pass when the amax is that of x itself (no transform): each thread
// streams whole runs of 16 along the rows of x, as the streaming encode
// does, and each CTA writes one partial maximum.  Runs are walked forwards,
// so the end of x is what stays in L2 for the encode pass, which walks
// backwards.  (With the transform along the rows it measured 1-2 % slower
// than the tiled amax pass, which keeps that case.)
__global__ void __launch_bounds__(kThreads) amax_rows(const uint16_t* __restrict__ x, int64_t ldx,
                                                     const TileParams p) {
  __shared__ uint32_t red[kThreads / 32];
  const OutParams& o = p.out[0];
  const int64_t kbs = o.col ? o.qr / 16 : o.kb_count;  // runs of 16 along a row of x (cols % 16 == 0)
  const int64_t rows = o.col ? o.qk : o.qr;             // rows of x
  const int64_t total = rows * kbs;
  uint32_t m = 0;
  if (total > 0) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t step_rows = stride / kbs, step_kb = stride - step_rows * kbs;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    int64_t row = i0 / kbs, kb = i0 - row * kbs;
    for (int64_t i = i0; i < total; i += stride) {
      const uint4* src = reinterpret_cast<const uint4*>(x + row * ldx + kb * 16);
      float v[16];
      unpack8(src[0], v);
      unpack8(src[1], v + 8);
      m = max(m, run_absmax_bits(v));
      row += step_rows;
      kb += step_kb;
      if (kb >= kbs) {
        kb -= kbs;
        ++row;
      }
    }
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) o.partials[blockIdx.x] = m;
}

// Amax pass of an activation pair (amax_tile_pair's case: output t is
// transformed down the columns, the other output is not transformed) without
// a tile: each thread takes two adjacent columns of a 16-row group (one
// 4-byte load per row, so a warp reads 128 contiguous bytes of each row),
// folds the transform's signs in, and keeps the largest |x| before the
// transform (the untransformed amax) and after it (the transformed one).
// Each CTA writes one partial per output.  Forwards, like amax_rows.
__global__ void __launch_bounds__(kThreads) amax_cols_pair(const uint16_t* __restrict__ x, int64_t ldx,
                                                          int64_t rows, int64_t cols, const TileParams p) {
  __shared__ uint32_t red[kThreads / 32];
  const int t = p.amax_pair;
  const uint32_t* sgn = p.out[t].rht_sgn;
  const int64_t pairs = cols / 2;
  const int64_t total = rows / 16 * pairs;
  uint32_t m_raw = 0, m_rht = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t step_grp = stride / pairs, step_cp = stride - step_grp * pairs;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  int64_t grp = i0 / pairs, cp = i0 - grp * pairs;
  for (int64_t i = i0; i < total; i += stride) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(x + grp * 16 * ldx + 2 * cp);
    float a[16], b[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t w = src[e * (ldx / 2)];
      a[e] = __uint_as_float((w << 16) ^ sgn[e]);
      b[e] = __uint_as_float((w & 0xFFFF0000u) ^ sgn[e]);
    }
    m_raw = max(m_raw, max(run_absmax_bits(a), run_absmax_bits(b)));
    m_rht = max(m_rht, max(hadamard16_absmax_bits(a), hadamard16_absmax_bits(b)));
    grp += step_grp;
    cp += step_cp;
    if (cp >= pairs) {
      cp -= pairs;
      ++grp;
    }
  }
  m_raw = block_max(m_raw, red);
  m_rht = block_max(m_rht, red);
  if (threadIdx.x == 0) {
    p.out[t].partials[blockIdx.x] = m_rht;
    p.out[1 - t].partials[blockIdx.x] = m_raw;
  }
}

// PAIRED: two outputs that share work -- pass 0 takes both amaxes from one
// sweep (p.amax_pair), pass 1 copies the transposed output from the other's
// staged tile (p.mirror).  Separate instantiations, so the other calls carry
// none of that code.
template <int PASS, bool PAIRED = false>
__global__ void __launch_bounds__(kThreads, 2) quant_tiles(const __grid_constant__ CUtensorMap xmap,
                                                           const TileParams p) {
  const int mirror = PASS == 1 && PAIRED ? p.mirror : -1;
  const int amax_pair = PASS == 0 && PAIRED ? p.amax_pair : -1;
  extern __shared__ uint8_t smem_raw[];
  constexpr int kStages = stages_of<PASS>();
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ uint32_t red[kThreads / 32];
  __shared__ int abort_flag;
  __shared__ DivTable dtab[kMaxQuantOutputs];  // encode pass only
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;

  float s_dec[kMaxQuantOutputs] = {1.0f, 1.0f};
  float rs[kMaxQuantOutputs] = {0.0f, 0.0f};  // RN(1/s_dec) where the fast block-scale division applies
  bool live[kMaxQuantOutputs] = {true, true};
  if (PASS == 1) {
#pragma unroll
    for (int o = 0; o < kMaxQuantOutputs; ++o) {
      if (o >= p.n_out) break;
      uint32_t m = 0;
      if (p.out[o].amax_in) {
        // delayed scaling: a finite amax >= 0 from the caller (anything else
        // is reported like a non-finite operand)
        const float a = *p.out[o].amax_in;
        m = (a >= 0.0f) ? __float_as_uint(fabsf(a)) : 0x7FC00000u;
      } else {
        const uint32_t* part = p.out[(o == 1 && p.amax_shared) ? 0 : o].partials;
        for (int i = tid; i < p.num_partials; i += kThreads) m = max(m, part[i]);
        m = block_max(m, red);
      }
      if (m >= 0x7F800000u) {  // inf or NaN somewhere in the input
        live[o] = false;
        if (blockIdx.x == 0 && tid == 0) {
          ptx::set_status(p.status, kDevNonFinite);
          *p.out[o].tensor_scale = __uint_as_float(0x7FC00000u);
        }
      } else {
        float s = __fdiv_rn(__uint_as_float(m), 2688.0f);
        if (s == 0.0f) s = 1.0f;
        s_dec[o] = s;
        rs[o] = (s >= 0x1p-70f && s < 0x1p126f) ? __frcp_rn(s) : 0.0f;
        if (blockIdx.x == 0 && tid == 0) *p.out[o].tensor_scale = s;
        if (tid >= 1 && tid < 127) {  // every nonzero finite E4M3 byte
          const float d = __fmul_rn(ptx::e4m3_to_float(static_cast<uint32_t>(tid)), s);
          const bool fast = d >= 0x1p-70f && d < (p.out[o].sr ? 0x1p14f : 0x1p126f);
          dtab[o].e[tid] = make_float2(d, fast ? __frcp_rn(d) : 0.0f);
        }
      }
    }
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(&full[s], 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();

  const int64_t G = gridDim.x;
  const int64_t n_my = blockIdx.x < p.num_tiles ? (p.num_tiles - 1 - blockIdx.x) / G + 1 : 0;
  auto tile_of = [&](int64_t i) {
    const int64_t it = blockIdx.x + i * G;
    return PASS == 1 ? p.num_tiles - 1 - it : it;
  };
  // Failure-detection test hook: CTA 0's first stage is never filled, so
  // its bounded wait runs out and the timeout path below is taken.
  const bool skip0 = p.skip_first_load && blockIdx.x == 0;
  auto issue = [&](int64_t i) {
    if (skip0 && i == 0) return;
    const int s = static_cast<int>(i % kStages);
    const int64_t tile = tile_of(i);
    const int32_t x0 = static_cast<int32_t>((tile % p.tiles_c) * kTile);
    const int32_t y0 = static_cast<int32_t>((tile / p.tiles_c) * kTile);
    uint8_t* dst = ring + s * kStageBytes;
    ptx::mbar_arrive_expect_tx(&full[s], kStageBytes);
    if (PASS == 1) {
      const uint64_t pol = ptx::policy_evict_first();
      ptx::tma_load_2d_hint(dst, &xmap, &full[s], x0, y0, pol);
      ptx::tma_load_2d_hint(dst + kBoxBytes, &xmap, &full[s], x0 + 64, y0, pol);
    } else {
      ptx::tma_load_2d(dst, &xmap, &full[s], x0, y0);
      ptx::tma_load_2d(dst + kBoxBytes, &xmap, &full[s], x0 + 64, y0);
    }
  };
  if (tid == 0 && n_my > 0) {
    ptx::prefetch_tensormap(&xmap);
    for (int64_t i = 0; i < kStages && i < n_my; ++i) issue(i);
  }

  uint32_t tmax[kMaxQuantOutputs] = {0u, 0u};
  bool timed_out = false;  // block-uniform
  for (int64_t i = 0; i < n_my; ++i) {
    const int s = static_cast<int>(i % kStages);
    const uint32_t parity = static_cast<uint32_t>((i / kStages) & 1);
    const bool ok = ptx::mbar_wait(&full[s], parity, &abort_flag);
    if (__syncthreads_or(!ok)) {
      // A wait ran out: record it, let every copy this CTA still has in
      // flight land (bounded waits) before the CTA leaves, and make the
      // failure visible in the outputs: pass 0 leaves a NaN-like partial
      // amax, so pass 1 writes tensor_scale = NaN and encodes nothing;
      // pass 1 writes tensor_scale = NaN itself.
      timed_out = true;
      if (tid == 0) {
        ptx::set_status(p.status, kDevTimeout);
        for (int64_t j = i; j < i + kStages && j < n_my; ++j) {
          if (skip0 && j == 0) continue;  // never issued
          volatile int never = 0;
          ptx::mbar_wait(&full[j % kStages], static_cast<uint32_t>((j / kStages) & 1), &never);
        }
        if (PASS == 1) {
          for (int o = 0; o < p.n_out; ++o) *p.out[o].tensor_scale = __uint_as_float(0x7FC00000u);
        }
      }
      break;
    }
    const uint8_t* stage = ring + s * kStageBytes;
    const int64_t tile = tile_of(i);
    const int64_t tr = tile / p.tiles_c, tc = tile - tr * p.tiles_c;
    uint8_t* stg = ring + kStgOffset + static_cast<int>(i & 1) * (kMaxQuantOutputs * kStgBytes);
    if (amax_pair == 1) amax_tile_pair(stage, p.out[1].rht_sgn, tmax[0], tmax[1]);
    if (amax_pair == 0) amax_tile_pair(stage, p.out[0].rht_sgn, tmax[1], tmax[0]);
#pragma unroll
    for (int o = 0; o < kMaxQuantOutputs; ++o) {
      if (o >= p.n_out) break;
      const OutParams& op = p.out[o];
      if (PASS == 0) {
        if (amax_pair >= 0) break;
        if (o == 1 && p.amax_shared) break;
        if (op.amax_in) continue;
        // without the transform the orientation does not change the amax
        tmax[o] = max(tmax[o], (op.rht && op.col) ? amax_tile<true>(stage, true, op.rht_sgn)
                                                   : amax_tile<false>(stage, op.rht != 0, op.rht_sgn));
      } else if (live[o] && o != mirror) {
        uint8_t* so = stg + o * kStgBytes;
        if (op.col) {
          if (op.sr)
            encode_tile<true, true>(stage, so, op, s_dec[o], rs[o], dtab[o], tr, tc, p.status);
          else
            encode_tile<true, false>(stage, so, op, s_dec[o], rs[o], dtab[o], tr, tc, p.status);
        } else {
          if (op.sr)
            encode_tile<false, true>(stage, so, op, s_dec[o], rs[o], dtab[o], tr, tc, p.status);
          else
            encode_tile<false, false>(stage, so, op, s_dec[o], rs[o], dtab[o], tr, tc, p.status);
        }
      }
    }
    if (mirror >= 0 && live[mirror]) {
      __syncthreads();  // the other output's tile is staged
      mirror_tile(stg + (1 - mirror) * kStgBytes, stg + mirror * kStgBytes);
    }
    // Every thread is done with this stage and, in pass 1, with its staged
    // results.  The staging buffers alternate between tiles, so the copy-out
    // below overlaps the next tile's encode without another barrier.
    __syncthreads();
    if (tid == 0 && i + kStages < n_my) issue(i + kStages);
    if (PASS == 1) {
#pragma unroll
      for (int o = 0; o < kMaxQuantOutputs; ++o) {
        if (o >= p.n_out) break;
        if (!live[o]) continue;
        const OutParams& op = p.out[o];
        copy_out(stg + o * kStgBytes, op, (op.col ? tc : tr) * kTile, (op.col ? tr : tc) * 8);
      }
    }
  }

  if (PASS == 0) {
#pragma unroll
    for (int o = 0; o < kMaxQuantOutputs; ++o) {
      if (o >= p.n_out || (o == 1 && p.amax_shared)) break;
      const uint32_t m = timed_out ? 0xFFFFFFFFu : block_max(tmax[o], red);
      if (tid == 0 && !p.out[o].amax_in) p.out[o].partials[blockIdx.x] = m;
    }
  }
}

template <int PASS>
int tiles_per_sm(cudaError_t* err) {
  // One-time setup per device, safe against concurrent first calls.
  static std::mutex setup_mutex;
  static int per_sm[64] = {0};  // 0: not set up yet
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return 0;
  }
  std::lock_guard<std::mutex> lock(setup_mutex);
  if (per_sm[dev] == 0) {
    *err = cudaFuncSetAttribute(quant_tiles<PASS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<PASS>());
    if (*err != cudaSuccess) return 0;
    *err = cudaFuncSetAttribute(quant_tiles<PASS, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_bytes<PASS>());
    if (*err != cudaSuccess) return 0;
    int b = 0;
    *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, quant_tiles<PASS>, kThreads, smem_bytes<PASS>());
    if (*err != cudaSuccess) return 0;
    per_sm[dev] = std::max(b, 1);
  }
  return per_sm[dev];
}

// Resident CTAs per SM of a streaming row encode (its grid), set up once per
// device like tiles_per_sm.
template <bool SR, bool RHT, bool BLOCK2D>
int rows_per_sm(cudaError_t* err) {
  static std::mutex setup_mutex;
  static int per_sm[64] = {0};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return 0;
  }
  std::lock_guard<std::mutex> lock(setup_mutex);
  if (per_sm[dev] == 0) {
    int b = 0;
    *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, quant_rows<SR, RHT, BLOCK2D>, kThreads, 0);
    if (*err != cudaSuccess) return 0;
    per_sm[dev] = std::max(b, 1);
  }
  return per_sm[dev];
}

// Resident CTAs per SM of a streaming amax kernel, set up once per device.
template <int KIND>  // 0: amax_rows, 1: amax_cols_pair
int amax_stream_per_sm(cudaError_t* err) {
  static std::mutex setup_mutex;
  static int per_sm[64] = {0};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return 0;
  }
  std::lock_guard<std::mutex> lock(setup_mutex);
  if (per_sm[dev] == 0) {
    int b = 0;
    if (KIND == 0)
      *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, amax_rows, kThreads, 0);
    else
      *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, amax_cols_pair, kThreads, 0);
    if (*err != cudaSuccess) return 0;
    per_sm[dev] = std::max(b, 1);
  }
  return per_sm[dev];
}

// Tensor map over x [rows, cols] BF16: box 64 columns x 128 rows, 128-byte
// swizzle, out-of-range elements read as zero.
bool make_x_map(CUtensorMap* map, const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kTile)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(x), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Scratch for nvfp4_quantize_noalloc: the status word (first 256 bytes) and
// the partial-amax slots of the amax pass, in one file-scope device array.
// Every GPU that loads the library holds it until the process exits.  In
// host code `g_noalloc_scratch` only names the symbol; its device address
// comes from cudaGetSymbolAddress, looked up once per CUDA context (with that
// context current) and cached under the context's unique ID, so a context
// created after a reset gets its own lookup instead of a stale address.
constexpr size_t kNoAllocScratchBytes = kWsHeaderBytes + kQuantScratchBytes;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxContexts = 64;
std::mutex g_noalloc_mutex;
unsigned long long g_noalloc_ctx_id[kMaxContexts] = {0};
void* g_noalloc_ptr[kMaxContexts] = {nullptr};
int g_noalloc_count = 0;

using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(ptr);
}

// Unique ID of the calling thread's current context (0 if there is none).
cudaError_t current_ctx_id(unsigned long long* id) {
  static PfnCtxGetCurrent get_current = driver_fn<PfnCtxGetCurrent>("cuCtxGetCurrent");
  static PfnCtxGetId get_id = driver_fn<PfnCtxGetId>("cuCtxGetId");
  *id = 0;
  if (!get_current || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

}  // namespace

cudaError_t noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  unsigned long long id = 0;
  e = current_ctx_id(&id);
  if (e != cudaSuccess) return e;
  for (int i = 0; id != 0 && i < g_noalloc_count; ++i) {
    if (g_noalloc_ctx_id[i] == id) {
      *ptr = g_noalloc_ptr[i];
      return cudaSuccess;
    }
  }
  // First call in this context (the lookup also makes the device's primary
  // context current if no context was).
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (id == 0) {
    e = current_ctx_id(&id);
    if (e != cudaSuccess) return e;
  }
  if (id != 0 && g_noalloc_count < kMaxContexts) {
    g_noalloc_ctx_id[g_noalloc_count] = id;
    g_noalloc_ptr[g_noalloc_count] = p;
    ++g_noalloc_count;
  }
  *ptr = p;
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
  if (a.n_out < 1 || a.n_out > kMaxQuantOutputs) return cudaErrorInvalidValue;
  TileParams p{};
  const int64_t tiles_r = (a.rows + kTile - 1) / kTile;
  p.tiles_c = (a.cols + kTile - 1) / kTile;
  p.num_tiles = (a.rows > 0 && a.cols > 0) ? tiles_r * p.tiles_c : 0;
  p.n_out = a.n_out;
  p.status = a.status;
  for (int o = 0; o < a.n_out; ++o) {
    const QuantOut& q = a.out[o];
    OutParams& op = p.out[o];
    op.codes = q.codes;
    op.sf = q.sf;
    op.tensor_scale = q.tensor_scale;
    op.partials = a.partials + o * kPartialsPerOutput;
    op.amax_in = q.amax_in;
    op.qr = q.transpose ? a.cols : a.rows;
    op.qk = q.transpose ? a.rows : a.cols;
    op.code_ld = op.qk / 2;
    op.kb_count = op.qk / 16;
    op.katoms = (op.kb_count + 3) / 4;
    op.rht_seed = q.rht_seed;
    op.sr_seed = q.sr_seed;
    op.sr_offset = q.sr_offset;
    philox_round_keys(q.sr_seed, op.sr_rk0, op.sr_rk1);  // Weyl schedule (Salmon et al., SC'11)
    rht_sign_words(q.rht_seed, q.rht != 0, op.rht_sgn);
    op.col = q.transpose;
    op.block2d = q.block2d;
    op.sr = q.sr;
    op.rht = q.rht;
    op.sf_mma = q.sf_mma;
    op.vec16 = (reinterpret_cast<uintptr_t>(q.codes) % 16 == 0) && (op.code_ld % 16 == 0);
  }
  p.amax_shared = a.n_out == 2 && !a.out[0].rht && !a.out[1].rht && !a.out[0].amax_in && !a.out[1].amax_in;
  // Two 16x16-block round-to-nearest outputs of opposite orientations under
  // one tensor scale: the transposed one is copied from the other's staged
  // tile (mirror_tile) instead of encoded again.
  p.mirror = -1;
  if (p.amax_shared && a.out[0].block2d && a.out[1].block2d && !a.out[0].sr && !a.out[1].sr &&
      a.out[0].transpose != a.out[1].transpose)
    p.mirror = a.out[0].transpose ? 0 : 1;
  // One transformed column output and one untransformed output, both
  // scanned: one sweep gives both amaxes (amax_tile_pair).
  p.amax_pair = -1;
  if (a.n_out == 2 && !a.out[0].amax_in && !a.out[1].amax_in) {
    for (int t = 0; t < 2; ++t)
      if (a.out[t].rht && a.out[t].transpose && !a.out[1 - t].rht) p.amax_pair = t;
  }
  bool scan = false;  // the amax pass runs unless every output has a supplied amax
  for (int o = 0; o < a.n_out; ++o) scan = scan || !a.out[o].amax_in;

  CUtensorMap xmap{};
  if (p.num_tiles > 0 && !make_x_map(&xmap, a.x, a.rows, a.cols, a.ldx)) return cudaErrorInvalidValue;
  cudaError_t err = cudaSuccess;
  const int b0 = tiles_per_sm<0>(&err);
  if (err != cudaSuccess) return err;
  const int b1 = tiles_per_sm<1>(&err);
  if (err != cudaSuccess) return err;
  // Both passes use one grid: pass 1 reduces one partial per CTA of pass 0.
  int64_t g = static_cast<int64_t>(std::min(b0, b1)) * device_sm_count();
  g = std::min<int64_t>(g, kPartialsPerOutput);
  g = std::max<int64_t>(std::min<int64_t>(g, p.num_tiles), 1);
  p.num_partials = static_cast<int>(g);
  // The amax streams along the rows of x when it is that of x itself: one
  // untransformed output, or two sharing the untransformed amax.  (The
  // failure-detection hook of the amax pass stays on the tiled kernel.)
  // Rows of x must consist of whole runs of 16 (a transposed output only
  // asks that of the columns of x).
  const bool rows_amax = scan && a.skip_load_pass != 1 && p.num_tiles > 0 && a.cols % 16 == 0 &&
                         ((a.n_out == 1 && !a.out[0].rht) || p.amax_shared);
  if (rows_amax) {
    const int per_sm = amax_stream_per_sm<0>(&err);
    if (err != cudaSuccess) return err;
    const int ga = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(per_sm) * device_sm_count(), kPartialsPerOutput));
    p.num_partials = ga;
    amax_rows<<<ga, kThreads, 0, stream>>>(a.x, a.ldx, p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  } else if (scan && p.amax_pair >= 0 && a.skip_load_pass != 1 && p.num_tiles > 0 && a.rows % 16 == 0 &&
             a.cols % 2 == 0) {
    // an activation pair: both amaxes streamed down the columns
    const int per_sm = amax_stream_per_sm<1>(&err);
    if (err != cudaSuccess) return err;
    const int ga = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(per_sm) * device_sm_count(), kPartialsPerOutput));
    p.num_partials = ga;
    amax_cols_pair<<<ga, kThreads, 0, stream>>>(a.x, a.ldx, a.rows, a.cols, p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  } else if (scan) {
    p.skip_first_load = a.skip_load_pass == 1;
    if (p.amax_pair >= 0)
      quant_tiles<0, true><<<static_cast<int>(g), kThreads, smem_bytes<0>(), stream>>>(xmap, p);
    else
      quant_tiles<0><<<static_cast<int>(g), kThreads, smem_bytes<0>(), stream>>>(xmap, p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  p.skip_first_load = a.skip_load_pass == 2;
  const QuantOut& q0 = a.out[0];
  // One row output: the streaming encode, except 16x16 blocks with
  // round-to-nearest and no transform, where its 16-row loads measured slower
  // than the staged tile (the failure-detection hook of the encode pass also
  // stays on the tiled kernel, which has a tile to leave unfilled).
  if (a.n_out == 1 && !q0.transpose && !(q0.block2d && !q0.sr && !q0.rht) && a.skip_load_pass != 2) {
    auto run = [&](auto kernel, int per_sm) {
      kernel<<<per_sm * device_sm_count(), kThreads, 0, stream>>>(a.x, a.ldx, p);
      return cudaGetLastError();
    };
#define NVFP4_ROWS(SR, RHT, B2D)                                            \
  if (!!q0.sr == SR && !!q0.rht == RHT && !!q0.block2d == B2D) {             \
    const int per_sm = rows_per_sm<SR, RHT, B2D>(&err);                      \
    if (err != cudaSuccess) return err;                                      \
    return run(quant_rows<SR, RHT, B2D>, per_sm);                            \
  }
    NVFP4_ROWS(false, false, false)
    NVFP4_ROWS(false, true, false)
    NVFP4_ROWS(false, true, true)
    NVFP4_ROWS(true, false, false)
    NVFP4_ROWS(true, false, true)
    NVFP4_ROWS(true, true, false)
    NVFP4_ROWS(true, true, true)
#undef NVFP4_ROWS
  }
  if (p.mirror >= 0)
    quant_tiles<1, true><<<static_cast<int>(g), kThreads, smem_bytes<1>(), stream>>>(xmap, p);
  else
    quant_tiles<1><<<static_cast<int>(g), kThreads, smem_bytes<1>(), stream>>>(xmap, p);
  return cudaGetLastError();
}

}  // namespace nvfp4
