/*
 * NVFP4 oracle -- TEST INFRASTRUCTURE ONLY (see oracle.h for scope, sources
 * and the list of pins).  Plain C, single-threaded, no vectorisation tricks.
 *
 * Build with contraction disabled (-ffp-contract=off) and without fast-math:
 * every FP32 step below is one IEEE round-to-nearest-even operation, which is
 * what makes the quantised codes a deterministic function of the input.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* E2M1 element codes.                                                        */
/* The 4-bit grid is sparse ("NVIDIA acelera o pre-treinamento de LLM: NVFP4  */
/* no Blackwell...", section "Por que cada porcento e importante"); its eight */
/* magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Bit 3 is the sign, bits 2..0   */
/* index the magnitude (sign-magnitude, exponent bits 2:1, mantissa bit 0).   */
/* ------------------------------------------------------------------------- */
static const double k_e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_value(uint8_t code) {
  double m = k_e2m1_mag[code & 7];
  return (code & 8) ? -m : m;
}

/* E4M3 (FP8, 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no      */
/* infinities, S.1111.111 is NaN, largest finite 448, subnormals m * 2^-9).  */
double oracle_e4m3_value(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int e = (byte >> 3) & 15;
  int m = byte & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

/* Nearest candidate to t >= 0 among ascending values[0..n-1] (all finite),
 * ties going to the candidate whose code has a clear lowest bit ("even
 * mantissa").  Values above the largest candidate pick the largest, which is
 * saturation.  Comparisons are done in double, where the two bracketing
 * candidates and t are exact and their differences are exact. */
static int nearest_even(double t, const double* values, const uint8_t* codes, int n) {
  int hi = 0;
  if (t >= values[n - 1]) return n - 1;
  while (values[hi] <= t) hi++;          /* values[hi] > t >= values[hi-1] */
  if (hi == 0) return 0;
  int lo = hi - 1;
  double dlo = t - values[lo], dhi = values[hi] - t;
  if (dlo < dhi) return lo;
  if (dhi < dlo) return hi;
  return (codes[lo] & 1) ? hi : lo;
}

static double k_e4m3_values[127];
static uint8_t k_e4m3_codes[127];
static int k_e4m3_ready = 0;

static void e4m3_table(void) {
  /* Bytes 0x00..0x7E are the non-negative finite E4M3 values in ascending
   * order (the encoding is monotone in the byte for a fixed sign). */
  if (k_e4m3_ready) return;
  for (int b = 0; b < 127; ++b) {
    k_e4m3_codes[b] = (uint8_t)b;
    k_e4m3_values[b] = oracle_e4m3_value((uint8_t)b);
  }
  k_e4m3_ready = 1;
}

/* Block-scale encoding: t (>= 0, finite) to the nearest E4M3 value, ties to
 * even mantissa, saturating at 448, subnormals kept (reading: the format
 * definition names an E4M3 scale and nothing else; this is the IEEE-style
 * choice). */
uint8_t oracle_e4m3_encode(float t) {
  e4m3_table();
  if (!(t >= 0.0f)) return 0;            /* never reached for valid input */
  return k_e4m3_codes[nearest_even((double)t, k_e4m3_values, k_e4m3_codes, 127)];
}

static const uint8_t k_e2m1_codes[8] = {0, 1, 2, 3, 4, 5, 6, 7};

/* Round-to-nearest-even onto the E2M1 grid.  Ties go to the even code, which
 * gives 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4; magnitudes
 * above 6 saturate to 6.  The sign is the sign bit of v, so a negative value
 * that rounds to zero is encoded 0x8 (reading: IEEE-style signed zero). */
uint8_t oracle_e2m1_encode_rne(float v) {
  double mag = fabs((double)v);
  uint8_t code = k_e2m1_codes[nearest_even(mag, k_e2m1_mag, k_e2m1_codes, 8)];
  return (uint8_t)(code | (signbit(v) ? 8 : 0));
}

/* Stochastic rounding onto the E2M1 grid (reading): for lo <= |v| < hi,
 * adjacent grid points, f = (|v| - lo) / (hi - lo) computed in FP32 (exact:
 * hi - lo is a power of two and |v| - lo is exact by Sterbenz' lemma);
 * u = (r >> 8) * 2^-24 from one 32-bit Philox word; round up iff u < f.
 * |v| >= 6 gives 6.  The sign is kept as in round-to-nearest. */
uint8_t oracle_e2m1_encode_sr(float v, uint32_t r) {
  float mag = fabsf(v);
  uint8_t code;
  if (mag >= 6.0f) {
    code = 7;
  } else {
    int lo = 0;
    while (lo < 7 && k_e2m1_mag[lo + 1] <= (double)mag) lo++;
    float lo_v = (float)k_e2m1_mag[lo];
    float step = (float)(k_e2m1_mag[lo + 1] - k_e2m1_mag[lo]);
    float f = (mag - lo_v) / step;
    float u = (float)(r >> 8) * 0x1p-24f;
    code = (uint8_t)((u < f) ? lo + 1 : lo);
  }
  return (uint8_t)(code | (signbit(v) ? 8 : 0));
}

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As    */
/* Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies, the      */
/* key bumped by the Weyl constants between rounds.                          */
/* ------------------------------------------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* ------------------------------------------------------------------------- */
/* Random Hadamard transform ("Full-Stack FP4...", section 2.2: Hadamard      */
/* mixing spreads the distribution before quantisation).                     */
/* Reading: sigma_j = -1 iff bit j of word 0 of Philox(key = seed,           */
/* counter = 0); x' = 1/4 * H16 * diag(sigma) * x, with H16 the Sylvester    */
/* Hadamard matrix, evaluated as butterflies of stride 1, 2, 4, 8 (each      */
/* output a+b or a-b rounded to FP32), then the exact scaling by 1/4.        */
/* ------------------------------------------------------------------------- */
void oracle_rht_signs(uint64_t seed, float sigma[16]) {
  uint32_t ctr[4] = {0, 0, 0, 0};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  for (int j = 0; j < 16; ++j) sigma[j] = ((out[0] >> j) & 1u) ? -1.0f : 1.0f;
}

void oracle_rht16(float v[16], const float sigma[16]) {
  for (int j = 0; j < 16; ++j) v[j] = v[j] * sigma[j];
  for (int stride = 1; stride < 16; stride *= 2) {
    for (int i = 0; i < 16; ++i) {
      if (i & stride) continue;
      float a = v[i], b = v[i + stride];
      v[i] = a + b;
      v[i + stride] = a - b;
    }
  }
  for (int j = 0; j < 16; ++j) v[j] = v[j] * 0.25f;
}

/* ------------------------------------------------------------------------- */
/* Quantisation                                                               */
/* ------------------------------------------------------------------------- */
static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Materialise the quantised operand Q [qr, qk] as FP32: Q = x or x^T, then the
 * optional transform on each run of 16 along K.  Returns NULL on OOM. */
static float* logical_operand(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                              const oracle_cfg* cfg, int64_t* qr, int64_t* qk) {
  int64_t R = cfg->transpose ? cols : rows;
  int64_t K = cfg->transpose ? rows : cols;
  *qr = R;
  *qk = K;
  float* q = (float*)malloc((size_t)(R * K + 1) * sizeof(float));
  if (!q) return NULL;
  for (int64_t i = 0; i < R; ++i)
    for (int64_t k = 0; k < K; ++k)
      q[i * K + k] = cfg->transpose ? bf16_to_float(x[k * ld + i]) : bf16_to_float(x[i * ld + k]);
  if (cfg->rht) {
    float sigma[16];
    oracle_rht_signs(cfg->rht_seed, sigma);
    for (int64_t i = 0; i < R; ++i)
      for (int64_t k = 0; k < K; k += 16) oracle_rht16(&q[i * K + k], sigma);
  }
  return q;
}

static int check_args(int64_t rows, int64_t cols, int64_t ld, const oracle_cfg* cfg) {
  if (!cfg || rows < 0 || cols < 0 || ld < cols) return ORACLE_ERR_INVALID_ARG;
  if (cfg->block < 0 || cfg->block > 1 || cfg->rounding < 0 || cfg->rounding > 1)
    return ORACLE_ERR_INVALID_ARG;
  int64_t R = cfg->transpose ? cols : rows;
  int64_t K = cfg->transpose ? rows : cols;
  if (K % 16 != 0) return ORACLE_ERR_UNSUPPORTED_SHAPE;
  if (cfg->block == 1 && R % 16 != 0) return ORACLE_ERR_UNSUPPORTED_SHAPE;
  return ORACLE_OK;
}

static float amax_of(const float* q, int64_t n) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(q[i]);
    if (isnan(a)) return NAN;
    if (a > amax) amax = a;
  }
  return amax;
}

int oracle_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                const oracle_cfg* cfg, float* amax) {
  int st = check_args(rows, cols, ld, cfg);
  if (st != ORACLE_OK) return st;
  int64_t R = 0, K = 0;
  float* q = logical_operand(x, rows, cols, ld, cfg, &R, &K);
  if (!q) return ORACLE_ERR_INVALID_ARG;
  *amax = amax_of(q, R * K);
  free(q);
  return ORACLE_OK;
}

/* Steps 3-5 for rows [row_begin, row_end) of the materialised operand q
 * [R, K] under the FP32 tensor scale s_dec.  codes / sf hold only those rows. */
static void encode_rows(const float* q, int64_t K, const oracle_cfg* cfg, float s_dec, int64_t row_begin,
                        int64_t row_end, uint8_t* codes, uint8_t* sf) {
  int64_t KB = K / 16;
  memset(codes, 0, (size_t)((row_end - row_begin) * (K / 2)));
  for (int64_t i = row_begin; i < row_end; ++i) {
    int64_t oi = i - row_begin;
    for (int64_t b = 0; b < KB; ++b) {
      /* Step 3: block amax over the 1x16 run, or over the whole 16x16 tile
       * the run belongs to (its scale is then repeated on the tile's 16 rows). */
      float bamax = 0.0f;
      int64_t r0 = (cfg->block == 1) ? (i / 16) * 16 : i;
      int64_t r1 = (cfg->block == 1) ? r0 + 16 : i + 1;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t k = b * 16; k < b * 16 + 16; ++k) {
          float a = fabsf(q[r * K + k]);
          if (a > bamax) bamax = a;
        }
      /* Step 4: block scale t = (bamax / 6) / s, two FP32 divisions, then
       * E4M3 round-to-nearest-even with saturation. */
      float t = (bamax / 6.0f) / s_dec;
      uint8_t sfb = oracle_e4m3_encode(t);
      sf[oi * KB + b] = sfb;
      /* Step 5: elements v = x / (scale * s), one FP32 multiply then one FP32
       * division, rounded onto the E2M1 grid.  A zero block scale encodes the
       * whole run as code 0. */
      float denom = (float)oracle_e4m3_value(sfb) * s_dec;
      for (int64_t k = b * 16; k < b * 16 + 16; ++k) {
        uint8_t code = 0;
        if (sfb != 0) {
          float v = q[i * K + k] / denom;
          if (cfg->rounding == 0) {
            code = oracle_e2m1_encode_rne(v);
          } else {
            /* Philox counter for element e = i*K + k of Q: (e >> 2 as a 64-bit
             * pair, sr_offset as a 64-bit pair), key = sr_seed; word e & 3. */
            uint64_t e = (uint64_t)(i * K + k);
            uint32_t ctr[4] = {(uint32_t)(e >> 2), (uint32_t)(e >> 34),
                               (uint32_t)cfg->sr_offset, (uint32_t)(cfg->sr_offset >> 32)};
            uint32_t key[2] = {(uint32_t)cfg->sr_seed, (uint32_t)(cfg->sr_seed >> 32)};
            uint32_t out[4];
            oracle_philox4x32_10(ctr, key, out);
            code = oracle_e2m1_encode_sr(v, out[e & 3]);
          }
        }
        /* Packing: element 2j in the low nibble of byte j, 2j+1 in the high. */
        codes[oi * (K / 2) + k / 2] |= (uint8_t)(code << (4 * (k & 1)));
      }
    }
  }
}

/* Step 2: FP32 tensor (decode) scale s = amax / (6 * 448): the largest block
 * can then reach both the largest E4M3 scale and the largest E2M1 element
 * (reading).  A zero scale (all-zero or subnormal-tiny tensor) is replaced by
 * 1, which makes every block scale and every code zero. */
static float tensor_scale_of(float amax) {
  float s_dec = amax / 2688.0f;
  if (s_dec == 0.0f) s_dec = 1.0f;
  return s_dec;
}

/* Encode rows [row_begin, row_end) of Q; the tensor scale always comes from
 * the amax of the whole operand.  codes / sf hold only the encoded rows. */
int oracle_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, const oracle_cfg* cfg,
                         int64_t row_begin, int64_t row_end, uint8_t* codes, uint8_t* sf, float* tensor_scale) {
  int st = check_args(rows, cols, ld, cfg);
  if (st != ORACLE_OK) return st;
  int64_t R = 0, K = 0;
  float* q = logical_operand(x, rows, cols, ld, cfg, &R, &K);
  if (!q) return ORACLE_ERR_INVALID_ARG;
  if (row_begin < 0 || row_end > R || row_begin > row_end) {
    free(q);
    return ORACLE_ERR_INVALID_ARG;
  }
  /* Step 1: tensor amax, taken after the transform (reading). */
  float amax = amax_of(q, R * K);
  if (!isfinite(amax)) {
    free(q);
    return ORACLE_ERR_NONFINITE;
  }
  float s_dec = tensor_scale_of(amax);
  *tensor_scale = s_dec;
  encode_rows(q, K, cfg, s_dec, row_begin, row_end, codes, sf);
  free(q);
  return ORACLE_OK;
}

/* Delayed scaling: step 1 is replaced by an amax the caller supplies (for
 * instance the one measured on the previous step), so the operand is not
 * scanned before it is encoded.  The supplied amax must be finite and >= 0;
 * so must every element (ORACLE_ERR_NONFINITE otherwise).  Elements above the
 * supplied amax saturate: their block scale stops at 448 and their codes at
 * +-6, both by the rounding rules of steps 4 and 5 (reading: the format pages
 * fix no scaling policy; this keeps every other step unchanged). */
int oracle_quantize_given_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                               const oracle_cfg* cfg, float amax, uint8_t* codes, uint8_t* sf,
                               float* tensor_scale) {
  int st = check_args(rows, cols, ld, cfg);
  if (st != ORACLE_OK) return st;
  if (!(amax >= 0.0f) || isinf(amax)) return ORACLE_ERR_NONFINITE;
  int64_t R = 0, K = 0;
  float* q = logical_operand(x, rows, cols, ld, cfg, &R, &K);
  if (!q) return ORACLE_ERR_INVALID_ARG;
  if (!isfinite(amax_of(q, R * K))) {
    free(q);
    return ORACLE_ERR_NONFINITE;
  }
  float s_dec = tensor_scale_of(fabsf(amax));
  *tensor_scale = s_dec;
  encode_rows(q, K, cfg, s_dec, 0, R, codes, sf);
  free(q);
  return ORACLE_OK;
}

int oracle_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                    const oracle_cfg* cfg, uint8_t* codes, uint8_t* sf, float* tensor_scale) {
  int st = check_args(rows, cols, ld, cfg);
  if (st != ORACLE_OK) return st;
  int64_t R = cfg->transpose ? cols : rows;
  return oracle_quantize_rows(x, rows, cols, ld, cfg, 0, R, codes, sf, tensor_scale);
}

/* ------------------------------------------------------------------------- */
/* Tensor-core scale layout: the operand's scales are cut into atoms of 128  */
/* rows x 4 scales (64 elements of K), 512 bytes each, atoms ordered by row   */
/* block then K block; inside an atom, scale (r, j) sits at byte              */
/* (r % 32) * 16 + (r / 32) * 4 + j.  Rows and scale columns beyond the      */
/* operand are padding and hold zero.                                        */
/* ------------------------------------------------------------------------- */
int64_t oracle_sf_mma_bytes(int64_t qr, int64_t qk) {
  int64_t row_atoms = (qr + 127) / 128;
  int64_t k_atoms = (qk / 16 + 3) / 4;
  return row_atoms * k_atoms * 512;
}

int64_t oracle_sf_mma_offset(int64_t r, int64_t kb, int64_t qk) {
  int64_t k_atoms = (qk / 16 + 3) / 4;
  int64_t atom = (r / 128) * k_atoms + kb / 4;
  int64_t rr = r % 128;
  return atom * 512 + (rr % 32) * 16 + (rr / 32) * 4 + (kb % 4);
}

void oracle_sf_to_mma(const uint8_t* sf, int64_t qr, int64_t qk, uint8_t* out) {
  memset(out, 0, (size_t)oracle_sf_mma_bytes(qr, qk));
  for (int64_t r = 0; r < qr; ++r)
    for (int64_t kb = 0; kb < qk / 16; ++kb) out[oracle_sf_mma_offset(r, kb, qk)] = sf[r * (qk / 16) + kb];
}

/* ------------------------------------------------------------------------- */
/* Dequantisation and the reference GEMM (FP64; the accumulators of the NVFP4 */
/* GEMM are FP32 per "NVIDIA acelera...", "Como o treinamento mixed-precision */
/* funciona com NVFP4", so FP64 is the exact-enough reference).               */
/* ------------------------------------------------------------------------- */
static double deq(const uint8_t* codes, const uint8_t* sf, double s, int64_t qk, int64_t i, int64_t k) {
  uint8_t byte = codes[i * (qk / 2) + k / 2];
  uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
  return oracle_e2m1_value(code) * oracle_e4m3_value(sf[i * (qk / 16) + k / 16]) * s;
}

void oracle_dequantize(const uint8_t* codes, const uint8_t* sf, float tensor_scale,
                       int64_t qr, int64_t qk, double* out) {
  for (int64_t i = 0; i < qr; ++i)
    for (int64_t k = 0; k < qk; ++k) out[i * qk + k] = deq(codes, sf, tensor_scale, qk, i, k);
}

void oracle_gemm_f64(const uint8_t* a_codes, const uint8_t* a_sf, float a_scale,
                     const uint8_t* b_codes, const uint8_t* b_sf, float b_scale,
                     int64_t M, int64_t N, int64_t K, double* out) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += deq(a_codes, a_sf, a_scale, K, m, k) * deq(b_codes, b_sf, b_scale, K, n, k);
      out[m * N + n] = acc;
    }
}

void oracle_gemm_f64_sampled(const uint8_t* a_codes, const uint8_t* a_sf, float a_scale,
                             const uint8_t* b_codes, const uint8_t* b_sf, float b_scale,
                             int64_t K, const int64_t* m_idx, const int64_t* n_idx,
                             int64_t count, double* out) {
  for (int64_t c = 0; c < count; ++c) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
      acc += deq(a_codes, a_sf, a_scale, K, m_idx[c], k) * deq(b_codes, b_sf, b_scale, K, n_idx[c], k);
    out[c] = acc;
  }
}

/* ------------------------------------------------------------------------- */
/* Quantised AdamW state codec ("Full-Stack FP4: Stable LLM Pretraining with  */
/* Quantized Projections, Optimizers, and Attention", section 2.2, Q-AdamW):  */
/* the first moment is Hadamard-mixed and stored in NVFP4 with stochastic     */
/* rounding and an adaptive 4/6 block mapping; the second moment is stored as */
/* sqrt, minus a BF16 tile mean, Hadamard-mixed, in NVFP4; reconstruction     */
/* inverts each step and squares.                                             */
/* ------------------------------------------------------------------------- */

/* Inverse of oracle_rht16: x = diag(sigma) * (1/4) * H16 * x' (H16 H16 = 16 I),
 * the same butterflies, then the exact scaling by 1/4, then the signs. */
void oracle_rht16_inverse(float v[16], const float sigma[16]) {
  for (int stride = 1; stride < 16; stride *= 2) {
    for (int i = 0; i < 16; ++i) {
      if (i & stride) continue;
      float a = v[i], b = v[i + stride];
      v[i] = a + b;
      v[i + stride] = a - b;
    }
  }
  for (int j = 0; j < 16; ++j) v[j] = v[j] * 0.25f;
  for (int j = 0; j < 16; ++j) v[j] = v[j] * sigma[j];
}

/* FP32 -> BF16 bits, round to nearest even (finite input). */
uint16_t oracle_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Round-to-nearest squared error of one run under scale byte sfb:
 * sum over j, in order, of (x_j - e2m1(RNE(x_j / d)) * d)^2 in FP32, d = e4m3(sfb) * s. */
static float run_rne_error(const float* x, uint8_t sfb, float s_dec) {
  float err = 0.0f;
  float d = (float)oracle_e4m3_value(sfb) * s_dec;
  for (int j = 0; j < 16; ++j) {
    float deq = 0.0f;
    if (sfb != 0) deq = (float)oracle_e2m1_value(oracle_e2m1_encode_rne(x[j] / d)) * d;
    float e = x[j] - deq;
    err = err + e * e;
  }
  return err;
}

static void sr_code_run(const float* x, uint8_t sfb, float s_dec, uint64_t e0, uint64_t sr_seed, uint64_t sr_offset,
                        uint8_t* codes_row, int64_t k0) {
  float d = (float)oracle_e4m3_value(sfb) * s_dec;
  for (int j = 0; j < 16; ++j) {
    uint8_t code = 0;
    if (sfb != 0) {
      uint64_t e = e0 + (uint64_t)j;
      uint32_t ctr[4] = {(uint32_t)(e >> 2), (uint32_t)(e >> 34), (uint32_t)sr_offset, (uint32_t)(sr_offset >> 32)};
      uint32_t key[2] = {(uint32_t)sr_seed, (uint32_t)(sr_seed >> 32)};
      uint32_t out[4];
      oracle_philox4x32_10(ctr, key, out);
      code = oracle_e2m1_encode_sr(x[j] / d, out[e & 3]);
    }
    int64_t k = k0 + j;
    codes_row[k / 2] |= (uint8_t)(code << (4 * (k & 1)));
  }
}

/* First moment m [rows, cols] (FP32, row-major, cols % 16 == 0):
 *  1. x = 1/4 H16 diag(sigma) m on every run of 16 along a row (sigma from rht_seed);
 *  2. s = amax(x) / 2688 (1 if zero);
 *  3. per run (reading of "adaptive 4/6"): candidate scale bytes E4M3((bamax/6)/s)
 *     and E4M3((bamax/4)/s); the one whose round-to-nearest squared error is
 *     smaller is kept, the 6-mapping on a tie;
 *  4. codes by stochastic rounding with the Philox stream of the quantiser
 *     (element index i * cols + k, key sr_seed, counter words 2..3 sr_offset).
 * Outputs: codes [rows, cols/2], sf [rows, cols/16] row-major, tensor_scale. */
int oracle_qadamw_m_encode(const float* m, int64_t rows, int64_t cols, uint64_t rht_seed, uint64_t sr_seed,
                           uint64_t sr_offset, uint8_t* codes, uint8_t* sf, float* tensor_scale) {
  if (rows < 0 || cols < 0) return ORACLE_ERR_INVALID_ARG;
  if (cols % 16 != 0) return ORACLE_ERR_UNSUPPORTED_SHAPE;
  int64_t n = rows * cols, KB = cols / 16;
  float* x = (float*)malloc((size_t)(n + 1) * sizeof(float));
  if (!x) return ORACLE_ERR_INVALID_ARG;
  memcpy(x, m, (size_t)n * sizeof(float));
  float sigma[16];
  oracle_rht_signs(rht_seed, sigma);
  for (int64_t i = 0; i < n; i += 16) oracle_rht16(&x[i], sigma);
  float amax = amax_of(x, n);
  if (!isfinite(amax)) {
    free(x);
    return ORACLE_ERR_NONFINITE;
  }
  float s_dec = tensor_scale_of(amax);
  *tensor_scale = s_dec;
  memset(codes, 0, (size_t)(n / 2));
  for (int64_t i = 0; i < rows; ++i)
    for (int64_t b = 0; b < KB; ++b) {
      const float* run = &x[i * cols + b * 16];
      float bamax = 0.0f;
      for (int j = 0; j < 16; ++j)
        if (fabsf(run[j]) > bamax) bamax = fabsf(run[j]);
      uint8_t sf6 = oracle_e4m3_encode((bamax / 6.0f) / s_dec);
      uint8_t sf4 = oracle_e4m3_encode((bamax / 4.0f) / s_dec);
      uint8_t sfb = run_rne_error(run, sf4, s_dec) < run_rne_error(run, sf6, s_dec) ? sf4 : sf6;
      sf[i * KB + b] = sfb;
      sr_code_run(run, sfb, s_dec, (uint64_t)(i * cols + b * 16), sr_seed, sr_offset, &codes[i * (cols / 2)], b * 16);
    }
  free(x);
  return ORACLE_OK;
}

/* m_hat = diag(sigma) 1/4 H16 (e2m1(code) * e4m3(sf) * s) per run, in FP32
 * (dequantised value: code value times the FP32 product e4m3(sf) * s). */
void oracle_qadamw_m_decode(const uint8_t* codes, const uint8_t* sf, float tensor_scale, int64_t rows, int64_t cols,
                            uint64_t rht_seed, float* m_out) {
  float sigma[16];
  oracle_rht_signs(rht_seed, sigma);
  int64_t KB = cols / 16;
  for (int64_t i = 0; i < rows; ++i)
    for (int64_t b = 0; b < KB; ++b) {
      float v[16];
      float d = (float)oracle_e4m3_value(sf[i * KB + b]) * tensor_scale;
      for (int j = 0; j < 16; ++j) {
        int64_t k = b * 16 + j;
        uint8_t byte = codes[i * (cols / 2) + k / 2];
        uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
        v[j] = (float)oracle_e2m1_value(code) * d;
      }
      oracle_rht16_inverse(v, sigma);
      memcpy(&m_out[i * cols + b * 16], v, sizeof(v));
    }
}

/* Second moment v [rows, cols] (FP32 >= 0, rows and cols multiples of 16):
 *  1. r = sqrt(v) (IEEE);
 *  2. per 16x16 tile, mu = BF16_RNE(T * 2^-8) where T sums the tile's row sums
 *     (each a left-to-right FP32 sum of 16) in row order (reading: "tile" =
 *     16 x 16, the 2-D block of the format);
 *  3. residual e = r - mu (FP32);
 *  4. x = 1/4 H16 diag(sigma) e per run of 16 along a row;
 *  5. s = amax(x) / 2688, then round-to-nearest NVFP4 with 1x16 blocks
 *     (E4M3((bamax/6)/s)), as the quantiser's steps 3-5.
 * Outputs: codes, sf (row-major), tensor_scale, tile means [rows/16, cols/16] as BF16 bits.
 * A negative or non-finite v is ORACLE_ERR_NONFINITE. */
int oracle_qadamw_v_encode(const float* v, int64_t rows, int64_t cols, uint64_t rht_seed, uint8_t* codes, uint8_t* sf,
                           float* tensor_scale, uint16_t* tile_mean) {
  if (rows < 0 || cols < 0) return ORACLE_ERR_INVALID_ARG;
  if (cols % 16 != 0 || rows % 16 != 0) return ORACLE_ERR_UNSUPPORTED_SHAPE;
  int64_t n = rows * cols, KB = cols / 16, TR = rows / 16;
  for (int64_t i = 0; i < n; ++i)
    if (!(v[i] >= 0.0f) || isinf(v[i])) return ORACLE_ERR_NONFINITE;
  float* x = (float*)malloc((size_t)(n + 1) * sizeof(float));
  if (!x) return ORACLE_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i) x[i] = sqrtf(v[i]);
  for (int64_t tr = 0; tr < TR; ++tr)
    for (int64_t tc = 0; tc < KB; ++tc) {
      float total = 0.0f;
      for (int i = 0; i < 16; ++i) {
        float row = 0.0f;
        for (int j = 0; j < 16; ++j) row = row + x[(tr * 16 + i) * cols + tc * 16 + j];
        total = total + row;
      }
      uint16_t mu = oracle_bf16_rne(total * 0.00390625f);
      tile_mean[tr * KB + tc] = mu;
      float muf = bf16_to_float(mu);
      for (int i = 0; i < 16; ++i)
        for (int j = 0; j < 16; ++j) {
          float* p = &x[(tr * 16 + i) * cols + tc * 16 + j];
          *p = *p - muf;
        }
    }
  float sigma[16];
  oracle_rht_signs(rht_seed, sigma);
  for (int64_t i = 0; i < n; i += 16) oracle_rht16(&x[i], sigma);
  float amax = amax_of(x, n);
  float s_dec = tensor_scale_of(amax);
  *tensor_scale = s_dec;
  oracle_cfg cfg;
  memset(&cfg, 0, sizeof(cfg));
  encode_rows(x, cols, &cfg, s_dec, 0, rows, codes, sf);
  free(x);
  return ORACLE_OK;
}

/* v_hat = (mu + diag(sigma) 1/4 H16 deq)^2 per element, in FP32. */
void oracle_qadamw_v_decode(const uint8_t* codes, const uint8_t* sf, float tensor_scale, const uint16_t* tile_mean,
                            int64_t rows, int64_t cols, uint64_t rht_seed, float* v_out) {
  float* r = (float*)malloc((size_t)(rows * cols + 1) * sizeof(float));
  if (!r) return;
  oracle_qadamw_m_decode(codes, sf, tensor_scale, rows, cols, rht_seed, r);
  int64_t KB = cols / 16;
  for (int64_t i = 0; i < rows; ++i)
    for (int64_t k = 0; k < cols; ++k) {
      float q = bf16_to_float(tile_mean[(i / 16) * KB + k / 16]) + r[i * cols + k];
      v_out[i * cols + k] = q * q;
    }
  free(r);
}

/* ------------------------------------------------------------------------- */
/* LoRA-SVD projection, forward ("Full-Stack FP4...", section 2.1): the      */
/* weight is W = W_res + beta * L2 L1, with the residual W_res in NVFP4 and    */
/* the principal low-rank part L2 [dout, r], L1 [r, din] in BF16.             */
/* Reading: Y = X W^T = (NVFP4 GEMM of X and W_res) + beta * (U L2^T), with   */
/* U = BF16_RNE(X L1^T) the branch's intermediate (its product summed in      */
/* FP64 over the BF16 inputs), U L2^T summed in FP64; Y in FP64.              */
/* ------------------------------------------------------------------------- */

/* The branch's first product for rows [t0, t1) of X: u_exact = X L1^T summed
 * in FP64, u_bf16 = its BF16 rounding (through FP32, as the intermediate is
 * stored).  Either output may be NULL. */
static void lora_down_rows(const uint16_t* x, const uint16_t* l1, int64_t din, int64_t r, int64_t t0, int64_t t1,
                           uint16_t* u_bf16, double* u_exact) {
  for (int64_t t = t0; t < t1; ++t)
    for (int64_t j = 0; j < r; ++j) {
      double acc = 0.0;
      for (int64_t k = 0; k < din; ++k) acc += (double)bf16_to_float(x[t * din + k]) * bf16_to_float(l1[j * din + k]);
      if (u_exact) u_exact[(t - t0) * r + j] = acc;
      if (u_bf16) u_bf16[(t - t0) * r + j] = oracle_bf16_rne((float)acc);
    }
}

void oracle_lora_down(const uint16_t* x, const uint16_t* l1, int64_t T, int64_t din, int64_t r, uint16_t* u_bf16,
                      double* u_exact) {
  lora_down_rows(x, l1, din, r, 0, T, u_bf16, u_exact);
}

void oracle_lora_forward(const uint8_t* xq_codes, const uint8_t* xq_sf, float xq_scale, const uint8_t* wq_codes,
                         const uint8_t* wq_sf, float wq_scale, const uint16_t* x, const uint16_t* l1,
                         const uint16_t* l2, double beta, int64_t T, int64_t din, int64_t dout, int64_t r,
                         double* out) {
  oracle_gemm_f64(xq_codes, xq_sf, xq_scale, wq_codes, wq_sf, wq_scale, T, dout, din, out);
  uint16_t* u = (uint16_t*)malloc((size_t)(T * r + 1) * sizeof(uint16_t));
  if (!u) return;
  oracle_lora_down(x, l1, T, din, r, u, NULL);
  for (int64_t t = 0; t < T; ++t)
    for (int64_t n = 0; n < dout; ++n) {
      double acc = 0.0;
      for (int64_t j = 0; j < r; ++j) acc += (double)bf16_to_float(u[t * r + j]) * bf16_to_float(l2[n * r + j]);
      out[t * dout + n] += beta * acc;
    }
  free(u);
}

/* The same Y at the listed (t, n) coordinates only. */
void oracle_lora_forward_sampled(const uint8_t* xq_codes, const uint8_t* xq_sf, float xq_scale,
                                 const uint8_t* wq_codes, const uint8_t* wq_sf, float wq_scale, const uint16_t* x,
                                 const uint16_t* l1, const uint16_t* l2, double beta, int64_t din, int64_t r,
                                 const int64_t* t_idx, const int64_t* n_idx, int64_t count, double* out) {
  oracle_gemm_f64_sampled(xq_codes, xq_sf, xq_scale, wq_codes, wq_sf, wq_scale, din, t_idx, n_idx, count, out);
  uint16_t* u = (uint16_t*)malloc((size_t)(r + 1) * sizeof(uint16_t));
  if (!u) return;
  for (int64_t c = 0; c < count; ++c) {
    lora_down_rows(x, l1, din, r, t_idx[c], t_idx[c] + 1, u, NULL);
    double acc = 0.0;
    for (int64_t j = 0; j < r; ++j) acc += (double)bf16_to_float(u[j]) * bf16_to_float(l2[n_idx[c] * r + j]);
    out[c] += beta * acc;
  }
  free(u);
}

/* ------------------------------------------------------------------------- */
/* p99 clipping for the NVFP4 Newton-Schulz products ("Full-Stack FP4...",    */
/* section 2.3): outliers above the 99th percentile are clipped before       */
/* quantisation.  Reading: nearest-rank percentile of |x| over the tensor,    */
/* i.e. the k-th smallest magnitude with k = ceil(p / 100 * n) (k >= 1).      */
/* ------------------------------------------------------------------------- */
static int cmp_float(const void* a, const void* b) {
  float x = *(const float*)a, y = *(const float*)b;
  return (x > y) - (x < y);
}

float oracle_abs_percentile_bf16(const uint16_t* x, int64_t n, double p) {
  if (n <= 0) return 0.0f;
  float* m = (float*)malloc((size_t)n * sizeof(float));
  if (!m) return NAN;
  for (int64_t i = 0; i < n; ++i) m[i] = fabsf(bf16_to_float(x[i]));
  qsort(m, (size_t)n, sizeof(float), cmp_float);
  int64_t k = (int64_t)ceil(p / 100.0 * (double)n);
  if (k < 1) k = 1;
  if (k > n) k = n;
  float v = m[k - 1];
  free(m);
  return v;
}

/* x clipped to [-c, c] element-wise (BF16 in, BF16 out; c a BF16 magnitude). */
void oracle_clip_bf16(const uint16_t* x, int64_t n, float c, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    float v = bf16_to_float(x[i]);
    if (v > c) v = c;
    if (v < -c) v = -c;
    out[i] = oracle_bf16_rne(v);
  }
}

/* ------------------------------------------------------------------------- */
/* One Newton-Schulz step of the Root optimizer with its matrix products in   */
/* NVFP4 ("Full-Stack FP4...", section 2.3: the NS products run directly in   */
/* NVFP4, stabilised by shape-dependent coefficients a, b, c and p99 outlier  */
/* clipping).  The pages print no coefficients and no formula; reading: the   */
/* quintic step on an iterate X [m, n] (m <= n is the caller's orientation),  */
/*     A = X X^T,   B = b A + c A A^T,   X' = a X + B X,                       */
/* where every matrix product L R^T is the NVFP4 GEMM of its two operands,    */
/* each clipped to [-q, q] (q its own p-th percentile magnitude) and then     */
/* quantised along its K with 1x16 blocks, round to nearest, no transform;    */
/* the products' results and the iterate are stored in BF16 (round to nearest */
/* even of the exact FP64 sum), the sums a X + ... and b A + ... in FP32.     */
/* Clipping applies only to the operands of a product: the linear terms use  */
/* the unclipped tensors.                                                    */
/* ------------------------------------------------------------------------- */

/* FP64 -> BF16 bits, one round to nearest even (no intermediate FP32 step):
 * the value is scaled by a power of two so that the BF16 quantum is 1,
 * rounded to an integer (ties to even), and scaled back. */
uint16_t oracle_bf16_rne_f64(double d) {
  if (isnan(d)) return 0x7FC0u;
  uint16_t sign = signbit(d) ? 0x8000u : 0u;
  double a = fabs(d);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);           /* a = f 2^e, f in [1/2, 1) */
  int q = e - 8;          /* quantum of 8 significant bits */
  if (q < -133) q = -133; /* BF16 subnormal quantum */
  double v = ldexp(nearbyint(ldexp(a, -q)), q);
  if (v >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
  float f = (float)v; /* exact: v has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | (u >> 16));
}

/* out = BF16_RNE(RN(RN(a x) + RN(b y))) elementwise, in FP32. */
void oracle_axpby_bf16(const uint16_t* x, const uint16_t* y, int64_t n, float a, float b, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    float ax = a * bf16_to_float(x[i]);
    float by = b * bf16_to_float(y[i]);
    float s = ax + by;
    out[i] = oracle_bf16_rne(s);
  }
}

/* BF16 result of the NVFP4 product L R^T, L [ml, k], R [nr, k] given as
 * clipped BF16 tensors, each quantised along k (R given transposed when
 * r_transposed: R^T [k, nr] row-major, quantised down its columns). */
static int ns_product(const uint16_t* l, int64_t ml, const uint16_t* rsrc, int64_t nr, int64_t k, int r_transposed,
                      uint16_t* out) {
  oracle_cfg cfg;
  memset(&cfg, 0, sizeof(cfg));
  uint8_t* lc = (uint8_t*)malloc((size_t)(ml * k / 2 + 1));
  uint8_t* ls = (uint8_t*)malloc((size_t)(ml * k / 16 + 1));
  uint8_t* rc = (uint8_t*)malloc((size_t)(nr * k / 2 + 1));
  uint8_t* rs = (uint8_t*)malloc((size_t)(nr * k / 16 + 1));
  double* d = (double*)malloc((size_t)(ml * nr + 1) * sizeof(double));
  int st = ORACLE_ERR_INVALID_ARG;
  float lsc = 0.0f, rsc = 0.0f;
  if (lc && ls && rc && rs && d) {
    st = oracle_quantize(l, ml, k, k, &cfg, lc, ls, &lsc);
    if (st == ORACLE_OK) {
      if (r_transposed) {
        cfg.transpose = 1;
        st = oracle_quantize(rsrc, k, nr, nr, &cfg, rc, rs, &rsc);
      } else {
        st = oracle_quantize(rsrc, nr, k, k, &cfg, rc, rs, &rsc);
      }
    }
    if (st == ORACLE_OK) {
      oracle_gemm_f64(lc, ls, lsc, rc, rs, rsc, ml, nr, k, d);
      for (int64_t i = 0; i < ml * nr; ++i) out[i] = oracle_bf16_rne_f64(d[i]);
    }
  }
  free(lc);
  free(ls);
  free(rc);
  free(rs);
  free(d);
  return st;
}

static void clip_to_percentile(const uint16_t* x, int64_t count, double p, float* q, uint16_t* out) {
  *q = oracle_abs_percentile_bf16(x, count, p);
  oracle_clip_bf16(x, count, *q, out);
}

int oracle_ns_step(const uint16_t* x, int64_t m, int64_t n, float a, float b, float c, double p, uint16_t* out,
                   oracle_ns_trace* trace) {
  if (m <= 0 || n <= 0 || m % 32 != 0 || n % 32 != 0) return ORACLE_ERR_UNSUPPORTED_SHAPE;
  size_t mn = (size_t)(m * n), mm = (size_t)(m * m);
  uint16_t* xc = (uint16_t*)malloc(mn * 2);
  uint16_t* am = (uint16_t*)malloc(mm * 2);
  uint16_t* ac = (uint16_t*)malloc(mm * 2);
  uint16_t* a2 = (uint16_t*)malloc(mm * 2);
  uint16_t* bm = (uint16_t*)malloc(mm * 2);
  uint16_t* bc = (uint16_t*)malloc(mm * 2);
  uint16_t* bx = (uint16_t*)malloc(mn * 2);
  float qx = 0.0f, qa = 0.0f, qb = 0.0f;
  int st = ORACLE_ERR_INVALID_ARG;
  if (xc && am && ac && a2 && bm && bc && bx) {
    clip_to_percentile(x, (int64_t)mn, p, &qx, xc);
    st = ns_product(xc, m, xc, m, n, 0, am); /* A = X X^T */
    if (st == ORACLE_OK) {
      clip_to_percentile(am, (int64_t)mm, p, &qa, ac);
      st = ns_product(ac, m, ac, m, m, 0, a2); /* A A^T */
    }
    if (st == ORACLE_OK) {
      oracle_axpby_bf16(am, a2, (int64_t)mm, b, c, bm); /* B = b A + c A A^T */
      clip_to_percentile(bm, (int64_t)mm, p, &qb, bc);
      st = ns_product(bc, m, xc, n, m, 1, bx); /* B X: R = X^T, given as X [m, n] */
    }
    if (st == ORACLE_OK) {
      float one = 1.0f;
      oracle_axpby_bf16(x, bx, (int64_t)mn, a, one, out); /* X' = a X + B X */
      if (trace) {
        trace->qx = qx;
        trace->qa = qa;
        trace->qb = qb;
        if (trace->xc) memcpy(trace->xc, xc, mn * 2);
        if (trace->a) memcpy(trace->a, am, mm * 2);
        if (trace->ac) memcpy(trace->ac, ac, mm * 2);
        if (trace->a2) memcpy(trace->a2, a2, mm * 2);
        if (trace->b) memcpy(trace->b, bm, mm * 2);
        if (trace->bc) memcpy(trace->bc, bc, mm * 2);
        if (trace->bx) memcpy(trace->bx, bx, mn * 2);
      }
    }
  }
  free(xc);
  free(am);
  free(ac);
  free(a2);
  free(bm);
  free(bc);
  free(bx);
  return st;
}
