/*
 * NVFP4 oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of what the NVFP4 linear-layer
 * hot path computes: block-scaled quantisation of BF16 tensors to E2M1 codes
 * with E4M3 block scales and an FP32 tensor scale, the optional 16-point random
 * Hadamard transform, stochastic rounding from a Philox4x32-10 stream,
 * dequantisation and the FP64 reference GEMM.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this code.  The GPU library shares nothing with it: no header, no
 * table, no helper.  Every decision it makes is written out in the order the
 * format definition gives it, so that it can be checked by eye.
 *
 * Sources (page title, section):
 *  - "NVIDIA acelera o pre-treinamento de LLM: NVFP4 no Blackwell em conjunto
 *    com JAX e MaxText", section "Por que cada porcento e importante": NVFP4 is
 *    a 4-bit floating-point format, twice as dense as FP8, whose numeric grid
 *    is sparse, so values must be brought into range by custom scaling.
 *  - same page, section "Como o treinamento mixed-precision funciona com
 *    NVFP4": NVFP4 is used for weights and activations inside GEMMs while the
 *    accumulators stay in BF16/FP32.
 *  - "Full-Stack FP4: Stable LLM Pretraining with Quantized Projections,
 *    Optimizers, and Attention", section 2.2: Hadamard mixing before
 *    quantisation and stochastic rounding (SR).
 *  The element grid {0, 0.5, 1, 1.5, 2, 3, 4, 6} (E2M1), the E4M3 scale per 16
 *  elements, the FP32 per-tensor scale, the 1x16 / 16x16 block shapes, the
 *  Philox SR stream and the 16x16 Hadamard with a seeded sign vector are the
 *  library's format definition; every point the pages leave open is a
 *  documented reading (see the comments at each step).
 *
 * Parity pins: every function here is checked by the CPU test suite against
 * values fixed independently of this file (exhaustive codec tables against
 * torch's float8_e4m3fn, the E2M1 grid, published Philox4x32-10 known-answer
 * vectors, H*H^T = 16 I, brute-force nearest-grid search, FP64 matmul on tiny
 * shapes, exact special cases).
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_OK = 0, ORACLE_ERR_INVALID_ARG = 1, ORACLE_ERR_UNSUPPORTED_SHAPE = 2,
       ORACLE_ERR_NONFINITE = 6 };

typedef struct oracle_cfg {
  int32_t block;      /* 0: 1x16 blocks along K, 1: 16x16 tiles            */
  int32_t rounding;   /* 0: round to nearest even, 1: stochastic rounding  */
  int32_t rht;        /* 1: apply the 16-point random Hadamard transform   */
  int32_t transpose;  /* 1: quantise x^T (blocks run down the rows of x)    */
  uint64_t rht_seed;
  uint64_t sr_seed;
  uint64_t sr_offset;
} oracle_cfg;

/* Codecs */
double  oracle_e2m1_value(uint8_t code);
double  oracle_e4m3_value(uint8_t byte);
uint8_t oracle_e4m3_encode(float t);             /* RNE, saturating, t >= 0 */
uint8_t oracle_e2m1_encode_rne(float v);
uint8_t oracle_e2m1_encode_sr(float v, uint32_t r);

/* Philox4x32-10 */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Random Hadamard transform of one 16-vector, in place. */
void oracle_rht_signs(uint64_t seed, float sigma[16]);
void oracle_rht16(float v[16], const float sigma[16]);

/* Quantise x (BF16 bit patterns, [rows, cols], row stride ld elements).
 * The quantised operand Q has qr = rows, qk = cols (or qr = cols, qk = rows
 * when transposed).  codes: [qr, qk/2] bytes; sf: [qr, qk/16] bytes row-major.
 */
int oracle_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                    const oracle_cfg* cfg, uint8_t* codes, uint8_t* sf, float* tensor_scale);

/* Same, encoding only rows [row_begin, row_end) of Q (the tensor scale is
 * still that of the whole operand); codes / sf receive just those rows. */
int oracle_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, const oracle_cfg* cfg,
                         int64_t row_begin, int64_t row_end, uint8_t* codes, uint8_t* sf, float* tensor_scale);

/* Delayed scaling: as oracle_quantize, but the tensor scale is amax / 2688
 * for a caller-supplied amax instead of the operand's own (elements above it
 * saturate).  The operand must be finite. */
int oracle_quantize_given_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                               const oracle_cfg* cfg, float amax, uint8_t* codes, uint8_t* sf,
                               float* tensor_scale);

/* Amax of the (optionally transformed) operand, as the quantiser sees it. */
int oracle_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                const oracle_cfg* cfg, float* amax);

/* Byte offset of scale (r, kb) in the tensor-core scale layout, and that
 * layout's padded size for a [qr, qk] operand. */
int64_t oracle_sf_mma_offset(int64_t r, int64_t kb, int64_t qk);
int64_t oracle_sf_mma_bytes(int64_t qr, int64_t qk);
/* Row-major scales [qr, qk/16] -> the padded tensor-core layout. */
void oracle_sf_to_mma(const uint8_t* sf, int64_t qr, int64_t qk, uint8_t* out);

/* y[i, k] = e2m1(code) * e4m3(sf) * tensor_scale, in FP64. */
void oracle_dequantize(const uint8_t* codes, const uint8_t* sf, float tensor_scale,
                       int64_t qr, int64_t qk, double* out);

/* ref[m, n] = sum_k deqA[m, k] * deqB[n, k] in FP64 (plain triple loop). */
void oracle_gemm_f64(const uint8_t* a_codes, const uint8_t* a_sf, float a_scale,
                     const uint8_t* b_codes, const uint8_t* b_sf, float b_scale,
                     int64_t M, int64_t N, int64_t K, double* out);

/* The same sum for a list of (m, n) output coordinates only. */
void oracle_gemm_f64_sampled(const uint8_t* a_codes, const uint8_t* a_sf, float a_scale,
                             const uint8_t* b_codes, const uint8_t* b_sf, float b_scale,
                             int64_t K, const int64_t* m_idx, const int64_t* n_idx,
                             int64_t count, double* out);

/* Quantised AdamW state codec (first moment m, second moment v); see oracle.c. */
void oracle_rht16_inverse(float v[16], const float sigma[16]);
uint16_t oracle_bf16_rne(float f);
int oracle_qadamw_m_encode(const float* m, int64_t rows, int64_t cols, uint64_t rht_seed, uint64_t sr_seed,
                           uint64_t sr_offset, uint8_t* codes, uint8_t* sf, float* tensor_scale);
void oracle_qadamw_m_decode(const uint8_t* codes, const uint8_t* sf, float tensor_scale, int64_t rows, int64_t cols,
                            uint64_t rht_seed, float* m_out);
int oracle_qadamw_v_encode(const float* v, int64_t rows, int64_t cols, uint64_t rht_seed, uint8_t* codes, uint8_t* sf,
                           float* tensor_scale, uint16_t* tile_mean);
void oracle_qadamw_v_decode(const uint8_t* codes, const uint8_t* sf, float tensor_scale, const uint16_t* tile_mean,
                            int64_t rows, int64_t cols, uint64_t rht_seed, float* v_out);

/* LoRA-SVD projection forward: NVFP4 GEMM of X and W_res plus beta * BF16(X L1^T) L2^T, in FP64.
 * oracle_lora_down gives the branch's intermediate U = BF16(X L1^T) [T, r] and its exact FP64 sums
 * (either output may be NULL); the sampled form evaluates Y at (t_idx[c], n_idx[c]) only. */
void oracle_lora_down(const uint16_t* x, const uint16_t* l1, int64_t T, int64_t din, int64_t r, uint16_t* u_bf16,
                      double* u_exact);
void oracle_lora_forward_sampled(const uint8_t* xq_codes, const uint8_t* xq_sf, float xq_scale,
                                 const uint8_t* wq_codes, const uint8_t* wq_sf, float wq_scale, const uint16_t* x,
                                 const uint16_t* l1, const uint16_t* l2, double beta, int64_t din, int64_t r,
                                 const int64_t* t_idx, const int64_t* n_idx, int64_t count, double* out);
void oracle_lora_forward(const uint8_t* xq_codes, const uint8_t* xq_sf, float xq_scale, const uint8_t* wq_codes,
                         const uint8_t* wq_sf, float wq_scale, const uint16_t* x, const uint16_t* l1,
                         const uint16_t* l2, double beta, int64_t T, int64_t din, int64_t dout, int64_t r,
                         double* out);

/* Nearest-rank percentile p (0..100] of |x| over n BF16 values, and clipping to [-c, c]. */
float oracle_abs_percentile_bf16(const uint16_t* x, int64_t n, double p);
void oracle_clip_bf16(const uint16_t* x, int64_t n, float c, uint16_t* out);

/* Newton-Schulz step of the Root optimizer with NVFP4 products (see oracle.c for the reading).
 * x, out: BF16 [m, n]; m % 32 == 0, n % 32 == 0.  trace (may be NULL) receives the clip
 * thresholds and, where its pointers are not NULL, the step's BF16 intermediates. */
uint16_t oracle_bf16_rne_f64(double d);
void oracle_axpby_bf16(const uint16_t* x, const uint16_t* y, int64_t n, float a, float b, uint16_t* out);
typedef struct oracle_ns_trace {
  float qx, qa, qb;  /* p-th percentile magnitudes of X, A and B */
  uint16_t* xc;      /* [m, n]  X clipped                         */
  uint16_t* a;       /* [m, m]  A = Q(Xc) Q(Xc)^T                 */
  uint16_t* ac;      /* [m, m]  A clipped                         */
  uint16_t* a2;      /* [m, m]  Q(Ac) Q(Ac)^T                     */
  uint16_t* b;       /* [m, m]  B = b A + c A2                    */
  uint16_t* bc;      /* [m, m]  B clipped                         */
  uint16_t* bx;      /* [m, n]  Q(Bc) Q(Xc^T)^T                   */
} oracle_ns_trace;
int oracle_ns_step(const uint16_t* x, int64_t m, int64_t n, float a, float b, float c, double p, uint16_t* out,
                   oracle_ns_trace* trace);

#ifdef __cplusplus
}
#endif
#endif
