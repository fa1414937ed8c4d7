// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// Every workspace starts with a 256-byte header; its first 32-bit word is the
// device status word.  The quantiser's scratch follows the header.
constexpr size_t kWsHeaderBytes = 256;
// Partial amax slots: the amax pass writes one per CTA and per output
// (at most kMaxQuantOutputs outputs of kPartialsPerOutput slots each).
constexpr int kMaxAmaxPartials = 4096;
constexpr int kMaxQuantOutputs = 2;
constexpr int kPartialsPerOutput = kMaxAmaxPartials / kMaxQuantOutputs;
constexpr size_t kQuantScratchBytes = kMaxAmaxPartials * sizeof(uint32_t);

// One quantised output of a BF16 tensor: Q = x (transpose 0) or Q = x^T.
struct QuantOut {
  int block2d, sr, rht, transpose, sf_mma;
  uint64_t rht_seed, sr_seed, sr_offset;
  uint8_t* codes;
  uint8_t* sf;
  float* tensor_scale;
  const float* amax_in;  // device; null: the amax pass scans the operand
};

// One read of x [rows, cols] (row-major, leading dimension ldx) produces
// n_out (1 or 2) quantised outputs.
struct QuantArgs {
  const uint16_t* x;   // BF16 input
  int64_t rows, cols, ldx;
  int n_out;
  QuantOut out[kMaxQuantOutputs];
  uint32_t* status;    // device status word
  uint32_t* partials;  // kMaxAmaxPartials slots
  // failure-detection test hook (see nvfp4_debug_quantize_skip_load): 1 or 2
  // makes CTA 0 of the amax (1) or encode (2) pass leave its first stage
  // unfilled, so its bounded wait runs out; 0 = off
  int skip_load_pass;
};

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t stream);
// Same launch with the status word and partial-amax scratch taken from a
// file-scope device array instead of a caller workspace.
cudaError_t launch_quantize_noalloc(QuantArgs a, cudaStream_t stream);
// Largest operand (elements) the scratch-free quantiser accepts.
constexpr int64_t kNoAllocMaxElements = int64_t(1) << 31;

struct DequantArgs {
  const uint8_t* codes;
  const uint8_t* sf;
  const float* tensor_scale;
  int64_t rows, k;
  int sf_mma;
  int out_f32;
  void* out;
  int64_t ldo;
};

cudaError_t launch_dequantize(const DequantArgs& a, cudaStream_t stream);

struct GemmArgs {
  const uint8_t* a_codes;
  const uint8_t* a_sf;
  const float* a_scale;
  const uint8_t* b_codes;
  const uint8_t* b_sf;
  const float* b_scale;
  int64_t M, N, K;
  int out_f32;
  void* d;
  int64_t ldd;
  uint32_t* status;
  int skip_first_load;  // failure-detection test hook (see nvfp4_debug_gemm_skip_load)
  // quantising epilogue (nvfp4_gemm_quantize): D's codes and block scales
  int quant;
  uint8_t* q_codes;
  uint8_t* q_sf;
  float* q_tensor_scale;
  const float* q_amax_in;
  float* q_amax_out;
  int q_sf_mma;
  // LoRA-SVD branch (nvfp4_lora_forward): extra BF16 k-blocks after the NVFP4
  // ones, A from lora_uhl [M, 2 lora_rpad] (hi / lo of (beta / alpha) U per 64
  // columns), B from lora_l2 [N, lora_r]; lora_r == 0: none
  const uint16_t* lora_uhl;
  const uint16_t* lora_l2;
  int64_t lora_r, lora_rpad;
  // split-K scratch (FP32 partial accumulators) for outputs with too few
  // tiles; null or too small: no split
  float* partial;
  size_t partial_bytes;
};

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream);
// Number of K splits launch_gemm uses for a GEMM shape (1: none), and the
// k-blocks (256 of K) per split.
int gemm_split_k(int64_t M, int64_t N, int64_t K, int* kb_per_split);
// Bytes of split-K scratch for that many splits (whole 128 x 256 FP32 blocks).
size_t gemm_split_k_bytes(int64_t M, int64_t N, int split_k);
// How launch_gemm schedules a plain (no LoRA, no quantising epilogue) GEMM
// shape given that many bytes of partial-sum scratch.
struct GemmPlan {
  int pair;                     // 1: CTA pairs on 256 x 256 tiles; 0: single CTAs on 128 x 256
  int ctas;                     // CTAs launched
  int units;                    // work units (tiles, split-K pieces or tail pieces)
  int split_k;                  // single mode: K splits (1: none)
  int kb_per_unit;              // k-blocks (256 of K) per split-K unit; num_kb otherwise
  int tail_tiles;               // pair mode: tiles past the last whole wave cut along K (0: none)
  int tail_split;               // pieces per tail tile
  int tail_kb;                  // k-blocks per tail piece
  size_t partial_bytes_needed;  // scratch the split would take (0: no split applies)
};
cudaError_t gemm_plan(int64_t M, int64_t N, int64_t K, size_t partial_bytes, GemmPlan* plan);

// LoRA-SVD branch, first half (lora.cu): U = BF16(X L1^T) and the hi / lo
// split of (beta / (sx sw)) U that the GEMM adds into its accumulator.
struct LoraArgs {
  const uint16_t* x;   // BF16 [T, din], row stride ldx
  int64_t T, din, ldx;
  const uint16_t* l1;  // BF16 [r, din] dense
  int64_t r;
  float beta;
  const float* sx;     // tensor scales of Q(X) and Q(W_res) (device)
  const float* sw;
  uint16_t* u;         // out: U [T, r]
  uint16_t* uhl;       // out: [T, 2 rpad], rpad = r rounded up to 64
  uint32_t* status;
};
cudaError_t launch_lora_down(const LoraArgs& a, cudaStream_t stream);
// Tensor map over a BF16 matrix: box 64 columns x box_rows, 128-byte swizzle.
bool make_lora_bf16_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                        uint32_t box_rows);

// Quantised AdamW state codec (qadamw.cu).
struct QadamwArgs {
  enum Op { kMEncode, kMDecode, kVEncode, kVDecode } op;
  const float* in;           // m or v (encode)
  float* out;                // m_hat or v_hat (decode)
  uint8_t* codes;            // [rows, cols/2]
  uint8_t* sf;               // [rows, cols/16] row-major
  float* tensor_scale;       // written by the encoders
  const float* tensor_scale_in;
  uint16_t* mean;            // v tile means, BF16 bits (v encode)
  const uint16_t* mean_in;   // (v decode)
  int64_t rows, cols;
  uint64_t rht_seed, sr_seed, sr_offset;
  void* workspace;           // encoders: status word + amax word
};
cudaError_t launch_qadamw(const QadamwArgs& a, cudaStream_t stream);

// Newton-Schulz step pieces (ns.cu).  hist: 384 zero-initialised (by the
// launcher) counters; q receives the k-th smallest |x| (1-based k).
cudaError_t launch_abs_percentile(const uint16_t* x, int64_t n, uint64_t k, uint32_t* hist, float* q,
                                  uint32_t* status, cudaStream_t stream);
constexpr size_t kPercentileHistBytes = 384 * sizeof(uint32_t);
cudaError_t launch_clip(const uint16_t* x, int64_t n, const float* q, uint16_t* out, cudaStream_t stream);
// Percentile selection and clip together (the selection runs in the clip
// kernel's blocks; q receives the threshold).
cudaError_t launch_percentile_clip(const uint16_t* x, int64_t n, uint64_t k, uint32_t* hist, float* q, uint16_t* out,
                                   uint32_t* status, cudaStream_t stream);
cudaError_t launch_axpby(const uint16_t* x, const uint16_t* y, int64_t n, float a, float b, uint16_t* out,
                         cudaStream_t stream);

int device_sm_count();

// Sign words of the 16-point transform: sigma_j = -1 (word 0x80000000, the
// FP32 sign bit) iff bit j of word 0 of Philox4x32-10(key = seed, counter 0);
// all zero when `on` is false.  Host code, the same generator the kernels run.
inline void rht_sign_words(uint64_t seed, bool on, uint32_t out[16]) {
  uint32_t c0 = 0, c1 = 0, c2 = 0, c3 = 0;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ k0, n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ k1;
    c1 = static_cast<uint32_t>(p1);
    c3 = static_cast<uint32_t>(p0);
    c0 = n0;
    c2 = n2;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  for (int j = 0; j < 16; ++j) out[j] = (on && ((c0 >> j) & 1u)) ? 0x80000000u : 0u;
}

// Weyl key schedule of Philox4x32-10 for a 64-bit key, one pair per round.
inline void philox_round_keys(uint64_t key, uint32_t rk0[10], uint32_t rk1[10]) {
  uint32_t k0 = static_cast<uint32_t>(key), k1 = static_cast<uint32_t>(key >> 32);
  for (int i = 0; i < 10; ++i) {
    rk0[i] = k0;
    rk1[i] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

// cuTensorMapEncodeTiled from the driver (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace nvfp4
