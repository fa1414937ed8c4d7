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
};

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream);

int device_sm_count();

// cuTensorMapEncodeTiled from the driver (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace nvfp4
