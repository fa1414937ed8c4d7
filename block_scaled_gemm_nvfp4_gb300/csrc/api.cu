// libnvfp4 C ABI: argument validation, workspace layout, launches and the
// linear-layer wrappers.  Nothing here computes on the host; every step of
// the path runs in the kernels of quantize.cu, dequantize.cu and gemm.cu.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "internal.h"

namespace nvfp4 {

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  // One cached value per device ordinal (up to 64 devices).
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

namespace {

// One-shot failure-detection test hooks (nvfp4_debug_*_skip_load).
std::atomic<int> g_skip_load_once{0};
std::atomic<int> g_quant_skip_once{0};  // 0 off, 1 amax pass, 2 encode pass

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

nvfp4_status check_cfg(const nvfp4_quant_cfg* c) {
  if (!c) return NVFP4_ERR_INVALID_ARG;
  if (c->block != NVFP4_BLOCK_1x16 && c->block != NVFP4_BLOCK_16x16) return NVFP4_ERR_INVALID_ARG;
  if (c->rounding != NVFP4_ROUND_RNE && c->rounding != NVFP4_ROUND_SR) return NVFP4_ERR_INVALID_ARG;
  if (c->rht != 0 && c->rht != 1) return NVFP4_ERR_INVALID_ARG;
  if (c->transpose != 0 && c->transpose != 1) return NVFP4_ERR_INVALID_ARG;
  if (c->sf_layout != NVFP4_SF_ROWMAJOR && c->sf_layout != NVFP4_SF_MMA) return NVFP4_ERR_INVALID_ARG;
  if (c->reserved != 0) return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

nvfp4_status check_quant_shape(int64_t rows, int64_t cols, const nvfp4_quant_cfg* c) {
  if (rows < 0 || cols < 0) return NVFP4_ERR_INVALID_ARG;
  const int64_t qr = c->transpose ? cols : rows;
  const int64_t qk = c->transpose ? rows : cols;
  if (qk % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (c->block == NVFP4_BLOCK_16x16 && qr % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  // Philox counters address elements with 64-bit indices; keep every index
  // and byte offset well inside int64.
  if (qr > (int64_t(1) << 31) || qk > (int64_t(1) << 31)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return NVFP4_OK;
}

nvfp4_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

size_t quant_ws_bytes() { return kWsHeaderBytes + kQuantScratchBytes; }

struct QuantizedOperand {
  uint8_t* codes;
  uint8_t* sf;
  float* scale;
};

// Carve a quantised operand [qr, qk] (MMA scale layout) out of a workspace.
size_t operand_bytes(int64_t qr, int64_t qk) {
  return align_up(nvfp4_codes_bytes(qr, qk)) + align_up(nvfp4_sf_bytes(qr, qk, NVFP4_SF_MMA)) + kAlign;
}
QuantizedOperand carve_operand(uint8_t*& cursor, int64_t qr, int64_t qk) {
  QuantizedOperand o;
  o.codes = cursor;
  cursor += align_up(nvfp4_codes_bytes(qr, qk));
  o.sf = cursor;
  cursor += align_up(nvfp4_sf_bytes(qr, qk, NVFP4_SF_MMA));
  o.scale = reinterpret_cast<float*>(cursor);
  cursor += kAlign;
  return o;
}

QuantOut make_out(const nvfp4_quant_cfg& cfg, void* codes, void* sf, float* scale) {
  QuantOut o{};
  o.block2d = cfg.block == NVFP4_BLOCK_16x16;
  o.sr = cfg.rounding == NVFP4_ROUND_SR;
  o.rht = cfg.rht;
  o.transpose = cfg.transpose;
  o.sf_mma = cfg.sf_layout == NVFP4_SF_MMA;
  o.rht_seed = cfg.rht_seed;
  o.sr_seed = cfg.sr_seed;
  o.sr_offset = cfg.sr_offset;
  o.codes = static_cast<uint8_t*>(codes);
  o.sf = static_cast<uint8_t*>(sf);
  o.tensor_scale = scale;
  return o;
}

// Quantise with an explicit status word and scratch (used by the wrappers).
nvfp4_status quantize_into(const void* x, int64_t rows, int64_t cols, int64_t ldx, const nvfp4_quant_cfg& cfg,
                           void* codes, void* sf, float* scale, uint32_t* status, uint32_t* partials,
                           cudaStream_t stream) {
  QuantArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.rows = rows;
  a.cols = cols;
  a.ldx = ldx;
  a.n_out = 1;
  a.out[0] = make_out(cfg, codes, sf, scale);
  a.status = status;
  a.partials = partials;
  a.skip_load_pass = g_quant_skip_once.exchange(0);
  return cuda_status(launch_quantize(a, stream));
}

// Checks shared by the quantiser entry points: the input and one output.
nvfp4_status check_quant_call(const void* x, int64_t rows, int64_t cols, int64_t ldx, const nvfp4_quant_cfg* cfg,
                              const void* codes, const void* sf, const float* tensor_scale) {
  nvfp4_status s = check_cfg(cfg);
  if (s != NVFP4_OK) return s;
  s = check_quant_shape(rows, cols, cfg);
  if (s != NVFP4_OK) return s;
  if (!tensor_scale) return NVFP4_ERR_INVALID_ARG;
  const bool empty = rows == 0 || cols == 0;
  if (!empty && (!x || !codes || !sf)) return NVFP4_ERR_INVALID_ARG;
  if (ldx < cols) return NVFP4_ERR_INVALID_ARG;
  if (!empty && (!aligned16(x) || ldx % 8 != 0)) return NVFP4_ERR_INVALID_ARG;
  if (!empty && (reinterpret_cast<uintptr_t>(codes) & 7u)) return NVFP4_ERR_INVALID_ARG;
  if (!empty && cfg->sf_layout == NVFP4_SF_MMA && !aligned16(sf)) return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

nvfp4_status check_tensor(const nvfp4_tensor* t) {
  if (!t || !t->tensor_scale) return NVFP4_ERR_INVALID_ARG;
  if (t->rows < 0 || t->k < 0 || t->reserved != 0) return NVFP4_ERR_INVALID_ARG;
  // an empty operand may come with null code / scale pointers
  if ((t->rows > 0 && t->k > 0) && (!t->codes || !t->sf)) return NVFP4_ERR_INVALID_ARG;
  if (t->sf_layout != NVFP4_SF_ROWMAJOR && t->sf_layout != NVFP4_SF_MMA) return NVFP4_ERR_INVALID_ARG;
  if (t->k % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return NVFP4_OK;
}


nvfp4_status gemm_into(const nvfp4_tensor* a, const nvfp4_tensor* b, int32_t out_dtype, void* d, int64_t ldd,
                       uint32_t* status, cudaStream_t stream) {
  GemmArgs g{};
  g.a_codes = static_cast<const uint8_t*>(a->codes);
  g.a_sf = static_cast<const uint8_t*>(a->sf);
  g.a_scale = a->tensor_scale;
  g.b_codes = static_cast<const uint8_t*>(b->codes);
  g.b_sf = static_cast<const uint8_t*>(b->sf);
  g.b_scale = b->tensor_scale;
  g.M = a->rows;
  g.N = b->rows;
  g.K = a->k;
  g.out_f32 = out_dtype == NVFP4_OUT_F32;
  g.d = d;
  g.ldd = ldd;
  g.status = status;
  g.skip_first_load = g_skip_load_once.exchange(0);
  const cudaError_t e = launch_gemm(g, stream);
  if (e == cudaErrorInvalidValue) return NVFP4_ERR_INVALID_ARG;
  return cuda_status(e);
}

nvfp4_quant_cfg default_cfg(int block, int rounding, int rht, uint64_t sr_seed) {
  nvfp4_quant_cfg c{};
  c.block = block;
  c.rounding = rounding;
  c.rht = rht;
  c.sf_layout = NVFP4_SF_MMA;
  c.transpose = 0;
  c.rht_seed = NVFP4_DEFAULT_RHT_SEED;
  c.sr_seed = sr_seed;
  c.sr_offset = 0;
  return c;
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_TIMEOUT: return "device-side wait timed out";
    case NVFP4_ERR_NONFINITE: return "non-finite input";
  }
  return "unknown status";
}

int32_t nvfp4_version(void) { return 100; }

size_t nvfp4_codes_bytes(int64_t qr, int64_t qk) {
  if (qr <= 0 || qk <= 0) return 0;
  return static_cast<size_t>(qr) * static_cast<size_t>(qk / 2);
}

size_t nvfp4_sf_bytes(int64_t qr, int64_t qk, int32_t sf_layout) {
  if (qr <= 0 || qk <= 0) return 0;
  const int64_t kb = qk / 16;
  if (sf_layout == NVFP4_SF_MMA) return static_cast<size_t>((qr + 127) / 128) * static_cast<size_t>((kb + 3) / 4) * 512;
  return static_cast<size_t>(qr) * static_cast<size_t>(kb);
}

nvfp4_status nvfp4_quantize_workspace_size(int64_t rows, int64_t cols, const nvfp4_quant_cfg* cfg, size_t* bytes) {
  if (!bytes) return NVFP4_ERR_INVALID_ARG;
  nvfp4_status s = check_cfg(cfg);
  if (s != NVFP4_OK) return s;
  s = check_quant_shape(rows, cols, cfg);
  if (s != NVFP4_OK) return s;
  *bytes = quant_ws_bytes();
  return NVFP4_OK;
}

nvfp4_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, const nvfp4_quant_cfg* cfg,
                            void* codes, void* sf, float* tensor_scale, void* workspace, size_t workspace_bytes,
                            nvfp4_stream_t stream) {
  nvfp4_status s = check_quant_call(x, rows, cols, ldx, cfg, codes, sf, tensor_scale);
  if (s != NVFP4_OK) return s;
  if (!workspace) return NVFP4_ERR_WORKSPACE;
  if (workspace_bytes < quant_ws_bytes()) return NVFP4_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return NVFP4_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return quantize_into(x, rows, cols, ldx, *cfg, codes, sf, tensor_scale, reinterpret_cast<uint32_t*>(ws),
                       reinterpret_cast<uint32_t*>(ws + kWsHeaderBytes), reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                 const nvfp4_quant_cfg* cfg_a, void* codes_a, void* sf_a, float* tensor_scale_a,
                                 const nvfp4_quant_cfg* cfg_b, void* codes_b, void* sf_b, float* tensor_scale_b,
                                 void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  nvfp4_status s = check_quant_call(x, rows, cols, ldx, cfg_a, codes_a, sf_a, tensor_scale_a);
  if (s != NVFP4_OK) return s;
  s = check_quant_call(x, rows, cols, ldx, cfg_b, codes_b, sf_b, tensor_scale_b);
  if (s != NVFP4_OK) return s;
  if (!workspace) return NVFP4_ERR_WORKSPACE;
  if (workspace_bytes < quant_ws_bytes()) return NVFP4_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return NVFP4_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  QuantArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.rows = rows;
  a.cols = cols;
  a.ldx = ldx;
  a.n_out = 2;
  a.out[0] = make_out(*cfg_a, codes_a, sf_a, tensor_scale_a);
  a.out[1] = make_out(*cfg_b, codes_b, sf_b, tensor_scale_b);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.partials = reinterpret_cast<uint32_t*>(ws + kWsHeaderBytes);
  a.skip_load_pass = g_quant_skip_once.exchange(0);
  return cuda_status(launch_quantize(a, reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_quantize_given_amax(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                       const nvfp4_quant_cfg* cfg, const float* amax, void* codes, void* sf,
                                       float* tensor_scale, void* workspace, size_t workspace_bytes,
                                       nvfp4_stream_t stream) {
  nvfp4_status s = check_quant_call(x, rows, cols, ldx, cfg, codes, sf, tensor_scale);
  if (s != NVFP4_OK) return s;
  if (!amax) return NVFP4_ERR_INVALID_ARG;
  if (!workspace) return NVFP4_ERR_WORKSPACE;
  if (workspace_bytes < quant_ws_bytes()) return NVFP4_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return NVFP4_ERR_INVALID_ARG;
  QuantArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.rows = rows;
  a.cols = cols;
  a.ldx = ldx;
  a.n_out = 1;
  a.out[0] = make_out(*cfg, codes, sf, tensor_scale);
  a.out[0].amax_in = amax;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.partials = reinterpret_cast<uint32_t*>(ws + kWsHeaderBytes);
  a.skip_load_pass = g_quant_skip_once.exchange(0);
  return cuda_status(launch_quantize(a, reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                    const nvfp4_quant_cfg* cfg, void* codes, void* sf, float* tensor_scale,
                                    nvfp4_stream_t stream) {
  nvfp4_status s = check_quant_call(x, rows, cols, ldx, cfg, codes, sf, tensor_scale);
  if (s != NVFP4_OK) return s;
  if (rows > 0 && cols > kNoAllocMaxElements / rows) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  QuantArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.rows = rows;
  a.cols = cols;
  a.ldx = ldx;
  a.n_out = 1;
  a.out[0] = make_out(*cfg, codes, sf, tensor_scale);
  a.skip_load_pass = g_quant_skip_once.exchange(0);
  return cuda_status(launch_quantize_noalloc(a, reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_dequantize(const nvfp4_tensor* q, int32_t out_dtype, void* out, int64_t ldo,
                              nvfp4_stream_t stream) {
  nvfp4_status s = check_tensor(q);
  if (s != NVFP4_OK) return s;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_INVALID_ARG;
  if (!out || ldo < q->k) return NVFP4_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q->codes) & 7u) return NVFP4_ERR_INVALID_ARG;
  DequantArgs a{};
  a.codes = static_cast<const uint8_t*>(q->codes);
  a.sf = static_cast<const uint8_t*>(q->sf);
  a.tensor_scale = q->tensor_scale;
  a.rows = q->rows;
  a.k = q->k;
  a.sf_mma = q->sf_layout == NVFP4_SF_MMA;
  a.out_f32 = out_dtype == NVFP4_OUT_F32;
  a.out = out;
  a.ldo = ldo;
  return cuda_status(launch_dequantize(a, reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
  if (!bytes || M < 0 || N < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
  if (K % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  *bytes = kWsHeaderBytes;
  return NVFP4_OK;
}

nvfp4_status nvfp4_gemm(const nvfp4_tensor* a, const nvfp4_tensor* b, int32_t out_dtype, void* d, int64_t ldd,
                        void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  nvfp4_status s = check_tensor(a);
  if (s != NVFP4_OK) return s;
  s = check_tensor(b);
  if (s != NVFP4_OK) return s;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_INVALID_ARG;
  if (a->k != b->k) return NVFP4_ERR_INVALID_ARG;
  if (a->k % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->sf_layout != NVFP4_SF_MMA || b->sf_layout != NVFP4_SF_MMA) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->rows > (int64_t(1) << 31) || b->rows > (int64_t(1) << 31) || a->k > (int64_t(1) << 31))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->rows == 0 || b->rows == 0) return NVFP4_OK;  // empty output: nothing to compute
  if (!d || ldd < b->rows) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(a->codes) || !aligned16(b->codes) || !aligned16(a->sf) || !aligned16(b->sf))
    return NVFP4_ERR_INVALID_ARG;

  if (!workspace) return NVFP4_ERR_WORKSPACE;
  if (workspace_bytes < kWsHeaderBytes) return NVFP4_ERR_WORKSPACE;
  return gemm_into(a, b, out_dtype, d, ldd, static_cast<uint32_t*>(workspace),
                   reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_gemm_quantize(const nvfp4_tensor* a, const nvfp4_tensor* b, void* d, int64_t ldd,
                                 const nvfp4_quant_out* q, void* workspace, size_t workspace_bytes,
                                 nvfp4_stream_t stream) {
  nvfp4_status s = check_tensor(a);
  if (s != NVFP4_OK) return s;
  s = check_tensor(b);
  if (s != NVFP4_OK) return s;
  if (!q || q->reserved != 0 || !q->amax_in || !q->tensor_scale) return NVFP4_ERR_INVALID_ARG;
  if (q->sf_layout != NVFP4_SF_ROWMAJOR && q->sf_layout != NVFP4_SF_MMA) return NVFP4_ERR_INVALID_ARG;
  if (a->k != b->k) return NVFP4_ERR_INVALID_ARG;
  if (a->k % 32 != 0 || a->k == 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->sf_layout != NVFP4_SF_MMA || b->sf_layout != NVFP4_SF_MMA) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->rows > (int64_t(1) << 31) || b->rows > (int64_t(1) << 31) || a->k > (int64_t(1) << 31))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (b->rows % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;  // N: whole 16-byte code pieces per 32 columns
  if (a->rows == 0 || b->rows == 0) return NVFP4_OK;
  if (d && ldd < b->rows) return NVFP4_ERR_INVALID_ARG;
  if (!q->codes || !q->sf || !aligned16(q->codes)) return NVFP4_ERR_INVALID_ARG;
  if (q->sf_layout == NVFP4_SF_MMA && !aligned16(q->sf)) return NVFP4_ERR_INVALID_ARG;
  if (q->amax_out && (reinterpret_cast<uintptr_t>(q->amax_out) & 3u)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(a->codes) || !aligned16(b->codes) || !aligned16(a->sf) || !aligned16(b->sf))
    return NVFP4_ERR_INVALID_ARG;
  if (!workspace) return NVFP4_ERR_WORKSPACE;
  if (workspace_bytes < kWsHeaderBytes) return NVFP4_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (q->amax_out && cudaMemsetAsync(q->amax_out, 0, sizeof(float), st) != cudaSuccess) return NVFP4_ERR_CUDA;
  GemmArgs g{};
  g.a_codes = static_cast<const uint8_t*>(a->codes);
  g.a_sf = static_cast<const uint8_t*>(a->sf);
  g.a_scale = a->tensor_scale;
  g.b_codes = static_cast<const uint8_t*>(b->codes);
  g.b_sf = static_cast<const uint8_t*>(b->sf);
  g.b_scale = b->tensor_scale;
  g.M = a->rows;
  g.N = b->rows;
  g.K = a->k;
  g.out_f32 = 0;
  g.d = d;
  g.ldd = d ? ldd : b->rows;
  g.status = static_cast<uint32_t*>(workspace);
  g.skip_first_load = g_skip_load_once.exchange(0);
  g.quant = 1;
  g.q_codes = static_cast<uint8_t*>(q->codes);
  g.q_sf = static_cast<uint8_t*>(q->sf);
  g.q_tensor_scale = q->tensor_scale;
  g.q_amax_in = q->amax_in;
  g.q_amax_out = q->amax_out;
  g.q_sf_mma = q->sf_layout == NVFP4_SF_MMA;
  const cudaError_t e = launch_gemm(g, st);
  if (e == cudaErrorInvalidValue) return NVFP4_ERR_INVALID_ARG;
  return cuda_status(e);
}

// ------------------------------------------------------- optimizer states
static nvfp4_status qadamw_shape(const void* state, int64_t rows, int64_t cols, bool v) {
  if (rows < 0 || cols < 0) return NVFP4_ERR_INVALID_ARG;
  if (cols % 16 != 0 || (v && rows % 16 != 0)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (rows > 0 && cols > 0 && (!state || !aligned16(state))) return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

static nvfp4_status qadamw_codes(const void* codes, const void* sf, const void* scale, int64_t rows, int64_t cols) {
  if (!scale) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0 && (!codes || !sf || (reinterpret_cast<uintptr_t>(codes) & 7u))) return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

static nvfp4_status qadamw_ws(const void* workspace, size_t bytes) {
  if (!workspace || bytes < kWsHeaderBytes) return NVFP4_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

static nvfp4_status qadamw_run(const QadamwArgs& a, nvfp4_stream_t stream) {
  const cudaError_t e = launch_qadamw(a, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(e);
}

nvfp4_status nvfp4_qadamw_workspace_size(size_t* bytes) {
  if (!bytes) return NVFP4_ERR_INVALID_ARG;
  *bytes = kWsHeaderBytes;
  return NVFP4_OK;
}

nvfp4_status nvfp4_qadamw_m_encode(const float* m, int64_t rows, int64_t cols, uint64_t rht_seed, uint64_t sr_seed,
                                   uint64_t sr_offset, void* codes, void* sf, float* tensor_scale, void* workspace,
                                   size_t workspace_bytes, nvfp4_stream_t stream) {
  nvfp4_status s = qadamw_shape(m, rows, cols, false);
  if (s == NVFP4_OK) s = qadamw_codes(codes, sf, tensor_scale, rows, cols);
  if (s == NVFP4_OK) s = qadamw_ws(workspace, workspace_bytes);
  if (s != NVFP4_OK) return s;
  QadamwArgs a{};
  a.op = QadamwArgs::kMEncode;
  a.in = m;
  a.codes = static_cast<uint8_t*>(codes);
  a.sf = static_cast<uint8_t*>(sf);
  a.tensor_scale = tensor_scale;
  a.rows = rows;
  a.cols = cols;
  a.rht_seed = rht_seed;
  a.sr_seed = sr_seed;
  a.sr_offset = sr_offset;
  a.workspace = workspace;
  return qadamw_run(a, stream);
}

nvfp4_status nvfp4_qadamw_m_decode(const void* codes, const void* sf, const float* tensor_scale, int64_t rows,
                                   int64_t cols, uint64_t rht_seed, float* m_out, nvfp4_stream_t stream) {
  nvfp4_status s = qadamw_shape(m_out, rows, cols, false);
  if (s == NVFP4_OK) s = qadamw_codes(codes, sf, tensor_scale, rows, cols);
  if (s != NVFP4_OK) return s;
  QadamwArgs a{};
  a.op = QadamwArgs::kMDecode;
  a.out = m_out;
  a.codes = const_cast<uint8_t*>(static_cast<const uint8_t*>(codes));
  a.sf = const_cast<uint8_t*>(static_cast<const uint8_t*>(sf));
  a.tensor_scale_in = tensor_scale;
  a.rows = rows;
  a.cols = cols;
  a.rht_seed = rht_seed;
  return qadamw_run(a, stream);
}

nvfp4_status nvfp4_qadamw_v_encode(const float* v, int64_t rows, int64_t cols, uint64_t rht_seed, void* codes,
                                   void* sf, float* tensor_scale, void* tile_mean, void* workspace,
                                   size_t workspace_bytes, nvfp4_stream_t stream) {
  nvfp4_status s = qadamw_shape(v, rows, cols, true);
  if (s == NVFP4_OK) s = qadamw_codes(codes, sf, tensor_scale, rows, cols);
  if (s == NVFP4_OK && rows > 0 && cols > 0 && (!tile_mean || (reinterpret_cast<uintptr_t>(tile_mean) & 1u)))
    s = NVFP4_ERR_INVALID_ARG;
  if (s == NVFP4_OK) s = qadamw_ws(workspace, workspace_bytes);
  if (s != NVFP4_OK) return s;
  QadamwArgs a{};
  a.op = QadamwArgs::kVEncode;
  a.in = v;
  a.codes = static_cast<uint8_t*>(codes);
  a.sf = static_cast<uint8_t*>(sf);
  a.tensor_scale = tensor_scale;
  a.mean = static_cast<uint16_t*>(tile_mean);
  a.rows = rows;
  a.cols = cols;
  a.rht_seed = rht_seed;
  a.workspace = workspace;
  return qadamw_run(a, stream);
}

nvfp4_status nvfp4_qadamw_v_decode(const void* codes, const void* sf, const float* tensor_scale,
                                   const void* tile_mean, int64_t rows, int64_t cols, uint64_t rht_seed,
                                   float* v_out, nvfp4_stream_t stream) {
  nvfp4_status s = qadamw_shape(v_out, rows, cols, true);
  if (s == NVFP4_OK) s = qadamw_codes(codes, sf, tensor_scale, rows, cols);
  if (s == NVFP4_OK && rows > 0 && cols > 0 && (!tile_mean || (reinterpret_cast<uintptr_t>(tile_mean) & 1u)))
    s = NVFP4_ERR_INVALID_ARG;
  if (s != NVFP4_OK) return s;
  QadamwArgs a{};
  a.op = QadamwArgs::kVDecode;
  a.out = v_out;
  a.codes = const_cast<uint8_t*>(static_cast<const uint8_t*>(codes));
  a.sf = const_cast<uint8_t*>(static_cast<const uint8_t*>(sf));
  a.tensor_scale_in = tensor_scale;
  a.mean_in = static_cast<const uint16_t*>(tile_mean);
  a.rows = rows;
  a.cols = cols;
  a.rht_seed = rht_seed;
  return qadamw_run(a, stream);
}

// ------------------------------------------------------------ linear layer
// Workspace: [header | quantiser scratch | operand A | operand B].
static size_t linear_ws(int64_t am, int64_t bn, int64_t k) {
  return kWsHeaderBytes + kQuantScratchBytes + operand_bytes(am, k) + operand_bytes(bn, k);
}

static nvfp4_status linear_shape(int32_t op, int64_t tokens, int64_t din, int64_t dout, int64_t* M, int64_t* N,
                                 int64_t* K) {
  if (tokens < 0 || din < 0 || dout < 0) return NVFP4_ERR_INVALID_ARG;
  if (din % 32 != 0 || dout % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  switch (op) {
    case NVFP4_LINEAR_FPROP: *M = tokens; *N = dout; *K = din; break;
    case NVFP4_LINEAR_DGRAD: *M = tokens; *N = din; *K = dout; break;
    case NVFP4_LINEAR_WGRAD:
      if (tokens % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
      *M = dout; *N = din; *K = tokens; break;
    default: return NVFP4_ERR_INVALID_ARG;
  }
  return NVFP4_OK;
}

nvfp4_status nvfp4_linear_workspace_size(int32_t op, int64_t tokens, int64_t din, int64_t dout, size_t* bytes) {
  if (!bytes) return NVFP4_ERR_INVALID_ARG;
  int64_t M, N, K;
  nvfp4_status s = linear_shape(op, tokens, din, dout, &M, &N, &K);
  if (s != NVFP4_OK) return s;
  *bytes = linear_ws(M, N, K);
  return NVFP4_OK;
}

// Shared body: quantise A-source into operand A [M, K], B-source into operand
// B [N, K], then D = A * B^T.
static nvfp4_status run_linear(int32_t op, const void* a_src, int64_t a_rows, int64_t a_cols,
                               const nvfp4_quant_cfg& ca, const void* b_src, int64_t b_rows, int64_t b_cols,
                               const nvfp4_quant_cfg& cb, int64_t M, int64_t N, int64_t K, int32_t out_dtype,
                               void* d, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  (void)op;
  if (!a_src || !b_src || !d) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(a_src) || !aligned16(b_src)) return NVFP4_ERR_INVALID_ARG;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_INVALID_ARG;
  nvfp4_status s = check_cfg(&ca);
  if (s != NVFP4_OK) return s;
  s = check_cfg(&cb);
  if (s != NVFP4_OK) return s;
  s = check_quant_shape(a_rows, a_cols, &ca);
  if (s != NVFP4_OK) return s;
  s = check_quant_shape(b_rows, b_cols, &cb);
  if (s != NVFP4_OK) return s;
  if (!workspace) return NVFP4_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return NVFP4_ERR_INVALID_ARG;
  if (workspace_bytes < linear_ws(M, N, K)) return NVFP4_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint32_t* partials = reinterpret_cast<uint32_t*>(ws + kWsHeaderBytes);
  uint8_t* cursor = ws + kWsHeaderBytes + kQuantScratchBytes;
  QuantizedOperand qa = carve_operand(cursor, M, K);
  QuantizedOperand qb = carve_operand(cursor, N, K);
  s = quantize_into(a_src, a_rows, a_cols, a_cols, ca, qa.codes, qa.sf, qa.scale, status, partials, stream);
  if (s != NVFP4_OK) return s;
  s = quantize_into(b_src, b_rows, b_cols, b_cols, cb, qb.codes, qb.sf, qb.scale, status, partials, stream);
  if (s != NVFP4_OK) return s;
  nvfp4_tensor ta{qa.codes, qa.sf, qa.scale, M, K, NVFP4_SF_MMA, 0};
  nvfp4_tensor tb{qb.codes, qb.sf, qb.scale, N, K, NVFP4_SF_MMA, 0};
  return gemm_into(&ta, &tb, out_dtype, d, N, status, stream);
}

static nvfp4_quant_cfg role_cfg(const nvfp4_quant_cfg* user, const nvfp4_quant_cfg& dflt, int transpose) {
  nvfp4_quant_cfg c = user ? *user : dflt;
  c.transpose = transpose;
  c.sf_layout = NVFP4_SF_MMA;
  return c;
}

nvfp4_status nvfp4_linear_fprop(const void* x, const void* w, int64_t tokens, int64_t din, int64_t dout,
                                const nvfp4_quant_cfg* cfg_x, const nvfp4_quant_cfg* cfg_w, int32_t out_dtype,
                                void* y, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  int64_t M, N, K;
  nvfp4_status s = linear_shape(NVFP4_LINEAR_FPROP, tokens, din, dout, &M, &N, &K);
  if (s != NVFP4_OK) return s;
  const nvfp4_quant_cfg cx = role_cfg(cfg_x, default_cfg(NVFP4_BLOCK_1x16, NVFP4_ROUND_RNE, 0, 1), 0);
  const nvfp4_quant_cfg cw = role_cfg(cfg_w, default_cfg(NVFP4_BLOCK_16x16, NVFP4_ROUND_RNE, 0, 2), 0);
  return run_linear(NVFP4_LINEAR_FPROP, x, tokens, din, cx, w, dout, din, cw, M, N, K, out_dtype, y, workspace,
                    workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_linear_dgrad(const void* dy, const void* w, int64_t tokens, int64_t din, int64_t dout,
                                const nvfp4_quant_cfg* cfg_dy, const nvfp4_quant_cfg* cfg_w, int32_t out_dtype,
                                void* dx, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  int64_t M, N, K;
  nvfp4_status s = linear_shape(NVFP4_LINEAR_DGRAD, tokens, din, dout, &M, &N, &K);
  if (s != NVFP4_OK) return s;
  const nvfp4_quant_cfg cdy = role_cfg(cfg_dy, default_cfg(NVFP4_BLOCK_1x16, NVFP4_ROUND_RNE, 0, 3), 0);
  // W^T [din, dout] quantised along dout: the transposed read of W [dout, din].
  const nvfp4_quant_cfg cw = role_cfg(cfg_w, default_cfg(NVFP4_BLOCK_16x16, NVFP4_ROUND_RNE, 0, 4), 1);
  return run_linear(NVFP4_LINEAR_DGRAD, dy, tokens, dout, cdy, w, dout, din, cw, M, N, K, out_dtype, dx, workspace,
                    workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_linear_wgrad(const void* dy, const void* x, int64_t tokens, int64_t din, int64_t dout,
                                const nvfp4_quant_cfg* cfg_dy, const nvfp4_quant_cfg* cfg_x, int32_t out_dtype,
                                void* dw, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  int64_t M, N, K;
  nvfp4_status s = linear_shape(NVFP4_LINEAR_WGRAD, tokens, din, dout, &M, &N, &K);
  if (s != NVFP4_OK) return s;
  // dY^T [dout, T] and X^T [din, T], both along T with the transform and
  // stochastic rounding; the shared rht_seed makes the transforms cancel.
  const nvfp4_quant_cfg cdy = role_cfg(cfg_dy, default_cfg(NVFP4_BLOCK_1x16, NVFP4_ROUND_SR, 1, 5), 1);
  const nvfp4_quant_cfg cx = role_cfg(cfg_x, default_cfg(NVFP4_BLOCK_1x16, NVFP4_ROUND_SR, 1, 6), 1);
  return run_linear(NVFP4_LINEAR_WGRAD, dy, tokens, dout, cdy, x, tokens, din, cx, M, N, K, out_dtype, dw, workspace,
                    workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

void nvfp4_debug_gemm_skip_load(int32_t enable) { g_skip_load_once.store(enable ? 1 : 0); }

void nvfp4_debug_quantize_skip_load(int32_t pass) { g_quant_skip_once.store(pass == 1 || pass == 2 ? pass : 0); }

nvfp4_status nvfp4_check_device_status(const void* workspace, nvfp4_stream_t stream) {
  if (!workspace) return NVFP4_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (word == 0) return NVFP4_OK;
  const uint32_t zero = 0;
  if (cudaMemcpy(const_cast<void*>(workspace), &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  const uint32_t code = word & 0xFFu;
  if (code == NVFP4_ERR_TIMEOUT || code == NVFP4_ERR_NONFINITE) return static_cast<nvfp4_status>(code);
  return NVFP4_ERR_CUDA;
}

}  // extern "C"
