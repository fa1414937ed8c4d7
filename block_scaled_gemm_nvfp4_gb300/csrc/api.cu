// libnvfp4 C ABI: argument validation, workspace layout, launches and the
// linear-layer wrappers.  Nothing here computes on the host; every step of
// the path runs in the kernels of quantize.cu, dequantize.cu and gemm.cu.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
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
                       uint32_t* status, cudaStream_t stream, float* partial = nullptr, size_t partial_bytes = 0) {
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
  g.partial = partial;
  g.partial_bytes = partial_bytes;
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
  // scratch for the split the GEMM would make with unlimited workspace (none
  // where no CUDA device can be queried: the GEMM then runs unsplit)
  GemmPlan g;
  if (gemm_plan(M, N, K, SIZE_MAX, &g) == cudaSuccess && g.partial_bytes_needed > 0)
    *bytes += align_up(g.partial_bytes_needed);
  return NVFP4_OK;
}

nvfp4_status nvfp4_gemm_plan(int64_t M, int64_t N, int64_t K, size_t workspace_bytes, int64_t* plan) {
  if (!plan || M < 0 || N < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
  if (K % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  GemmPlan g;
  const size_t part = workspace_bytes > kWsHeaderBytes ? workspace_bytes - kWsHeaderBytes : 0;
  const cudaError_t e = gemm_plan(M, N, K, part, &g);
  if (e != cudaSuccess) return cuda_status(e);
  plan[0] = g.pair;
  plan[1] = g.ctas;
  plan[2] = g.units;
  plan[3] = g.split_k;
  plan[4] = g.kb_per_unit;
  plan[5] = g.tail_tiles;
  plan[6] = g.tail_split;
  plan[7] = g.tail_kb;
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
  // Anything past the header is split-K scratch; a workspace of just the
  // header runs the GEMM unsplit.
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return gemm_into(a, b, out_dtype, d, ldd, reinterpret_cast<uint32_t*>(ws), reinterpret_cast<cudaStream_t>(stream),
                   reinterpret_cast<float*>(ws + kWsHeaderBytes), workspace_bytes - kWsHeaderBytes);
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

// ------------------------------------------------------- LoRA-SVD projection
static int64_t lora_rpad(int64_t r) { return (r + 63) / 64 * 64; }

nvfp4_status nvfp4_lora_workspace_size(int64_t tokens, int64_t rank, size_t* bytes) {
  if (!bytes || tokens < 0) return NVFP4_ERR_INVALID_ARG;
  if (rank < 8 || rank > 256 || rank % 8 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  *bytes = kWsHeaderBytes + align_up(static_cast<size_t>(tokens) * 2 * lora_rpad(rank) * 2);
  return NVFP4_OK;
}

nvfp4_status nvfp4_lora_forward(const nvfp4_tensor* xq, const nvfp4_tensor* wq, const void* x, int64_t ldx,
                                const void* l1, const void* l2, int64_t rank, float beta, int32_t out_dtype, void* y,
                                int64_t ldy, void* u, void* workspace, size_t workspace_bytes,
                                nvfp4_stream_t stream) {
  nvfp4_status s = check_tensor(xq);
  if (s != NVFP4_OK) return s;
  s = check_tensor(wq);
  if (s != NVFP4_OK) return s;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_INVALID_ARG;
  if (xq->k != wq->k) return NVFP4_ERR_INVALID_ARG;
  const int64_t T = xq->rows, din = xq->k, dout = wq->rows;
  if (din % 32 != 0 || din == 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (rank < 8 || rank > 256 || rank % 8 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (xq->sf_layout != NVFP4_SF_MMA || wq->sf_layout != NVFP4_SF_MMA) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (T > (int64_t(1) << 31) || dout > (int64_t(1) << 31) || din > (int64_t(1) << 31))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!(beta == beta) || beta - beta != 0.0f) return NVFP4_ERR_INVALID_ARG;  // NaN or inf
  if (T == 0 || dout == 0) return NVFP4_OK;
  if (!x || !l1 || !l2 || !u || !y) return NVFP4_ERR_INVALID_ARG;
  if (ldx < din || ldx % 8 != 0 || !aligned16(x) || !aligned16(l1) || !aligned16(l2) || !aligned16(u))
    return NVFP4_ERR_INVALID_ARG;
  if (ldy < dout) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(xq->codes) || !aligned16(wq->codes) || !aligned16(xq->sf) || !aligned16(wq->sf))
    return NVFP4_ERR_INVALID_ARG;
  size_t need = 0;
  s = nvfp4_lora_workspace_size(T, rank, &need);
  if (s != NVFP4_OK) return s;
  if (!workspace || workspace_bytes < need) return NVFP4_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return NVFP4_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint16_t* uhl = reinterpret_cast<uint16_t*>(ws + kWsHeaderBytes);
  LoraArgs la{};
  la.x = static_cast<const uint16_t*>(x);
  la.T = T;
  la.din = din;
  la.ldx = ldx;
  la.l1 = static_cast<const uint16_t*>(l1);
  la.r = rank;
  la.beta = beta;
  la.sx = xq->tensor_scale;
  la.sw = wq->tensor_scale;
  la.u = static_cast<uint16_t*>(u);
  la.uhl = uhl;
  la.status = status;
  cudaError_t e = launch_lora_down(la, st);
  if (e == cudaErrorInvalidValue) return NVFP4_ERR_INVALID_ARG;
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  GemmArgs g{};
  g.a_codes = static_cast<const uint8_t*>(xq->codes);
  g.a_sf = static_cast<const uint8_t*>(xq->sf);
  g.a_scale = xq->tensor_scale;
  g.b_codes = static_cast<const uint8_t*>(wq->codes);
  g.b_sf = static_cast<const uint8_t*>(wq->sf);
  g.b_scale = wq->tensor_scale;
  g.M = T;
  g.N = dout;
  g.K = din;
  g.out_f32 = out_dtype == NVFP4_OUT_F32;
  g.d = y;
  g.ldd = ldy;
  g.status = status;
  g.skip_first_load = g_skip_load_once.exchange(0);
  g.lora_uhl = uhl;
  g.lora_l2 = static_cast<const uint16_t*>(l2);
  g.lora_r = rank;
  g.lora_rpad = lora_rpad(rank);
  e = launch_gemm(g, st);
  if (e == cudaErrorInvalidValue) return NVFP4_ERR_INVALID_ARG;
  return cuda_status(e);
}

// ------------------------------------------- Newton-Schulz step (Q-Root)
static bool percentile_rank(int64_t n, double p, uint64_t* k) {
  // nearest rank: the k-th smallest of n with k = ceil(p / 100 * n), 1 <= k <= n
  if (!(p > 0.0 && p <= 100.0)) return false;
  int64_t r = static_cast<int64_t>(std::ceil(p / 100.0 * static_cast<double>(n)));
  if (r < 1) r = 1;
  if (r > n) r = n;
  *k = static_cast<uint64_t>(r);
  return true;
}

static size_t percentile_ws_bytes() { return kWsHeaderBytes + align_up(kPercentileHistBytes); }

nvfp4_status nvfp4_abs_percentile_workspace_size(size_t* bytes) {
  if (!bytes) return NVFP4_ERR_INVALID_ARG;
  *bytes = percentile_ws_bytes();
  return NVFP4_OK;
}

nvfp4_status nvfp4_abs_percentile_bf16(const void* x, int64_t n, double p, float* q, void* workspace,
                                       size_t workspace_bytes, nvfp4_stream_t stream) {
  if (!q || n < 0 || n > (int64_t(1) << 40)) return NVFP4_ERR_INVALID_ARG;
  uint64_t k = 0;
  if (n > 0 && !percentile_rank(n, p, &k)) return NVFP4_ERR_INVALID_ARG;
  if (n > 0 && (!x || !aligned16(x))) return NVFP4_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < percentile_ws_bytes()) return NVFP4_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return NVFP4_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n == 0) return cuda_status(cudaMemsetAsync(q, 0, sizeof(float), st));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return cuda_status(launch_abs_percentile(static_cast<const uint16_t*>(x), n, k,
                                           reinterpret_cast<uint32_t*>(ws + kWsHeaderBytes), q,
                                           reinterpret_cast<uint32_t*>(ws), st));
}

nvfp4_status nvfp4_clip_bf16(const void* x, int64_t n, const float* q, void* out, nvfp4_stream_t stream) {
  if (!q || n < 0) return NVFP4_ERR_INVALID_ARG;
  if (n == 0) return NVFP4_OK;
  if (!x || !out || !aligned16(x) || !aligned16(out)) return NVFP4_ERR_INVALID_ARG;
  return cuda_status(launch_clip(static_cast<const uint16_t*>(x), n, q, static_cast<uint16_t*>(out),
                                 reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_axpby_bf16(const void* x, const void* y, int64_t n, float a, float b, void* out,
                              nvfp4_stream_t stream) {
  if (n < 0) return NVFP4_ERR_INVALID_ARG;
  if (n == 0) return NVFP4_OK;
  if (!x || !y || !out || !aligned16(x) || !aligned16(y) || !aligned16(out)) return NVFP4_ERR_INVALID_ARG;
  return cuda_status(launch_axpby(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(y), n, a, b,
                                  static_cast<uint16_t*>(out), reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
// Workspace of nvfp4_ns_step, in order (each part 256-byte aligned): header,
// three percentile histograms, three clip thresholds, quantiser scratch,
// Xc [m, n], A, Ac, A A^T, B, Bc [m, m], B X [m, n], and the quantised
// operands Q(Xc) [m, n], Q(Xc^T) [n, m], Q(Ac), Q(Bc) [m, m].
struct NsLayout {
  size_t hist, q, partials, xc, a, ac, a2, b, bc, bx, qx, qxt, qa, qb, total;
};
NsLayout ns_layout(int64_t m, int64_t n) {
  NsLayout L{};
  size_t off = kWsHeaderBytes;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  const size_t mn2 = static_cast<size_t>(m) * n * 2, mm2 = static_cast<size_t>(m) * m * 2;
  L.hist = take(3 * kPercentileHistBytes);
  L.q = take(3 * sizeof(float));
  L.partials = take(kQuantScratchBytes);
  L.xc = take(mn2);
  L.a = take(mm2);
  L.ac = take(mm2);
  L.a2 = take(mm2);
  L.b = take(mm2);
  L.bc = take(mm2);
  L.bx = take(mn2);
  L.qx = off;
  off += operand_bytes(m, n);
  L.qxt = off;
  off += operand_bytes(n, m);
  L.qa = off;
  off += operand_bytes(m, m);
  L.qb = off;
  off += operand_bytes(m, m);
  L.total = off;
  return L;
}
}  // namespace

nvfp4_status nvfp4_ns_workspace_size(int64_t m, int64_t n, size_t* bytes) {
  if (!bytes || m < 0 || n < 0) return NVFP4_ERR_INVALID_ARG;
  if (m == 0 || n == 0 || m % 32 != 0 || n % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (m > (int64_t(1) << 20) || n > (int64_t(1) << 20)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  *bytes = ns_layout(m, n).total;
  return NVFP4_OK;
}

nvfp4_status nvfp4_ns_step(const void* x, int64_t m, int64_t n, float a, float b, float c, double p, void* x_out,
                           void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  size_t need = 0;
  nvfp4_status s = nvfp4_ns_workspace_size(m, n, &need);
  if (s != NVFP4_OK) return s;
  if (!x || !x_out || !aligned16(x) || !aligned16(x_out)) return NVFP4_ERR_INVALID_ARG;
  uint64_t kx = 0, ka = 0;
  if (!percentile_rank(m * n, p, &kx) || !percentile_rank(m * m, p, &ka)) return NVFP4_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need) return NVFP4_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return NVFP4_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const NsLayout L = ns_layout(m, n);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint32_t* partials = reinterpret_cast<uint32_t*>(ws + L.partials);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  float* q = reinterpret_cast<float*>(ws + L.q);
  auto bf = [&](size_t off) { return reinterpret_cast<uint16_t*>(ws + off); };
  uint8_t* cur = ws + L.qx;
  QuantizedOperand qx = carve_operand(cur, m, n);
  cur = ws + L.qxt;
  QuantizedOperand qxt = carve_operand(cur, n, m);
  cur = ws + L.qa;
  QuantizedOperand qa = carve_operand(cur, m, m);
  cur = ws + L.qb;
  QuantizedOperand qb = carve_operand(cur, m, m);
  const nvfp4_quant_cfg rows = default_cfg(NVFP4_BLOCK_1x16, NVFP4_ROUND_RNE, 0, 0);
  nvfp4_quant_cfg cols = rows;
  cols.transpose = 1;
  const uint16_t* xin = static_cast<const uint16_t*>(x);
  cudaError_t e;
#define NS_TRY(call)                        \
  do {                                      \
    e = (call);                             \
    if (e != cudaSuccess) return NVFP4_ERR_CUDA; \
  } while (0)
  // Xc = clip(X); Q(Xc) along n and Q(Xc^T) along m from one read
  NS_TRY(launch_percentile_clip(xin, m * n, kx, hist, q, bf(L.xc), status, st));
  {
    QuantArgs qa2{};
    qa2.x = bf(L.xc);
    qa2.rows = m;
    qa2.cols = n;
    qa2.ldx = n;
    qa2.n_out = 2;
    qa2.out[0] = make_out(rows, qx.codes, qx.sf, qx.scale);
    qa2.out[1] = make_out(cols, qxt.codes, qxt.sf, qxt.scale);
    qa2.status = status;
    qa2.partials = partials;
    NS_TRY(launch_quantize(qa2, st));
  }
  // A = Q(Xc) Q(Xc)^T
  nvfp4_tensor tx{qx.codes, qx.sf, qx.scale, m, n, NVFP4_SF_MMA, 0};
  s = gemm_into(&tx, &tx, NVFP4_OUT_BF16, bf(L.a), m, status, st);
  if (s != NVFP4_OK) return s;
  // A A^T from Q(clip(A))
  NS_TRY(launch_percentile_clip(bf(L.a), m * m, ka, hist + 384, q + 1, bf(L.ac), status, st));
  s = quantize_into(bf(L.ac), m, m, m, rows, qa.codes, qa.sf, qa.scale, status, partials, st);
  if (s != NVFP4_OK) return s;
  nvfp4_tensor ta{qa.codes, qa.sf, qa.scale, m, m, NVFP4_SF_MMA, 0};
  s = gemm_into(&ta, &ta, NVFP4_OUT_BF16, bf(L.a2), m, status, st);
  if (s != NVFP4_OK) return s;
  // B = b A + c A A^T; B X from Q(clip(B)) and Q(Xc^T)
  NS_TRY(launch_axpby(bf(L.a), bf(L.a2), m * m, b, c, bf(L.b), st));
  NS_TRY(launch_percentile_clip(bf(L.b), m * m, ka, hist + 768, q + 2, bf(L.bc), status, st));
  s = quantize_into(bf(L.bc), m, m, m, rows, qb.codes, qb.sf, qb.scale, status, partials, st);
  if (s != NVFP4_OK) return s;
  nvfp4_tensor tb{qb.codes, qb.sf, qb.scale, m, m, NVFP4_SF_MMA, 0};
  nvfp4_tensor txt{qxt.codes, qxt.sf, qxt.scale, n, m, NVFP4_SF_MMA, 0};
  s = gemm_into(&tb, &txt, NVFP4_OUT_BF16, bf(L.bx), n, status, st);
  if (s != NVFP4_OK) return s;
  // X' = a X + B X
  NS_TRY(launch_axpby(xin, bf(L.bx), m * n, a, 1.0f, static_cast<uint16_t*>(x_out), st));
#undef NS_TRY
  return NVFP4_OK;
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
// Workspace: [header | quantiser scratch | operand A | operand B | GEMM
// partial sums]; the last part is optional (a workspace without it runs the
// GEMM unsplit), so the minimum is linear_ws_min.
static size_t linear_ws_min(int64_t am, int64_t bn, int64_t k) {
  return kWsHeaderBytes + kQuantScratchBytes + operand_bytes(am, k) + operand_bytes(bn, k);
}
static size_t linear_ws(int64_t am, int64_t bn, int64_t k) {
  GemmPlan g;
  size_t part = 0;
  if (gemm_plan(am, bn, k, SIZE_MAX, &g) == cudaSuccess) part = align_up(g.partial_bytes_needed);
  return linear_ws_min(am, bn, k) + part;
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
  if (workspace_bytes < linear_ws_min(M, N, K)) return NVFP4_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint32_t* partials = reinterpret_cast<uint32_t*>(ws + kWsHeaderBytes);
  uint8_t* cursor = ws + kWsHeaderBytes + kQuantScratchBytes;
  QuantizedOperand qa = carve_operand(cursor, M, K);
  QuantizedOperand qb = carve_operand(cursor, N, K);
  const size_t used = static_cast<size_t>(cursor - ws);  // the rest holds the GEMM's partial sums
  s = quantize_into(a_src, a_rows, a_cols, a_cols, ca, qa.codes, qa.sf, qa.scale, status, partials, stream);
  if (s != NVFP4_OK) return s;
  s = quantize_into(b_src, b_rows, b_cols, b_cols, cb, qb.codes, qb.sf, qb.scale, status, partials, stream);
  if (s != NVFP4_OK) return s;
  nvfp4_tensor ta{qa.codes, qa.sf, qa.scale, M, K, NVFP4_SF_MMA, 0};
  nvfp4_tensor tb{qb.codes, qb.sf, qb.scale, N, K, NVFP4_SF_MMA, 0};
  return gemm_into(&ta, &tb, out_dtype, d, N, status, stream, reinterpret_cast<float*>(cursor),
                   workspace_bytes - used);
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
