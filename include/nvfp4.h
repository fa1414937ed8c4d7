/*
 * libnvfp4 -- NVFP4 quantisation and block-scaled FP4 GEMM for GB300 (sm_103a).
 *
 * What the library computes (sources are the pages' titles and sections):
 *
 *  - NVFP4 is a 4-bit floating-point format with a sparse grid, used for the
 *    weights and activations that enter GEMMs while accumulators stay in
 *    FP32 ("NVIDIA acelera o pre-treinamento de LLM: NVFP4 no Blackwell em
 *    conjunto com JAX e MaxText", sections "Por que cada porcento e
 *    importante" and "Como o treinamento mixed-precision funciona com NVFP4").
 *    Values are brought into the grid's range by custom scaling (same page).
 *  - Element codes are E2M1 on {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6};
 *    every run of 16 elements along K has an E4M3 block scale (1x16 blocks),
 *    or every 16x16 tile shares one (16x16 blocks); the tensor has one FP32
 *    decode scale s = amax / (6 * 448).
 *  - Hadamard mixing before quantisation and stochastic rounding come from
 *    "Full-Stack FP4: Stable LLM Pretraining with Quantized Projections,
 *    Optimizers, and Attention", section 2.2.  Here: a 16-point random
 *    Hadamard transform 1/4 * H16 * diag(sigma) on each run of 16 along K,
 *    sigma drawn from a seeded Philox4x32-10 word, and stochastic rounding
 *    from a counter-based Philox4x32-10 stream.
 *  - The GEMM computes D = A * B^T on NVFP4 operands, both stored K-major,
 *    with FP32 accumulation and the two tensor scales applied in the
 *    epilogue; the NVFP4 GEMM speed-up on Blackwell Ultra is the subject of
 *    "NVFP4 Treina com Precisao de 16 Bits e a Velocidade de 4 Bits para
 *    Pre-treinamento em Grande Escala", TL;DR.
 *
 * Every rounding decision is a fixed sequence of IEEE FP32 operations, so the
 * quantised codes, block scales and stochastic-rounding draws are a
 * deterministic function of (input, configuration, seeds):
 *    s      = amax / 2688           (one FP32 division; 1 if that is zero)
 *    t      = (bamax / 6) / s        (two FP32 divisions)
 *    scale  = E4M3(t)                (round to nearest even, saturate at 448)
 *    v      = x / (scale * s)        (one FP32 multiply, one FP32 division)
 *    code   = E2M1(v)                (round to nearest even, or stochastic)
 * A zero block scale encodes its whole run as code 0.  A negative v that
 * rounds to zero is encoded 0x8.  Packing: element 2j of a row is the low
 * nibble of byte j, element 2j+1 the high nibble.
 *
 * Conventions for every call:
 *  - Ownership: the caller owns every buffer (device memory unless stated).
 *    The library never allocates device memory.
 *  - Execution: calls enqueue kernels on `stream` and return at once.
 *  - Errors: argument errors are returned before anything is launched.
 *    A launch failure returns NVFP4_ERR_CUDA.  Errors found on the device
 *    (non-finite input, a wait that ran out) are recorded in the status word
 *    at the start of the call's workspace; nvfp4_check_device_status reads
 *    and clears it.  Workspaces must be zero-filled once before first use.
 *  - Concurrency: calls that may run at the same time need separate
 *    workspaces.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvfp4_stream_t; /* same type as cudaStream_t */

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, bad stride       */
  NVFP4_ERR_UNSUPPORTED_SHAPE = 2, /* a shape rule below is broken             */
  NVFP4_ERR_WORKSPACE = 3,         /* workspace missing or too small           */
  NVFP4_ERR_CUDA = 4,              /* a CUDA call failed                       */
  NVFP4_ERR_TIMEOUT = 5,           /* a device-side wait ran out (device word) */
  NVFP4_ERR_NONFINITE = 6          /* input holds inf or NaN (device word)     */
} nvfp4_status;

typedef enum { NVFP4_BLOCK_1x16 = 0, NVFP4_BLOCK_16x16 = 1 } nvfp4_block;
typedef enum { NVFP4_ROUND_RNE = 0, NVFP4_ROUND_SR = 1 } nvfp4_rounding;
/* Block-scale storage.  ROWMAJOR: byte (r, kb) at r * (K/16) + kb.
 * MMA: the tensor-core layout the GEMM reads -- atoms of 128 rows x 4 scales
 * (512 bytes), ordered by row block then K block; inside an atom scale
 * (r, j) is at byte (r % 32) * 16 + (r / 32) * 4 + j.  Rows are padded to a
 * multiple of 128 and scale columns to a multiple of 4; padding holds 0. */
typedef enum { NVFP4_SF_ROWMAJOR = 0, NVFP4_SF_MMA = 1 } nvfp4_sf_layout;
typedef enum { NVFP4_OUT_BF16 = 0, NVFP4_OUT_F32 = 1 } nvfp4_out_dtype;

/* Quantiser configuration.  All fields are 32- or 64-bit for a stable ABI. */
typedef struct nvfp4_quant_cfg {
  int32_t block;      /* nvfp4_block                                          */
  int32_t rounding;   /* nvfp4_rounding                                       */
  int32_t rht;        /* 1: 16-point random Hadamard transform along K        */
  int32_t sf_layout;  /* nvfp4_sf_layout of the block scales written          */
  int32_t transpose;  /* 1: quantise x^T, i.e. blocks run down the rows of x  */
  int32_t reserved;   /* must be 0                                            */
  uint64_t rht_seed;  /* sigma_j = -1 iff bit j of Philox(key=rht_seed, ctr=0) word 0 */
  uint64_t sr_seed;   /* Philox key for stochastic rounding                   */
  uint64_t sr_offset; /* Philox counter words 2..3 for stochastic rounding    */
} nvfp4_quant_cfg;

/* A quantised operand Q [rows, k], K-major (device pointers). */
typedef struct nvfp4_tensor {
  const void* codes;          /* rows * k / 2 bytes, row stride k / 2       */
  const void* sf;             /* block scales in `sf_layout`                */
  const float* tensor_scale;  /* one FP32 decode scale (device memory)      */
  int64_t rows;
  int64_t k;
  int32_t sf_layout;          /* nvfp4_sf_layout                            */
  int32_t reserved;           /* must be 0                                  */
} nvfp4_tensor;

const char* nvfp4_status_string(nvfp4_status status);
/* Library version as major * 10000 + minor * 100 + patch. */
int32_t nvfp4_version(void);

/* Sizes of the quantiser's outputs for Q [qr, qk]: codes qr * qk / 2 bytes;
 * block scales qr * qk / 16 bytes (ROWMAJOR) or the padded MMA size. */
size_t nvfp4_codes_bytes(int64_t qr, int64_t qk);
size_t nvfp4_sf_bytes(int64_t qr, int64_t qk, int32_t sf_layout);

/*
 * nvfp4_quantize: BF16 x [rows, cols] (row stride ldx elements, ldx >= cols,
 * device memory) -> Q = x (or x^T when cfg->transpose), qr x qk with
 * qr = rows, qk = cols (transposed: qr = cols, qk = rows).
 * Outputs: codes [qr, qk/2] bytes; sf in cfg->sf_layout; tensor_scale[0] = s.
 * Two passes over x: the tensor amax (after the transform, if any), then the
 * per-block encode.  Shape rules: qk % 16 == 0; 16x16 blocks also need
 * qr % 16 == 0; ldx % 8 == 0 and x 16-byte aligned; codes 8-byte aligned;
 * MMA-layout sf 16-byte aligned.
 * Non-finite input: the device status word is set to NVFP4_ERR_NONFINITE,
 * tensor_scale[0] is set to NaN and codes/sf are left unspecified.  A
 * bounded wait that ran out: NVFP4_ERR_TIMEOUT in the status word and, as
 * well, tensor_scale[0] = NaN (codes/sf unspecified).
 * Workspace: nvfp4_quantize_workspace_size bytes, device memory.
 * Sources: the encode steps listed at the top of this header.
 */
nvfp4_status nvfp4_quantize_workspace_size(int64_t rows, int64_t cols, const nvfp4_quant_cfg* cfg,
                                           size_t* bytes);
nvfp4_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                            const nvfp4_quant_cfg* cfg, void* codes, void* sf, float* tensor_scale,
                            void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_dual: two quantised outputs from one read of x, each with
 * its own configuration (orientation, block shape, rounding, transform,
 * seeds, scale layout) and its own tensor scale.  A training step needs X and
 * dY both along rows (fprop, dgrad) and along columns (wgrad), and W both ways
 * (fprop, dgrad); this call reads the BF16 tensor twice (amax pass, encode
 * pass) instead of four times.  Output A is bit-identical to nvfp4_quantize
 * with cfg_a, output B to nvfp4_quantize with cfg_b.
 * Arguments and rules as nvfp4_quantize for each output; the two outputs
 * must not overlap.  Workspace: nvfp4_quantize_workspace_size bytes (the same
 * size serves both outputs).  Source: the encode steps at the top of this
 * header; quantising every GEMM operand along its own K is the pages' NVFP4
 * training recipe ("NVIDIA acelera o pre-treinamento de LLM: NVFP4 no
 * Blackwell...", section "Como o treinamento mixed-precision funciona com
 * NVFP4").
 */
nvfp4_status nvfp4_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                 const nvfp4_quant_cfg* cfg_a, void* codes_a, void* sf_a, float* tensor_scale_a,
                                 const nvfp4_quant_cfg* cfg_b, void* codes_b, void* sf_b, float* tensor_scale_b,
                                 void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_given_amax: nvfp4_quantize under delayed scaling.  The
 * tensor scale is s = amax[0] / 2688 (1 if that is zero) for an amax the
 * caller supplies in device memory -- typically the one measured on the
 * previous step, for instance by nvfp4_gemm_quantize's amax_out -- so x is
 * read once (one pass) instead of twice.  Elements above amax[0] saturate:
 * their block scale stops at 448 and their codes at +-6, by the rounding
 * rules at the top of this header.  Every other step is nvfp4_quantize's, so
 * with amax[0] equal to the operand's own amax the outputs are identical.
 * amax[0] must be finite and >= 0: otherwise the device status word is set
 * to NVFP4_ERR_NONFINITE, tensor_scale[0] to NaN, and codes/sf are not
 * written.  x must be finite (it is not scanned first): a run holding inf or
 * NaN sets NVFP4_ERR_NONFINITE and its codes are unspecified.
 * Arguments, shape rules and workspace otherwise as nvfp4_quantize.
 * Source: custom scaling of NVFP4 values ("Por que cada porcento e
 * importante", JAX/MaxText page); the pages fix no scaling policy, and this
 * is the delayed-scaling reading with every other step unchanged.
 */
nvfp4_status nvfp4_quantize_given_amax(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                       const nvfp4_quant_cfg* cfg, const float* amax, void* codes, void* sf,
                                       float* tensor_scale, void* workspace, size_t workspace_bytes,
                                       nvfp4_stream_t stream);

/*
 * nvfp4_quantize_noalloc: nvfp4_quantize for callers that cannot allocate
 * device memory: a host framework or embedding runtime that owns every
 * device allocation and forbids others (so no workspace can be created for
 * this call), code running inside another allocator's callbacks, where
 * allocating would re-enter it, or latency-critical paths that must never
 * reach an allocator.  It takes no workspace: its status word and
 * partial-amax scratch live in one file-scope device array of the library
 * (16.6 KB, held on every GPU that loads the library until the process
 * exits).  The paper has no counterpart to this entry point; it belongs to
 * the library interface only.
 * Same arguments, shape rules and outputs as nvfp4_quantize, with a limit of
 * rows * cols <= 2^31 elements (NVFP4_ERR_UNSUPPORTED_SHAPE beyond).
 * Errors found on the device have one channel here, since the status word
 * sits in the library's array where the caller cannot read it: after the
 * call, tensor_scale[0] is NaN if the input held inf or NaN, or if one of
 * the kernel's bounded waits ran out (codes and sf are then unspecified);
 * otherwise it is the finite tensor scale.
 * The first call in a CUDA context looks up the array's device address
 * (cudaGetSymbolAddress) with that context current and caches it under the
 * context's unique ID; make that first call before any stream capture.  It
 * calls no cudaMalloc, cudaFree or allocating library routine.  All calls
 * share the one array, which keeps the last call's contents (the status
 * word is cleared at the start of every call, the partial maxima are
 * rewritten by every call before they are read): calls that overlap on the
 * GPU -- on different streams, or from host threads without ordering
 * between them -- race and must not be issued.
 */
nvfp4_status nvfp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                    const nvfp4_quant_cfg* cfg, void* codes, void* sf, float* tensor_scale,
                                    nvfp4_stream_t stream);

/*
 * nvfp4_dequantize: Q -> out [rows, k] with row stride ldo elements, as
 * e2m1(code) * e4m3(scale) * s computed in FP32 (exact product, one rounding
 * on the final multiply); BF16 output is that FP32 value rounded to nearest
 * even.  Any sf layout.  Needs no workspace.
 */
nvfp4_status nvfp4_dequantize(const nvfp4_tensor* q, int32_t out_dtype, void* out, int64_t ldo,
                              nvfp4_stream_t stream);

/*
 * nvfp4_gemm: D [M, N] = sA * sB * sum_k (eA * scaleA)(eB * scaleB), i.e.
 * D = A * B^T for A [M, K] and B [N, K] (M = A->rows, N = B->rows,
 * K = A->k = B->k), FP32 accumulation on the tensor cores (tcgen05
 * block-scaled MMA), FP32 epilogue multiply by sA * sB, then BF16 (round to
 * nearest even) or FP32 store, row stride ldd elements.
 * Shape rules: K % 32 == 0; both operands' scales in NVFP4_SF_MMA layout;
 * codes 16-byte aligned; ldd >= N.  M, N are arbitrary (ragged tiles are
 * handled).  Workspace: nvfp4_gemm_workspace_size bytes: the status word,
 * and FP32 scratch for partial sums where K is split:
 *   - outputs of one 128-row block with too few tiles to occupy the GPU (a
 *     decode-like M <= 128): split-K over the whole output;
 *   - M > 128 (CTA pairs on 256 x 256 tiles): when the tiles left after the
 *     last whole wave of CTA pairs would leave at least half the pairs idle
 *     and the split takes enough of K off that wave, each of those tiles is
 *     cut along K into pieces, one per pair.
 * K is split into whole groups of 1024; each piece's accumulator is stored
 * unscaled, and a reduction adds a tile's pieces in piece order, multiplies
 * by sA * sB and converts.  A workspace holding only the 256-byte header
 * (or too small for the split) runs the same GEMM unsplit; nvfp4_gemm_plan
 * reports the schedule.  The split depends on the current device (its SM
 * count and how many CTA pairs fit at once), so nvfp4_gemm_workspace_size
 * asks the device (setting the GEMM kernel up for it once, as the first
 * nvfp4_gemm would); with no usable CUDA device it returns the header size,
 * which is still valid and runs the GEMM unsplit.
 * Source: "Como o treinamento mixed-precision funciona com NVFP4" (NVFP4
 * operands, FP32 accumulators) on the JAX/MaxText page.
 */
nvfp4_status nvfp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);

/*
 * nvfp4_gemm_plan: how nvfp4_gemm schedules D [M, N] = A [M, K] * B [N, K]^T
 * on the current device given a workspace of workspace_bytes (the split
 * rules are those of nvfp4_gemm above; the schedule does not change the
 * result beyond the order of the FP32 sums).  Writes eight values to plan:
 *   plan[0] 1: CTA pairs on 256 x 256 tiles; 0: single CTAs on 128 x 256 tiles
 *   plan[1] CTAs launched (persistent, at most one per SM)
 *   plan[2] work units (tiles, split-K pieces or tail pieces)
 *   plan[3] split-K splits over the whole output (1: none; M <= 128 only)
 *   plan[4] k-blocks of 256 per split-K unit (all of K when unsplit)
 *   plan[5] tiles past the last whole wave cut along K (0: none; M > 128 only)
 *   plan[6] pieces per such tile
 *   plan[7] k-blocks of 256 per piece
 * M, N or K == 0 gives all zeros.  The caller owns plan (8 values).  Errors:
 * plan NULL or a negative size -> NVFP4_ERR_INVALID_ARG; K % 32 != 0 ->
 * NVFP4_ERR_UNSUPPORTED_SHAPE; no usable CUDA device -> NVFP4_ERR_CUDA.
 * Sets up the GEMM kernel for the device once (shared-memory opt-in,
 * occupancy query); launches nothing.  The pages have no counterpart: it
 * exposes a scheduling decision for tests and measurements.
 */
nvfp4_status nvfp4_gemm_plan(int64_t M, int64_t N, int64_t K, size_t workspace_bytes, int64_t* plan);
nvfp4_status nvfp4_gemm(const nvfp4_tensor* a, const nvfp4_tensor* b, int32_t out_dtype, void* d,
                        int64_t ldd, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* The quantised output of nvfp4_gemm_quantize (device pointers). */
typedef struct nvfp4_quant_out {
  const float* amax_in;  /* amax for the tensor scale s = amax_in[0] / 2688    */
  float* amax_out;       /* NULL, or receives max |D| over the BF16 outputs    */
  void* codes;           /* [M, N/2] bytes, 16-byte aligned                    */
  void* sf;              /* block scales in sf_layout (MMA: 16-byte aligned)   */
  float* tensor_scale;   /* receives s                                         */
  int32_t sf_layout;     /* nvfp4_sf_layout                                    */
  int32_t reserved;      /* must be 0                                          */
} nvfp4_quant_out;

/*
 * nvfp4_gemm_quantize: nvfp4_gemm with BF16 output whose epilogue also
 * quantises D for the next layer, straight from the accumulator: 1x16 blocks
 * along N (the next GEMM's K), round to nearest even, no transform, tensor
 * scale from q->amax_in (delayed scaling).  The codes, block scales and
 * tensor scale equal nvfp4_quantize_given_amax of the BF16 D with the same
 * amax, bit for bit, without D being read back from memory.
 * d may be NULL: D is then not stored (ldd is ignored).  q->amax_out, if not
 * NULL, is overwritten with max |D| of the BF16 values, the amax for the next
 * step's delayed scale.
 * Shape rules: as nvfp4_gemm, plus N % 32 == 0 and K > 0.  M == 0 or N == 0
 * launches nothing and writes nothing.
 * Errors: q->amax_in negative or non-finite -> NVFP4_ERR_NONFINITE in the
 * status word, tensor_scale NaN, codes/sf not written (D still is).  A D
 * value that overflows BF16 -> NVFP4_ERR_NONFINITE, codes of its block
 * unspecified.  Workspace: nvfp4_gemm_workspace_size bytes.
 * Source: the NVFP4 recipe quantises every GEMM input, activations included
 * ("Como o treinamento mixed-precision funciona com NVFP4", JAX/MaxText
 * page); the next layer's input is this GEMM's output, so the epilogue that
 * already holds it in registers encodes it.
 */
nvfp4_status nvfp4_gemm_quantize(const nvfp4_tensor* a, const nvfp4_tensor* b, void* d, int64_t ldd,
                                 const nvfp4_quant_out* q, void* workspace, size_t workspace_bytes,
                                 nvfp4_stream_t stream);

/*
 * nvfp4_lora_forward: the forward GEMM of a LoRA-SVD projection ("Full-Stack
 * FP4: Stable LLM Pretraining with Quantized Projections, Optimizers, and
 * Attention", section 2.1: the weight is W = W_res + beta L2 L1, the
 * residual W_res in NVFP4, the principal low-rank part L2 [dout, r],
 * L1 [r, din] in BF16; section 3 calls the reparametrisation fusable):
 *     Y [T, dout] = Q(X) Q(W_res)^T + beta U L2^T,   U = BF16(X L1^T) [T, r].
 * xq = Q(X) [T, din] and wq = Q(W_res) [dout, din] as for nvfp4_gemm (MMA
 * scale layout); x is the BF16 X [T, din] they came from (row stride ldx
 * elements, ldx % 8 == 0, 16-byte aligned); l1 BF16 [r, din] and l2 BF16
 * [dout, r], both dense row-major and 16-byte aligned; rank r with 8 <= r <=
 * 256 and r % 8 == 0; beta finite.  Output: y [T, dout] (row stride ldy >=
 * dout) in BF16 (round to nearest even) or FP32, and u [T, r] (dense BF16,
 * 16-byte aligned) receives U.
 * Two kernels: U = X L1^T on the tensor cores (BF16, FP32 accumulation,
 * rounded to BF16), written with the split hi + lo = (beta / (sX sW)) U into
 * the workspace; then the NVFP4 GEMM with the branch added into the same
 * FP32 accumulator as extra BF16 k-blocks (hi and lo against L2), scaled by
 * sX sW with the NVFP4 part in the epilogue.  The split keeps the branch to
 * about 2^-16 relative of beta U L2^T; U itself differs from the exactly
 * rounded BF16(X L1^T) only where the FP32 accumulation lands on the other
 * side of a BF16 rounding boundary.  Shape rules: din % 32 == 0, din > 0;
 * T and dout arbitrary.  |beta U / (sX sW)| must stay in BF16 range.
 * Workspace: nvfp4_lora_workspace_size(T, r) bytes (status word, then the
 * hi/lo buffer); errors as nvfp4_gemm.
 */
nvfp4_status nvfp4_lora_workspace_size(int64_t tokens, int64_t rank, size_t* bytes);
nvfp4_status nvfp4_lora_forward(const nvfp4_tensor* xq, const nvfp4_tensor* wq, const void* x, int64_t ldx,
                                const void* l1, const void* l2, int64_t rank, float beta, int32_t out_dtype, void* y,
                                int64_t ldy, void* u, void* workspace, size_t workspace_bytes,
                                nvfp4_stream_t stream);

/*
 * Newton-Schulz step of the Root optimizer with NVFP4 products ("Full-Stack
 * FP4: Stable LLM Pretraining with Quantized Projections, Optimizers, and
 * Attention", section 2.3, Q-Root: the NS matrix products run directly in
 * NVFP4, stabilised by shape-dependent coefficients a, b, c -- not printed on
 * the page, so they are arguments here -- and clipping of p99 outliers).
 *
 * nvfp4_abs_percentile_bf16: q[0] = the p-th percentile of |x| over the n
 * BF16 values of x (device, 16-byte aligned), nearest rank: the k-th
 * smallest magnitude with k = ceil(p / 100 * n) clamped to [1, n], exactly
 * (a radix selection on the magnitude bits); 0 < p <= 100; q[0] = 0 for
 * n == 0.  x must be finite: a NaN sets NVFP4_ERR_NONFINITE in the status
 * word and q is then unspecified.  Workspace:
 * nvfp4_abs_percentile_workspace_size bytes.
 * nvfp4_clip_bf16: out = x clipped to [-q[0], q[0]] elementwise (q[0] a BF16
 * magnitude, as the percentile gives; BF16 in and out, exact); out may be x.
 * nvfp4_axpby_bf16: out = BF16(RN(RN(a x) + RN(b y))) elementwise in FP32,
 * rounded to nearest even; out may alias x or y.  Needs no workspace.
 *
 * nvfp4_ns_step: one step on the BF16 iterate X [m, n] (row-major, dense;
 * m % 32 == 0, n % 32 == 0; put the shorter side first):
 *     A = X X^T,   B = b A + c A A^T,   X' = a X + B X,
 * where each product L R^T is the NVFP4 GEMM of its two operands, each first
 * clipped to its own p-th percentile magnitude and quantised along its K
 * (1x16 blocks, round to nearest even, no transform; Q(Xc) and Q(Xc^T) come
 * from one read), with BF16 results; B and X' are formed by
 * nvfp4_axpby_bf16 from the unclipped A and X.  x_out may be x.  Workspace:
 * nvfp4_ns_workspace_size(m, n) bytes (about 6 m^2 + 4 m n bytes plus the
 * quantised operands; it holds every intermediate).  Device-side errors as
 * the calls it is made of.  Reading of the page: the coefficients and the
 * percentile are the caller's; the step's form is the quintic
 * Newton-Schulz iteration, and clipping applies only to product operands.
 */
nvfp4_status nvfp4_abs_percentile_workspace_size(size_t* bytes);
nvfp4_status nvfp4_abs_percentile_bf16(const void* x, int64_t n, double p, float* q, void* workspace,
                                       size_t workspace_bytes, nvfp4_stream_t stream);
nvfp4_status nvfp4_clip_bf16(const void* x, int64_t n, const float* q, void* out, nvfp4_stream_t stream);
nvfp4_status nvfp4_axpby_bf16(const void* x, const void* y, int64_t n, float a, float b, void* out,
                              nvfp4_stream_t stream);
nvfp4_status nvfp4_ns_workspace_size(int64_t m, int64_t n, size_t* bytes);
nvfp4_status nvfp4_ns_step(const void* x, int64_t m, int64_t n, float a, float b, float c, double p, void* x_out,
                           void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * Quantised AdamW state codec ("Full-Stack FP4: Stable LLM Pretraining with
 * Quantized Projections, Optimizers, and Attention", section 2.2, Q-AdamW):
 * the optimizer's moments stored in NVFP4 (codes [rows, cols/2], row-major
 * block scales [rows, cols/16], one FP32 tensor scale), FP32 states in and out,
 * all row-major with row stride cols, 16-byte aligned.
 *
 * nvfp4_qadamw_m_encode: first moment.  Each run of 16 along a row is mixed by
 * the 16-point transform 1/4 H16 diag(sigma) (sigma from rht_seed as in
 * nvfp4_quant_cfg); s = amax / 2688 of the mixed tensor; per run the block
 * scale maps the run's maximum to 6 or to 4, whichever gives the smaller
 * round-to-nearest squared error (6 on a tie), and the codes are rounded
 * stochastically (Philox4x32-10 from sr_seed / sr_offset, element index
 * row * cols + col, as nvfp4_quantize).  cols % 16 == 0.
 * nvfp4_qadamw_m_decode: m_hat = diag(sigma) 1/4 H16 (code * scale * s) per run.
 * nvfp4_qadamw_v_encode: second moment (v >= 0).  r = sqrt(v); per 16x16 tile
 * the mean of r (row sums added in row order, times 2^-8) is stored as BF16
 * in tile_mean [rows/16, cols/16]; the residual r - mean is mixed by the
 * transform and rounded to nearest (1x16 blocks, maximum to 6).  rows % 16 ==
 * 0 and cols % 16 == 0.  A negative or non-finite v sets NVFP4_ERR_NONFINITE
 * in the status word and tensor_scale NaN.
 * nvfp4_qadamw_v_decode: v_hat = (mean + diag(sigma) 1/4 H16 deq)^2.
 * The encoders need nvfp4_qadamw_workspace_size bytes of workspace (status
 * word and the amax); the decoders need none.
 * The pages fix neither the 4/6 decision rule nor the tile size; these are the
 * readings above.
 */
nvfp4_status nvfp4_qadamw_workspace_size(size_t* bytes);
nvfp4_status nvfp4_qadamw_m_encode(const float* m, int64_t rows, int64_t cols, uint64_t rht_seed, uint64_t sr_seed,
                                   uint64_t sr_offset, void* codes, void* sf, float* tensor_scale, void* workspace,
                                   size_t workspace_bytes, nvfp4_stream_t stream);
nvfp4_status nvfp4_qadamw_m_decode(const void* codes, const void* sf, const float* tensor_scale, int64_t rows,
                                   int64_t cols, uint64_t rht_seed, float* m_out, nvfp4_stream_t stream);
nvfp4_status nvfp4_qadamw_v_encode(const float* v, int64_t rows, int64_t cols, uint64_t rht_seed, void* codes,
                                   void* sf, float* tensor_scale, void* tile_mean, void* workspace,
                                   size_t workspace_bytes, nvfp4_stream_t stream);
nvfp4_status nvfp4_qadamw_v_decode(const void* codes, const void* sf, const float* tensor_scale,
                                   const void* tile_mean, int64_t rows, int64_t cols, uint64_t rht_seed,
                                   float* v_out, nvfp4_stream_t stream);

/*
 * The linear layer Y = X W^T with X [T, din], W [dout, din], Y [T, dout]
 * (all BF16, row-major, densely packed), and its two backward GEMMs:
 *   fprop:  Y  = Q(X) Q(W)^T           X: 1x16 along din, W: 16x16 along din
 *   dgrad:  dX = Q(dY) Q(W^T)^T        dY: 1x16 along dout, W^T: 16x16 along dout
 *   wgrad:  dW = Q(dY^T) Q(X^T)^T      dY^T, X^T: 1x16 along T, RHT + SR
 * Each wrapper quantises its two operands into its workspace, in the
 * orientation its GEMM needs, then runs nvfp4_gemm (with the rest of the
 * workspace as its partial-sum scratch: nvfp4_linear_workspace_size includes
 * what nvfp4_gemm_workspace_size adds for the GEMM's shape; a workspace
 * without that part runs the GEMM unsplit).  cfg_* may be NULL for
 * the defaults above (seeds: rht_seed NVFP4_DEFAULT_RHT_SEED for every
 * operand, sr_seed 5 for dY^T and 6 for X^T in wgrad, sr_offset 0); a given
 * cfg is used as is except that the wrapper sets `transpose` (by role) and
 * `sf_layout` (MMA).  In wgrad both operands must share rht_seed for the
 * transform to cancel in the product.
 * Shape rules: din % 32 == 0, dout % 32 == 0, T % 32 == 0 (wgrad) and
 * T % 16 == 0 otherwise.  Output dtype per out_dtype.
 * Source: NVFP4 on weights and activations in GEMMs ("Como o treinamento
 * mixed-precision funciona com NVFP4", JAX/MaxText page).
 */
#define NVFP4_DEFAULT_RHT_SEED 0x5EEDC0DE0F4ull
typedef enum { NVFP4_LINEAR_FPROP = 0, NVFP4_LINEAR_DGRAD = 1, NVFP4_LINEAR_WGRAD = 2 } nvfp4_linear_op;
nvfp4_status nvfp4_linear_workspace_size(int32_t op, int64_t tokens, int64_t din, int64_t dout,
                                         size_t* bytes);
nvfp4_status nvfp4_linear_fprop(const void* x, const void* w, int64_t tokens, int64_t din, int64_t dout,
                                const nvfp4_quant_cfg* cfg_x, const nvfp4_quant_cfg* cfg_w,
                                int32_t out_dtype, void* y, void* workspace, size_t workspace_bytes,
                                nvfp4_stream_t stream);
nvfp4_status nvfp4_linear_dgrad(const void* dy, const void* w, int64_t tokens, int64_t din, int64_t dout,
                                const nvfp4_quant_cfg* cfg_dy, const nvfp4_quant_cfg* cfg_w,
                                int32_t out_dtype, void* dx, void* workspace, size_t workspace_bytes,
                                nvfp4_stream_t stream);
nvfp4_status nvfp4_linear_wgrad(const void* dy, const void* x, int64_t tokens, int64_t din, int64_t dout,
                                const nvfp4_quant_cfg* cfg_dy, const nvfp4_quant_cfg* cfg_x,
                                int32_t out_dtype, void* dw, void* workspace, size_t workspace_bytes,
                                nvfp4_stream_t stream);

/*
 * Synchronises `stream`, reads the status word of `workspace` (any workspace
 * used by the calls above), clears it and returns it: NVFP4_OK,
 * NVFP4_ERR_TIMEOUT or NVFP4_ERR_NONFINITE (or NVFP4_ERR_CUDA if the stream
 * reports an error).
 */
nvfp4_status nvfp4_check_device_status(const void* workspace, nvfp4_stream_t stream);

/*
 * Failure-detection test hook.  With enable != 0, the next nvfp4_gemm
 * launch (including one made by a linear wrapper) leaves the first
 * shared-memory stage of CTA 0 unfilled: that CTA's bounded wait runs out
 * after about one second, it records NVFP4_ERR_TIMEOUT in the workspace
 * status word, drains its in-flight copies, frees its tensor memory and
 * exits; the rest of the grid completes and the CUDA context stays usable.
 * The output of that launch is unspecified.  One-shot: the flag clears
 * itself when the launch takes it.  Nothing faults, traps or hangs.
 */
void nvfp4_debug_gemm_skip_load(int32_t enable);

/*
 * Failure-detection test hook for the quantiser.  pass = 1 (the amax pass)
 * or 2 (the encode pass): the next quantiser launch made by any entry point
 * above leaves CTA 0's first tile of that pass unfilled, so its bounded wait
 * runs out after about one second.  The CTA records NVFP4_ERR_TIMEOUT in
 * the status word, lets its other copies in flight land, and leaves; the
 * tensor scale of every output becomes NaN (an amax-pass timeout leaves a
 * NaN-like partial maximum, so the encode pass writes NaN and encodes
 * nothing).  Codes and scales of that call are unspecified; the CUDA context
 * stays usable.  A pass the call does not run (the amax pass under a
 * supplied amax) is not affected.  One-shot; pass = 0 clears it.
 */
void nvfp4_debug_quantize_skip_load(int32_t pass);

/*
 * Measurement of the tensor-core instruction the GEMM is built on, issued in
 * isolation: one CTA per SM (kind 0, 2: a CTA pair per two SMs), one thread
 * issuing `iters` back-to-back MMAs on fixed shared-memory operands into one
 * TMEM accumulator, five timed launches after two untimed ones.  The pages
 * have no counterpart: it gives the rate the GEMM's tensor-pipe time is
 * compared with (the GEMM's roofline).
 *   kind 0: block-scaled E2M1 (E4M3 scales per 16), cta_group::2, 256x256x64
 *   kind 1: the same, cta_group::1, 128x256x64
 *   kind 2: BF16 -> FP32, cta_group::2, 256x256x16
 *   kind 3: the same, cta_group::1, 128x256x16
 * Writes *tflops (whole GPU, CUDA events) and *cycles_per_mma (mean
 * clock64 cycles per instruction in an issuing CTA, the final wait
 * included).  Synchronous; allocates and frees a few bytes of device
 * memory; uses the current device.  iters in [16, 2^20] and non-null
 * outputs, else NVFP4_ERR_INVALID_ARG; NVFP4_ERR_CUDA if a CUDA call fails;
 * NVFP4_ERR_TIMEOUT if the bounded wait ran out.
 */
nvfp4_status nvfp4_debug_mma_rate(int32_t kind, int32_t iters, double* tflops, double* cycles_per_mma);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_H */
