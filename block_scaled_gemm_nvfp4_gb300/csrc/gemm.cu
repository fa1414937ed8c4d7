// Block-scaled NVFP4 GEMM on sm_103a tensor cores (tcgen05, kind::mxf4nvf4).
//
//   D[m, n] = sA * sB * sum_k (eA[m,k] * scaleA[m,k/16]) * (eB[n,k] * scaleB[n,k/16])
//
// NVFP4 operands with FP32 accumulation ("NVIDIA acelera o pre-treinamento de
// LLM: NVFP4 no Blackwell...", section "Como o treinamento mixed-precision
// funciona com NVFP4"); both operands K-major (D = A * B^T).
//
// Persistent, warp-specialised kernel, one CTA per SM, two modes:
//   pair mode (M > 128): a cluster of two CTAs computes a 256 x 256 tile with
//     cta_group::2 MMAs.  Each CTA holds 128 rows of A and 128 rows of B per
//     code stage (32 KB, five stages); the leader CTA issues the MMAs, which
//     read both CTAs' shared memory and write each CTA's 128 x 256 FP32
//     accumulator in its own TMEM;
//   single mode (M <= 128): one CTA per 128 x 256 tile, cta_group::1, three
//     48 KB code stages.
// Codes and block scales travel in separate rings.  A scale stage holds four
// k-blocks (three 8 KB copies) and runs ahead of the code ring; the staging
// warps move each k-block's scales into the TMEM slot of its code stage as
// soon as the stage's previous MMAs are done and arrive on the stage's own
// barrier, so the scale copies and the staging are hidden behind earlier
// k-blocks.  The MMA issuer then has one barrier per k-block and commits once
// per k-block.  The tensor pipe holds almost no issued work beyond the MMA in
// flight, so every cycle the issuing thread spends between MMAs idles it: the
// issuer tests the next k-block's barrier without blocking, ahead of the
// current k-block's MMAs, and blocks only when that test failed, and every
// extra barrier hop on its path (a separate scale-ready barrier with the peer
// CTA's remote arrivals cost about a quarter of the throughput) shows up
// directly in the k-block period (measured on GB300 with traces and variants).
// Warp roles (15 warps):
//   warp 0     TMA producer for the packed E2M1 codes (tiled TMA, 128-byte
//              swizzle);
//   warp 1     TMEM allocation; in the leader (or single) CTA the MMA issuer;
//   warps 2-9  epilogue, two warps per TMEM lane quarter, each owning 128 of
//              the 256 columns: TMEM -> registers (tcgen05.ld, two loads per
//              wait), times sA * sB, BF16 (RNE) or FP32.  In BF16 mode the
//              accumulator is released before anything is stored, and D
//              leaves as 32 x 32 chunks staged in a 2 KB shared-memory buffer
//              per warp and written by TMA tensor stores; the quantising
//              variant also encodes D along N (1x16, RNE, supplied amax) and
//              stores its codes the same way;
//   warps 10-13 stage each k-block's block scales from the scale ring into a
//              TMEM slot with tcgen05.st (one warp per lane quarter), keeping
//              the scale traffic off the tensor pipe, where a tcgen05.cp per
//              64-wide K step and 128 rows serialises with the MMAs;
//   warp 14    bulk-copy producer for the block scales.
// LoRA-SVD projection ("Full-Stack FP4...", section 2.1, W = W_res +
// beta L2 L1): the branch beta U L2^T joins the same accumulator as extra
// k-blocks after the NVFP4 ones -- BF16 operands (U's scaled hi / lo parts
// and L2, 64 columns per k-block, the byte layout of a k-block of codes) in
// kind::f16 MMAs; the staging warps only take part in those stages'
// barriers, and the epilogue's alpha scaling covers both terms.
// Work units are handed out round-robin to the persistent CTAs (pairs).  When
// K is split -- over the whole output for one-row-block outputs with too few
// tiles (split-K), or for the tiles past the last whole wave of CTA pairs
// (tail split) -- a unit covers whole scale stages of one tile's K and stores
// its raw FP32 accumulator; partial_reduce_kernel, launched as this kernel's
// programmatic dependent, sums a tile's partials in K order.
// Every mbarrier wait is bounded; on a timeout the CTA records
// NVFP4_ERR_TIMEOUT in the status word, drains its in-flight copies and MMAs,
// frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "encode.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

namespace {

constexpr int BM = 128;                       // accumulator rows per CTA
constexpr int BN = 256;                       // accumulator columns
constexpr int BK = 256;                       // elements of K per stage
constexpr int kRowBytes = BK / 2;             // 128 bytes of packed codes per row per stage
constexpr int kABytes = BM * kRowBytes;       // 16 KB
constexpr int kSfAtomBytes = 512;             // 128 rows x 4 scales
constexpr int kSfaBytes = 4 * kSfAtomBytes;   // one row atom x 4 K atoms
constexpr int kThreads = 480;                 // 15 warps
constexpr int kEpiWarps = 8;
constexpr int kSfWarps = 4;
constexpr int kFirstSfWarp = 10;
constexpr int kSfProducerWarp = 14;
constexpr int kEpiCols = BN / 2;              // columns per epilogue warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;
constexpr uint32_t kSfaCol = 256;             // + slot * 16 + kk * 4
constexpr int kMaxStages = 5;                 // code stages = TMEM scale slots (one k-block each)
constexpr uint32_t kSfbCol = kSfaCol + 16 * kMaxStages;  // + stage * 32 + kk * 8 + row_atom * 4
constexpr int kSfGroup = 4;                   // k-blocks per scale stage
constexpr int kSfaGroupBytes = kSfGroup * kSfaBytes;     // 8 KB: 16 K atoms of one A row block
constexpr int kSfStageBytes = 3 * kSfaGroupBytes;        // A + two B row blocks: 24 KB
// Operand panels a raster group keeps in L2.  Measured on GB300 (DRAM bytes
// per launch of the MLP-up GEMMs and 16384^3): 32 MB groups leave fprop and
// wgrad at their algorithmic operand reads and cut dgrad's from 427 to 321 MB;
// 64 and 96 MB groups are evicted before their reuse and re-read far more.
constexpr double kGroupL2Bytes = 32.0e6;
// A tail split pays for its partial stores and the separate reduction (a few
// microseconds) only when it takes this many k-blocks (~0.3 us each on a
// 256 x 256 tile) off the last wave.
constexpr int kTailMinGainKb = 24;
// BF16 output leaves through shared memory: each epilogue warp stages a
// 32-row x 32-column chunk (64-byte rows, 64-byte swizzle) and a TMA store
// writes it, so global writes are whole 64-byte row segments instead of one
// 16-byte piece per row per store instruction.
constexpr int kEpiChunkCols = 32;
constexpr int kEpiStgBytes = 32 * kEpiChunkCols * 2;       // 2 KB per warp
constexpr int kEpiStgTotal = kEpiWarps * kEpiStgBytes;     // 16 KB
static_assert(kSfbCol + 32 * kMaxStages <= kTmemCols, "TMEM budget");

// Per-mode layout.  Codes and block scales travel in separate rings: a code
// stage holds one k-block of A and B codes (and owns one TMEM scale slot); a
// scale stage holds four k-blocks of scales, so the small scale copies are
// issued ahead of the codes and their latency stays off the MMA's path.
//   PAIR: B rows per CTA 128, five 32 KB code stages;
//   single: B rows 256, three 48 KB code stages;
// both with two 24 KB scale stages.
template <bool PAIR>
struct Layout {
  static constexpr int kBRows = PAIR ? BN / 2 : BN;
  static constexpr int kBBytes = kBRows * kRowBytes;
  static constexpr int kStages = PAIR ? 5 : 3;
  static constexpr int kSfStages = 2;
  static_assert(kStages <= kMaxStages, "one TMEM scale slot per code stage");
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kSfRing = kStages * kStageBytes;  // offset of the scale ring
  static constexpr int kEpiStg = kSfRing + kSfStages * kSfStageBytes;  // epilogue staging
  static constexpr int kCtl = kEpiStg + kEpiStgTotal;                  // barriers
  static constexpr int kSmemBytes = kCtl + 1024 /*barriers*/ + 1024 /*alignment*/;
  // Instruction descriptor for kind::mxf4nvf4: dense, A and B E2M1 (format 1),
  // both K-major, N >> 3 at bit 17, UE4M3 scales (bit 23 = 0), M >> 4 at bit
  // 24 (M = 256 across the pair in PAIR mode), scale-factor ids 0.
  static constexpr uint32_t kIdesc =
      (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((PAIR ? 2 * BM : BM) >> 4) << 24);
  // Instruction descriptor for the LoRA branch's kind::f16 MMAs: F32
  // accumulator (bit 4), A and B BF16 (format 1 at bits 7 and 10), both
  // K-major, the same N and M.  A 64-wide BF16 k-block is 128 bytes per row,
  // the layout of a k-block of E2M1 codes, so it uses the same stages.
  static constexpr uint32_t kIdescF16 =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((PAIR ? 2 * BM : BM) >> 4) << 24);
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for 128B swizzle");
  static_assert(kSfStageBytes % 16 == 0, "bulk copies need 16-byte alignment");
  static_assert(kEpiStg % 1024 == 0, "staging buffers keep the 64-byte swizzle's 512-byte alignment");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct GParams {
  int64_t M, N, K;
  int num_kb;        // K stages
  int tiles_m, tiles_n, num_tiles;
  int tiles_mp;      // row-block pairs (pair mode)
  int num_units;     // tiles, or tile pairs in pair mode
  int64_t sf_katoms; // 64-wide K atoms per row block in the scale layout
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  const float* a_scale;
  const float* b_scale;
  void* d;
  int64_t ldd;
  int vec_store;
  int tma_store;        // BF16 D leaves by TMA stores (tensor map tmap_d)
  int group_n;          // raster groups column blocks instead of row blocks
  int group;            // row or column blocks per raster group
  int skip_first_load;  // test hook: CTA 0 never loads its first stage
  uint32_t* status;
  // quantising epilogue (QUANT kernels): D's NVFP4 codes and block scales
  // along N under the tensor scale amax_in / 2688
  uint8_t* q_codes;
  uint8_t* q_sf;
  float* q_tensor_scale;
  const float* q_amax_in;
  uint32_t* q_amax_out;  // max |D| as FP32 bits, or null
  int q_sf_mma;
  int64_t q_kb_count;    // N / 16
  int64_t q_katoms;      // 64-wide N atoms of the MMA scale layout
  // LoRA-SVD branch: lora_kb BF16 k-blocks after the NVFP4 ones (A from
  // tmap_lu, B from tmap_l2; kind::f16 MMAs into the same accumulator);
  // 0 for a plain GEMM
  int lora_kb;
  // split-K (single mode, FP32 kernel): unit = tile * split_k + s covers
  // k-blocks [s * kb_per_split, (s + 1) * kb_per_split) and stores its raw
  // FP32 accumulator (alpha not applied) as a whole column-major 128 x 256
  // block at part + (s * num_tiles + tile) * BM * BN (element (r, c) at
  // c * BM + r), so a warp's 32 lanes write 128 consecutive bytes per
  // column; 1 = no split
  int split_k;
  int kb_per_split;
  // Tail split (pair mode): the tail_tiles tiles past the last whole wave of
  // CTA pairs (tiles tail_first ..) are cut along K into pieces of tail_kb
  // k-blocks; piece s of tail tile i is unit tail_first + s * tail_tiles + i
  // and stores its raw accumulator like a split-K partial, one block per CTA
  // of the pair at part + ((s * tail_tiles + i) * 2 + rank) * BM * BN, and
  // a reduction launched after the kernel sums them into D.
  // tail_tiles == 0: none.
  int tail_first;
  int tail_tiles;
  int tail_kb;
  float* part;  // FP32 partial blocks of split-K units and tail pieces
};

// Tile index, k-block range and partial block of a work unit; `part` says
// whether the unit stores a raw partial accumulator instead of D.  SPLIT:
// the kernel may split K (not with LoRA k-blocks or the quantising epilogue).
template <bool SPLIT>
__device__ __forceinline__ void unit_split(const GParams& p, int unit, int& tile, int& kb_lo, int& kb_hi,
                                           int64_t& d_off, bool& part) {
  if (SPLIT && p.split_k > 1) {
    tile = unit / p.split_k;
    const int s = unit - tile * p.split_k;
    kb_lo = s * p.kb_per_split;
    kb_hi = min(p.num_kb, kb_lo + p.kb_per_split);
    d_off = (static_cast<int64_t>(s) * p.num_tiles + tile) * (BM * BN);
    part = true;
  } else if (SPLIT && p.tail_tiles > 0 && unit >= p.tail_first) {
    const int idx = unit - p.tail_first;
    const int s = idx / p.tail_tiles;
    const int i = idx - s * p.tail_tiles;
    tile = p.tail_first + i;
    kb_lo = s * p.tail_kb;
    kb_hi = min(p.num_kb, kb_lo + p.tail_kb);
    d_off = (static_cast<int64_t>(s) * p.tail_tiles + i) * (2 * BM * BN);
    part = true;
  } else {
    tile = unit;
    kb_lo = 0;
    kb_hi = p.num_kb;
    d_off = 0;
    part = false;
  }
}

template <int STAGES, int SF_STAGES>
struct __align__(8) SmemCtl {
  uint64_t full[STAGES];          // k-block ready: codes landed and scales in TMEM (pair mode:
                                  // both CTAs', leader's copy)
  uint64_t empty[STAGES];         // code stage and its TMEM scale slot no longer read by MMAs
  uint64_t sf_full[SF_STAGES];    // this CTA's block scales landed in the scale ring
  uint64_t sf_empty[SF_STAGES];   // scale ring stage copied into TMEM
  uint64_t acc_full;
  uint64_t acc_empty;             // accumulator drained (pair mode: both CTAs', leader's copy)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Tile raster: tiles are taken in groups of p.group row blocks (sweeping every
// column block) or p.group column blocks (sweeping every row block), whichever
// re-reads fewer operand bytes from DRAM; inside a group the fast index runs
// over the group so concurrent CTAs share operand panels in L2.
__device__ __forceinline__ void tile_coords(const GParams& p, int tile, int tiles_m, int& m_blk, int& n_blk) {
  const int slow_tiles = p.group_n ? tiles_m : p.tiles_n;
  const int fast_tiles = p.group_n ? p.tiles_n : tiles_m;
  const int per_group = p.group * slow_tiles;
  const int group = tile / per_group;
  const int first = group * p.group;
  const int g = min(fast_tiles - first, p.group);
  const int local = tile - group * per_group;
  const int fast = first + local % g;
  const int slow = local / g;
  m_blk = p.group_n ? slow : fast;
  n_blk = p.group_n ? fast : slow;
}

// A work unit is one tile, or in pair mode one 256-row tile computed by the
// two CTAs of a cluster (row blocks 2i and 2i+1); `rank` picks this CTA's half.
template <bool PAIR>
__device__ __forceinline__ void unit_coords(const GParams& p, int unit, uint32_t rank, int& m_blk, int& n_blk) {
  if (!PAIR) {
    tile_coords(p, unit, p.tiles_m, m_blk, n_blk);
  } else {
    int mp;
    tile_coords(p, unit, p.tiles_mp, mp, n_blk);
    m_blk = 2 * mp + static_cast<int>(rank);
  }
}

__device__ __forceinline__ int kk_count_for(const GParams& p, int kb) {
  const int64_t rem = p.K - static_cast<int64_t>(kb) * BK;
  return static_cast<int>(min(static_cast<int64_t>(4), (rem + 63) / 64));
}

__device__ __forceinline__ void fail(int* abort, const GParams& p, uint32_t where) {
  ptx::set_status(p.status, kDevTimeout | (where << 8));
  *reinterpret_cast<volatile int*>(abort) = 1;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int lane) {
  uint32_t ok = 1;
  if (lane == 0) ok = ptx::mbar_wait(bar, parity, abort_flag) ? 1u : 0u;
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// Arrive on the leader CTA's copy of a barrier: a local arrive in the
// leader (or single) CTA, a relaxed remote arrive from the follower.  Callers
// have completed the TMEM accesses being signalled (tcgen05.wait::st or
// wait::ld, then tcgen05.fence::before_thread_sync).
template <bool PAIR>
__device__ __forceinline__ void arrive_leader(uint64_t* bar, uint32_t rank) {
  if (PAIR && rank != 0)
    ptx::mbar_arrive_cluster_relaxed(ptx::mapa_shared(ptx::smem_u32(bar), 0));
  else
    ptx::mbar_arrive(bar);
}

// Quantising epilogue for this thread's 128 BF16 outputs of row `row`
// (columns col0 .. col0 + 127, two per word of `packed`): eight runs of 16
// along N, each with its E4M3 block scale and E2M1 codes (round to nearest
// even) under the tensor scale s_dec -- the quantiser's steps applied to the
// BF16 values D holds, so the result equals quantising the stored D.  Rows
// past M and blocks past N are not encoded; in the tensor-core scale layout
// their scale bytes are written as the layout's zero padding.
struct QuantHalf {
  uint32_t codes[kEpiCols / 8];  // 16 bytes of codes per 32 columns
  uint32_t sfw[2];               // block kb0 + j in byte (j & 3) of word j >> 2
  uint32_t amax_bits;            // largest |value| of the valid runs (FP32 bits, NaN propagated)
};

// Encode chunk c (columns col0 + 32 c .. + 31: two runs).  N % 32 == 0, so
// the chunk is either wholly inside N or wholly outside.
__device__ __forceinline__ void quantize_chunk(const GParams& p, const uint32_t (&packed)[kEpiCols / 2], int c,
                                               bool row_ok, int64_t kb0, float s_dec, float rs, QuantHalf& qh) {
  const bool in = row_ok && kb0 + 2 * c < p.q_kb_count;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = 2 * c + h;
    float v[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w = packed[r * 8 + j];
      v[2 * j] = __uint_as_float(w << 16);
      v[2 * j + 1] = __uint_as_float(w & 0xFFFF0000u);
    }
    const uint32_t m = run_absmax_nan(v);
    const uint32_t sfb = in ? block_scale_byte_rcp(m, s_dec, rs) : 0u;
    if (in) qh.amax_bits = max(qh.amax_bits, m);
    qh.codes[2 * r] = 0u;
    qh.codes[2 * r + 1] = 0u;
    if (sfb != 0) {
      divide_run<false>(v, __fmul_rn(ptx::e4m3_to_float(sfb), s_dec), v);  // elementwise, in place
      qh.codes[2 * r] = ptx::cvt_e2m1x8(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
      qh.codes[2 * r + 1] = ptx::cvt_e2m1x8(v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]);
    }
    qh.sfw[r >> 2] |= sfb << (8 * (r & 3));
  }
}

// Write the encoded half: the warp's codes (32 rows x 64 bytes) leave like D,
// staged in its buffer (64-byte swizzle) once the previous store has read it,
// then one TMA store; the block scales go straight to their layout.
__device__ __forceinline__ void store_quantised(const GParams& p, const CUtensorMap* tmap_q, uint8_t* stg,
                                                const QuantHalf& qh, int64_t row, int64_t row0, int64_t col0, int q,
                                                int lane) {
  const int64_t kb0 = col0 / 16;
  const bool box = row0 < p.M && col0 < p.N;   // warp-uniform: some of the box is inside D
  if (lane == 0) ptx::bulk_wait_group_read0();  // a D store may still be reading the buffer
  __syncwarp();
  uint8_t* srow = stg + lane * 64;
#pragma unroll
  for (int c = 0; c < kEpiCols / 32; ++c)
    *reinterpret_cast<uint4*>(srow + ((c ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(qh.codes[4 * c], qh.codes[4 * c + 1], qh.codes[4 * c + 2], qh.codes[4 * c + 3]);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (box && lane == 0) {
    ptx::tma_store_2d(tmap_q, stg, static_cast<int32_t>(col0 / 2), static_cast<int32_t>(row0));
    ptx::bulk_commit_group();
  }
  if (p.q_sf_mma) {
    // atoms of 128 rows x 4 blocks: this thread's four blocks of an atom are
    // the 4-byte word at lane * 16 + q * 4 (row % 32 = lane, row % 128 / 32 = q).
    // In pair mode with an odd number of row blocks the follower's last tile
    // lies wholly past M: its row atom does not exist and is not written.
    const bool atom_row_ok = row / BM < p.tiles_m;
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int64_t katom = kb0 / 4 + a;
      if (atom_row_ok && katom < p.q_katoms)
        *reinterpret_cast<uint32_t*>(p.q_sf + ((row / BM) * p.q_katoms + katom) * 512 + lane * 16 + q * 4) =
            qh.sfw[a];
    }
  } else if (row < p.M) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (kb0 + j < p.q_kb_count)
        p.q_sf[row * p.q_kb_count + kb0 + j] = static_cast<uint8_t>(qh.sfw[j >> 2] >> (8 * (j & 3)));
  }
}

// Epilogue for one 128 x 128 half of a tile: TMEM -> registers -> global.
// The warp's lane quarter q gives its 32 rows.  Releases the accumulator (one
// arrival per warp on the leader's acc_empty) as soon as it has been read.
template <bool OUT_F32, bool PAIR, bool QUANT>
__device__ __forceinline__ void epilogue_half(const GParams& p, const CUtensorMap* tmap_d, const CUtensorMap* tmap_q,
                                              uint8_t* stg,
                                              uint64_t* acc_empty, uint32_t tmem, int m_blk,
                                              int n_blk, int q, int half, int lane, float alpha, uint32_t rank,
                                              float s_dec, float rs, uint32_t& amax_bits, int64_t d_off,
                                              bool part) {
  const int64_t row = static_cast<int64_t>(m_blk) * BM + q * 32 + lane;
  const int64_t col0 = static_cast<int64_t>(n_blk) * BN + half * kEpiCols;
  const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + kAccCol + half * kEpiCols;
  if (!QUANT && part) {
    // split-K partial or tail piece: raw accumulator, column-major block
    // (coalesced across the warp's lanes, which hold consecutive rows);
    // padding rows and columns of ragged tiles hold the zeros their
    // out-of-range operands gave
    float* blk = p.part + d_off + (PAIR ? static_cast<int64_t>(rank) * (BM * BN) : 0) +
                 static_cast<int64_t>(half * kEpiCols) * BM + q * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < kEpiCols / 32; ++c) {
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
      ptx::tmem_ld_wait();
      ptx::tmem_ld_regs_ready(r);
#pragma unroll
      for (int j = 0; j < 32; ++j) blk[(c * 32 + j) * BM] = __uint_as_float(r[j]);
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive_leader<PAIR>(acc_empty, rank);
  } else if (!OUT_F32) {
    uint32_t packed[kEpiCols / 2];
    QuantHalf qh;  // used by the quantising epilogue only
    qh.sfw[0] = qh.sfw[1] = 0u;
    qh.amax_bits = 0u;
    // Four 32-column loads in two waits: chunks 2 and 3 are requested while
    // chunks 0 and 1 are converted, which shortens the accumulator hand-off.
    static_assert(kEpiCols == 128, "four 32-column chunks");
    uint32_t r0[32], r1[32];
    ptx::tmem_ld_32x32b_x32(taddr, r0);
    ptx::tmem_ld_32x32b_x32(taddr + 32, r1);
    ptx::tmem_ld_wait();
    ptx::tmem_ld_regs_ready(r0);
    ptx::tmem_ld_regs_ready(r1);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      packed[j] = pack_bf16(__fmul_rn(alpha, __uint_as_float(r0[2 * j])), __fmul_rn(alpha, __uint_as_float(r0[2 * j + 1])));
    ptx::tmem_ld_32x32b_x32(taddr + 64, r0);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      packed[16 + j] =
          pack_bf16(__fmul_rn(alpha, __uint_as_float(r1[2 * j])), __fmul_rn(alpha, __uint_as_float(r1[2 * j + 1])));
    ptx::tmem_ld_32x32b_x32(taddr + 96, r1);
    ptx::tmem_ld_wait();
    ptx::tmem_ld_regs_ready(r0);
    ptx::tmem_ld_regs_ready(r1);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      packed[32 + j] =
          pack_bf16(__fmul_rn(alpha, __uint_as_float(r0[2 * j])), __fmul_rn(alpha, __uint_as_float(r0[2 * j + 1])));
      packed[48 + j] =
          pack_bf16(__fmul_rn(alpha, __uint_as_float(r1[2 * j])), __fmul_rn(alpha, __uint_as_float(r1[2 * j + 1])));
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive_leader<PAIR>(acc_empty, rank);
    if (p.tma_store) {
      // Chunk c (columns col0 + 32 c ..): lane l writes its row's 64 bytes
      // into row l of the warp's buffer, 16-byte piece j at slot
      // j ^ ((l >> 1) & 3) (the 64-byte swizzle the tensor map names, which
      // also keeps the writes free of bank conflicts); one lane then stores
      // the box.  Boxes wholly past M or N are skipped; ragged boxes are
      // clipped by the TMA unit.  The buffer is reused once the previous
      // store has finished reading it.
      const int64_t row0 = static_cast<int64_t>(m_blk) * BM + q * 32;
#pragma unroll
      for (int c = 0; c < kEpiCols / kEpiChunkCols; ++c) {
        const int64_t col = col0 + c * kEpiChunkCols;
        if (row0 >= p.M || col >= p.N) {  // warp-uniform
          if constexpr (QUANT) quantize_chunk(p, packed, c, row < p.M, col0 / 16, s_dec, rs, qh);
          continue;
        }
        if (lane == 0) ptx::bulk_wait_group_read0();
        __syncwarp();
        uint8_t* rowp = stg + lane * 64;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(rowp + ((j ^ ((lane >> 1) & 3)) << 4)) =
              make_uint4(packed[c * 16 + 4 * j], packed[c * 16 + 4 * j + 1], packed[c * 16 + 4 * j + 2],
                         packed[c * 16 + 4 * j + 3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(tmap_d, stg, static_cast<int32_t>(col), static_cast<int32_t>(row0));
          ptx::bulk_commit_group();
        }
        // encode this chunk while the store reads the buffer
        if constexpr (QUANT) quantize_chunk(p, packed, c, row < p.M, col0 / 16, s_dec, rs, qh);
      }
    } else if (row < p.M && p.d != nullptr) {  // D is optional for the quantising epilogue
      __nv_bfloat16* drow = static_cast<__nv_bfloat16*>(p.d) + row * p.ldd;
#pragma unroll
      for (int c8 = 0; c8 < kEpiCols / 8; ++c8) {
        const int64_t col = col0 + c8 * 8;
        if (p.vec_store && col + 8 <= p.N) {
          __stcs(reinterpret_cast<uint4*>(drow + col),
                 make_uint4(packed[c8 * 4], packed[c8 * 4 + 1], packed[c8 * 4 + 2], packed[c8 * 4 + 3]));
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (col + j < p.N) {
              const uint32_t w = packed[c8 * 4 + j / 2];
              const uint16_t h = static_cast<uint16_t>((j & 1) ? (w >> 16) : (w & 0xFFFFu));
              reinterpret_cast<uint16_t*>(drow)[col + j] = h;
            }
          }
        }
      }
    }
    if constexpr (QUANT) {
      if (!p.tma_store) {
#pragma unroll
        for (int c = 0; c < kEpiCols / kEpiChunkCols; ++c) quantize_chunk(p, packed, c, row < p.M, col0 / 16, s_dec, rs, qh);
      }
      store_quantised(p, tmap_q, stg, qh, row, static_cast<int64_t>(m_blk) * BM + q * 32, col0, q, lane);
      amax_bits = max(amax_bits, qh.amax_bits);
    }
  } else {
    float* drow = static_cast<float*>(p.d) + d_off + row * p.ldd;
#pragma unroll 1
    for (int c = 0; c < kEpiCols / 32; ++c) {
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
      ptx::tmem_ld_wait();
      ptx::tmem_ld_regs_ready(r);
      if (row < p.M) {
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const int64_t col = col0 + c * 32 + j4 * 4;
          const float4 v = make_float4(__fmul_rn(alpha, __uint_as_float(r[4 * j4])),
                                       __fmul_rn(alpha, __uint_as_float(r[4 * j4 + 1])),
                                       __fmul_rn(alpha, __uint_as_float(r[4 * j4 + 2])),
                                       __fmul_rn(alpha, __uint_as_float(r[4 * j4 + 3])));
          if (p.vec_store && col + 4 <= p.N) {
            __stcs(reinterpret_cast<float4*>(drow + col), v);
          } else {
            if (col < p.N) drow[col] = v.x;
            if (col + 1 < p.N) drow[col + 1] = v.y;
            if (col + 2 < p.N) drow[col + 2] = v.z;
            if (col + 3 < p.N) drow[col + 3] = v.w;
          }
        }
      }
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive_leader<PAIR>(acc_empty, rank);
  }
}

// Scale staging for one k-block.  Layout the block-scaled MMA reads
// (scale_vec::4X): for a 128-row operand block and one K = 64 step, TMEM lane
// 32 q + l, column base + j holds the four scales of row l + 32 j; every lane
// quarter q holds the whole block, because the quarter that computes output
// rows 32 q .. 32 q + 31 reads the B scales of all N rows from its own lanes
// (and the A scales of its own rows from column base + q).  That is one
// 16-byte row of a 512-byte scale atom per lane, so each staging warp (lane
// quarter q) copies atom row `lane` into its own lanes.  Columns of TMEM
// slot t: A at kSfaCol + 16 t + 4 kk, B row block rb at kSfbCol + 32 t + 8 kk
// + 4 rb (a 256-row B operand is read as columns base .. base + 7).
__device__ __forceinline__ void stage_scales(const uint8_t* sfa, const uint8_t* sfb, int sfb_rb_stride,
                                             uint32_t tmem, int slot, int q, int lane) {
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
  uint32_t va[16];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint4 v = *reinterpret_cast<const uint4*>(sfa + kk * kSfAtomBytes + lane * 16);
    va[4 * kk] = v.x;
    va[4 * kk + 1] = v.y;
    va[4 * kk + 2] = v.z;
    va[4 * kk + 3] = v.w;
  }
  ptx::tmem_st_32x32b_x16(lane_base + kSfaCol + slot * 16, va);
  uint32_t vb[32];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
    for (int rb = 0; rb < 2; ++rb) {
      const uint4 v = *reinterpret_cast<const uint4*>(sfb + rb * sfb_rb_stride + kk * kSfAtomBytes + lane * 16);
      vb[8 * kk + 4 * rb] = v.x;
      vb[8 * kk + 4 * rb + 1] = v.y;
      vb[8 * kk + 4 * rb + 2] = v.z;
      vb[8 * kk + 4 * rb + 3] = v.w;
    }
  }
  ptx::tmem_st_32x32b_x32(lane_base + kSfbCol + slot * 32, vb);
}

// LORA: the kernel also runs the LoRA-SVD branch's BF16 k-blocks.  It is a
// template parameter because even an untaken per-k-block branch on the MMA
// issuer's path cost the plain GEMM about 13 % (measured on GB300).
template <bool OUT_F32, bool PAIR, bool QUANT, bool LORA>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ CUtensorMap tmap_q,
                const __grid_constant__ CUtensorMap tmap_lu, const __grid_constant__ CUtensorMap tmap_l2,
                const GParams p) {
  using L = Layout<PAIR>;
  constexpr int S = L::kStages;
  constexpr int SS = L::kSfStages;
  const int lora_kb = LORA ? p.lora_kb : 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sf_ring = smem + L::kSfRing;
  SmemCtl<S, SS>* ctl = reinterpret_cast<SmemCtl<S, SS>*>(smem + L::kCtl);
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ustep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // the code producer's arrival (with the tiles' byte count) and one
      // arrival per scale-staging warp of each CTA
      ptx::mbar_init(&ctl->full[s], 1 + (PAIR ? 2 : 1) * kSfWarps);
      ptx::mbar_init(&ctl->empty[s], 1);
    }
    for (int s = 0; s < SS; ++s) {
      ptx::mbar_init(&ctl->sf_full[s], 1);
      ptx::mbar_init(&ctl->sf_empty[s], kSfWarps);
    }
    ptx::mbar_init(&ctl->acc_full, 1);
    ptx::mbar_init(&ctl->acc_empty, PAIR ? 2 * kEpiWarps : kEpiWarps);
    ptx::mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (threadIdx.x == 0 && (p.split_k > 1 || p.tail_tiles > 0)) {
    // the partial-sum reduction may be scheduled now: its CTAs take SMs as
    // this grid's CTAs leave and wait for the whole grid before reading
    ptx::griddep_launch_dependents();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&tmap_a);
    ptx::prefetch_tensormap(&tmap_b);
    if (p.tma_store) ptx::prefetch_tensormap(&tmap_d);
    if (QUANT) ptx::prefetch_tensormap(&tmap_q);
    if (LORA) {
      ptx::prefetch_tensormap(&tmap_lu);
      ptx::prefetch_tensormap(&tmap_l2);
    }
  }
  if (warp == 1) {
    // pair mode: one warp of each CTA of the pair allocates collectively
    if (PAIR) {
      ptx::tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&ctl->tmem_base, kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // the peer's barriers must be initialised before anything reaches them
  if (PAIR) ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ code producer
    if (lane == 0) {
      uint32_t issued_mask = 0, issued_parity = 0;
      const uint64_t l2_keep = ptx::policy_evict_last();
      const uint32_t full_leader0 = PAIR ? ptx::mapa_shared(ptx::smem_u32(&ctl->full[0]), 0) : 0u;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int unit = unit0; unit < p.num_units && ok; unit += ustep) {
        int m_blk, n_blk, tile, kb_lo, kb_hi;
        int64_t d_off;
        bool part;
        unit_split<!QUANT && !LORA>(p, unit, tile, kb_lo, kb_hi, d_off, part);
        unit_coords<PAIR>(p, tile, rank, m_blk, n_blk);
        for (int kb = kb_lo; kb < kb_hi + lora_kb; ++kb) {
          if (!ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, abort_flag)) {
            fail(&ctl->abort, p, 1);
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * L::kStageBytes;
          if (p.skip_first_load && blockIdx.x == 0 && unit == unit0 && kb == kb_lo) {
            // Failure-detection test hook: this stage is never filled, so the
            // bounded waits on it run out and the CTA reports a timeout.
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (LORA && kb >= kb_hi) {
            // LoRA branch k-block j: A = hi (j even) or lo (j odd) of the
            // branch's 64-column chunk j / 2, B = that chunk of L2; the same
            // box sizes and swizzle as a k-block of codes
            const int j = kb - kb_hi;
            if (PAIR) {
              const uint32_t bar = full_leader0 + static_cast<uint32_t>(stage * sizeof(uint64_t));
              if (leader) ptx::mbar_arrive_expect_tx(&ctl->full[stage], 2u * (kABytes + L::kBBytes));
              ptx::tma_load_2d_pair(st, &tmap_lu, bar, j * 64, m_blk * BM);
              ptx::tma_load_2d_pair(st + kABytes, &tmap_l2, bar, (j >> 1) * 64,
                                    n_blk * BN + static_cast<int>(rank) * L::kBRows);
            } else {
              ptx::mbar_arrive_expect_tx(&ctl->full[stage], static_cast<uint32_t>(kABytes + L::kBBytes));
              ptx::tma_load_2d(st, &tmap_lu, &ctl->full[stage], j * 64, m_blk * BM);
              ptx::tma_load_2d(st + kABytes, &tmap_l2, &ctl->full[stage], (j >> 1) * 64, n_blk * BN);
            }
          } else if (PAIR) {
            // both CTAs' code tiles complete on the leader's barrier
            const uint32_t bar = full_leader0 + static_cast<uint32_t>(stage * sizeof(uint64_t));
            if (leader) ptx::mbar_arrive_expect_tx(&ctl->full[stage], 2u * (kABytes + L::kBBytes));
            ptx::tma_load_2d_pair_hint(st, &tmap_a, bar, kb * kRowBytes, m_blk * BM, l2_keep);
            ptx::tma_load_2d_pair_hint(st + kABytes, &tmap_b, bar, kb * kRowBytes,
                                       n_blk * BN + static_cast<int>(rank) * L::kBRows, l2_keep);
          } else {
            ptx::mbar_arrive_expect_tx(&ctl->full[stage], static_cast<uint32_t>(kABytes + L::kBBytes));
            ptx::tma_load_2d_hint(st, &tmap_a, &ctl->full[stage], kb * kRowBytes, m_blk * BM, l2_keep);
            ptx::tma_load_2d_hint(st + kABytes, &tmap_b, &ctl->full[stage], kb * kRowBytes, n_blk * BN, l2_keep);
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every copy this thread issued must have landed before exit.
      // (Pair mode: the code tiles complete on the leader's barrier, which
      // the leader drains; the final cluster barrier keeps the follower
      // alive until then.  The stage-free barrier of each CTA also takes the
      // leader's last multicast commits.)
      for (int s = 0; s < S; ++s) {
        if (issued_mask & (1u << s)) {
          volatile int never = 0;
          const uint32_t par = (issued_parity >> s) & 1u;
          if ((!PAIR || leader) && !ptx::mbar_wait(&ctl->full[s], par, &never)) fail(&ctl->abort, p, 2);
          if (PAIR && ok && !ptx::mbar_wait(&ctl->empty[s], par, abort_flag)) fail(&ctl->abort, p, 2);
        }
      }
    }
  } else if (warp == kSfProducerWarp) {
    // ----------------------------------------------------- scale producer
    if (lane == 0) {
      uint32_t issued_mask = 0, issued_parity = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int unit = unit0; unit < p.num_units && ok; unit += ustep) {
        int m_blk, n_blk, tile, kb_lo, kb_hi;
        int64_t d_off;
        bool part;
        unit_split<!QUANT && !LORA>(p, unit, tile, kb_lo, kb_hi, d_off, part);
        unit_coords<PAIR>(p, tile, rank, m_blk, n_blk);
        const int64_t n_rows_left = p.N - static_cast<int64_t>(n_blk) * BN;
        const int nb_atoms = static_cast<int>(min(static_cast<int64_t>(2), (n_rows_left + 127) / 128));
        // (a row block past the end -- the odd last half of a pair -- has no
        // scales to load; its rows are never stored)
        const bool a_valid = m_blk < p.tiles_m;
        for (int kb0 = kb_lo; kb0 < kb_hi; kb0 += kSfGroup) {
          if (!ptx::mbar_wait(&ctl->sf_empty[stage], phase ^ 1u, abort_flag)) {
            fail(&ctl->abort, p, 9);
            ok = false;
            break;
          }
          // the 64-wide K atoms of k-blocks kb0 .. kb0 + 3, contiguous per row block
          const int64_t atom0 = static_cast<int64_t>(kb0) * 4;
          const uint32_t bytes =
              static_cast<uint32_t>(min(static_cast<int64_t>(4 * kSfGroup), p.sf_katoms - atom0) * kSfAtomBytes);
          uint8_t* st = sf_ring + stage * kSfStageBytes;
          ptx::mbar_arrive_expect_tx(&ctl->sf_full[stage], bytes * ((a_valid ? 1 : 0) + nb_atoms));
          if (a_valid)
            ptx::bulk_load(st, p.a_sf + (static_cast<int64_t>(m_blk) * p.sf_katoms + atom0) * kSfAtomBytes, bytes,
                           &ctl->sf_full[stage]);
          for (int rb = 0; rb < nb_atoms; ++rb)
            ptx::bulk_load(st + (1 + rb) * kSfaGroupBytes,
                           p.b_sf + (static_cast<int64_t>(n_blk * 2 + rb) * p.sf_katoms + atom0) * kSfAtomBytes, bytes,
                           &ctl->sf_full[stage]);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == SS) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < SS; ++s) {
        if (issued_mask & (1u << s)) {
          volatile int never = 0;
          if (!ptx::mbar_wait(&ctl->sf_full[s], (issued_parity >> s) & 1u, &never)) fail(&ctl->abort, p, 10);
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, issued = false;
      // The tensor pipe holds little issued work, so each cycle this thread
      // spends outside MMA issue between k-blocks idles it; a blocking wait
      // on an already-completed barrier costs ~150-200 cycles.  Each full
      // k-block therefore tests the next stage's barrier without blocking,
      // ahead of its own MMAs, and the next k-block waits only if that test
      // failed.
      bool next_ready = false;
      // descriptors of stage 0; other stages and K steps are plain offsets
      // of the 14-bit start-address field (shared-memory addresses < 256 KB)
      const uint64_t a_desc0 = ptx::smem_desc(ptx::smem_u32(smem), 16, 1024, ptx::kSwizzle128B);
      const uint64_t b_desc0 = ptx::smem_desc(ptx::smem_u32(smem + kABytes), 16, 1024, ptx::kSwizzle128B);
      for (int unit = unit0; unit < p.num_units && ok; unit += ustep) {
        int tile, kb_lo, kb_hi;
        int64_t d_off;
        bool part;
        unit_split<!QUANT && !LORA>(p, unit, tile, kb_lo, kb_hi, d_off, part);
        if (!ptx::mbar_wait(&ctl->acc_empty, acc_phase ^ 1u, abort_flag)) {
          fail(&ctl->abort, p, 3);
          break;
        }
        ptx::tc_fence_after();
        for (int kb = kb_lo; kb < kb_hi + lora_kb; ++kb) {
          // One wait per k-block: the stage's barrier completes when its code
          // tiles have landed (pair mode: both CTAs') and every staging warp
          // (both CTAs') has put its scales into the stage's TMEM slot.
          // CTA-scope waits suffice: the peer's arrivals follow completed
          // TMEM writes, and the code tiles are TMA (async-proxy) writes read
          // by the tensor core.
          if (!next_ready && !ptx::mbar_wait(&ctl->full[stage], phase, abort_flag)) {
            fail(&ctl->abort, p, 4);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t st_off = static_cast<uint32_t>(stage * L::kStageBytes);
          const uint64_t adesc0 = a_desc0 + (st_off >> 4);
          const uint64_t bdesc0 = b_desc0 + (st_off >> 4);
          if (LORA && kb >= kb_hi) {
            // LoRA branch: four BF16 MMAs of K = 16 (32 bytes along the
            // swizzled 128-byte rows), added to the NVFP4 accumulation
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              if (PAIR)
                ptx::tc_mma_f16_pair(tmem + kAccCol, adesc0 + 2 * kk, bdesc0 + 2 * kk, L::kIdescF16, 1u);
              else
                ptx::tc_mma_f16(tmem + kAccCol, adesc0 + 2 * kk, bdesc0 + 2 * kk, L::kIdescF16, 1u);
            }
            if (PAIR)
              ptx::tc_commit_pair_multicast(&ctl->empty[stage], static_cast<uint16_t>(0x3));
            else
              ptx::tc_commit(&ctl->empty[stage]);
            next_ready = false;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          const int kk_n = kk_count_for(p, kb);
          const uint32_t sfa_t0 = tmem + kSfaCol + stage * 16;
          const uint32_t sfb_t0 = tmem + kSfbCol + stage * 32;
          if (kk_n == 4) {
            // the next stage's barrier: the phase the next k-block waits for
            const int nstage = stage + 1 == S ? 0 : stage + 1;
            const uint32_t nphase = stage + 1 == S ? phase ^ 1u : phase;
            // +32 bytes along K inside the swizzled 128-byte rows per MMA
            next_ready = ptx::tc_mma_nvf4_x2_probe<PAIR>(
                             tmem + kAccCol, adesc0, bdesc0, adesc0 + 2, bdesc0 + 2, L::kIdesc, sfa_t0, sfb_t0,
                             sfa_t0 + 4, sfb_t0 + 8, kb != kb_lo ? 1u : 0u, ptx::smem_u32(&ctl->full[nstage]),
                             nphase) != 0u;
#pragma unroll
            for (int kk = 2; kk < 4; ++kk) {
              if (PAIR)
                ptx::tc_mma_nvf4_pair(tmem + kAccCol, adesc0 + 2 * kk, bdesc0 + 2 * kk, L::kIdesc, sfa_t0 + kk * 4,
                                      sfb_t0 + kk * 8, 1u);
              else
                ptx::tc_mma_nvf4(tmem + kAccCol, adesc0 + 2 * kk, bdesc0 + 2 * kk, L::kIdesc, sfa_t0 + kk * 4,
                                 sfb_t0 + kk * 8, 1u);
            }
          } else {
            // the ragged last k-block of K
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              if (kk < kk_n) {
                const uint64_t adesc = adesc0 + 2 * kk, bdesc = bdesc0 + 2 * kk;
                const uint32_t acc = (kb != kb_lo || kk != 0) ? 1u : 0u;
                if (PAIR)
                  ptx::tc_mma_nvf4_pair(tmem + kAccCol, adesc, bdesc, L::kIdesc, sfa_t0 + kk * 4, sfb_t0 + kk * 8,
                                        acc);
                else
                  ptx::tc_mma_nvf4(tmem + kAccCol, adesc, bdesc, L::kIdesc, sfa_t0 + kk * 4, sfb_t0 + kk * 8, acc);
              }
            }
            next_ready = false;
          }
          // one commit frees the code stage and its TMEM scale slot
          if (PAIR)
            ptx::tc_commit_pair_multicast(&ctl->empty[stage], static_cast<uint16_t>(0x3));
          else
            ptx::tc_commit(&ctl->empty[stage]);
          issued = true;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR)
          ptx::tc_commit_pair_multicast(&ctl->acc_full, static_cast<uint16_t>(0x3));
        else
          ptx::tc_commit(&ctl->acc_full);
        acc_phase ^= 1u;
      }
      if (issued) {
        // Wait for every MMA issued above before TMEM is freed.
        if (PAIR)
          ptx::tc_commit_pair(&ctl->drain);
        else
          ptx::tc_commit(&ctl->drain);
        volatile int never = 0;
        if (!ptx::mbar_wait(&ctl->drain, 0, &never)) fail(&ctl->abort, p, 5);
      }
    }
  } else if (warp >= kFirstSfWarp) {
    // ------------------------------------------------------ scale staging
    // One k-block per iteration: wait until the scales are in the ring (one
    // wait per scale stage) and the MMAs that last read this TMEM slot (one
    // ring lap earlier, in the same code stage) have completed, copy this
    // warp's lane quarter, arrive.  (Staging two k-blocks per pass, with
    // one shared wait::st, measured about 1.5 % slower once the MMA issuer
    // probed its barriers ahead.)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int sstage = 0, slot = 0;
    uint32_t sphase = 0, tphase = 0;
    bool ok = true;
    const uint32_t full_leader0 = PAIR ? ptx::mapa_shared(ptx::smem_u32(&ctl->full[0]), 0) : 0u;
    auto arrive_full = [&](int s_) {
      // the stage's ready barrier lives in the leader (or single) CTA
      if (PAIR && !leader)
        ptx::mbar_arrive_cluster_relaxed(full_leader0 + static_cast<uint32_t>(s_ * sizeof(uint64_t)));
      else
        ptx::mbar_arrive(&ctl->full[s_]);
    };
    for (int unit = unit0; unit < p.num_units && ok; unit += ustep) {
      int tile, kb_lo, kb_hi;
      int64_t d_off;
      bool part;
      unit_split<!QUANT && !LORA>(p, unit, tile, kb_lo, kb_hi, d_off, part);
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        const int j = kb % kSfGroup;
        if ((j == 0 && !warp_wait(&ctl->sf_full[sstage], sphase, abort_flag, lane)) ||
            !warp_wait(&ctl->empty[slot], tphase ^ 1u, abort_flag, lane)) {
          if (lane == 0) fail(&ctl->abort, p, 7);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint8_t* st = sf_ring + sstage * kSfStageBytes;
        stage_scales(st + j * kSfaBytes, st + kSfaGroupBytes + j * kSfaBytes, kSfaGroupBytes, tmem, slot, q, lane);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        const bool group_done = j + 1 == kSfGroup || kb + 1 == kb_hi;
        if (lane == 0) {
          if (group_done) ptx::mbar_arrive(&ctl->sf_empty[sstage]);
          arrive_full(slot);
        }
        if (group_done && ++sstage == SS) {
          sstage = 0;
          sphase ^= 1u;
        }
        if (++slot == S) {
          slot = 0;
          tphase ^= 1u;
        }
      }
      // LoRA branch k-blocks need no scales: the staging warps only take
      // part in their stages' barriers, once the stage is free again.
      for (int j = 0; LORA && j < lora_kb && ok; ++j) {
        if (!warp_wait(&ctl->empty[slot], tphase ^ 1u, abort_flag, lane)) {
          if (lane == 0) fail(&ctl->abort, p, 8);
          ok = false;
          break;
        }
        if (lane == 0) arrive_full(slot);
        if (++slot == S) {
          slot = 0;
          tphase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;    // which 128 columns of the tile it stores
    uint8_t* stg = smem + L::kEpiStg + (warp - 2) * kEpiStgBytes;  // this warp's output staging
    // (partial accumulators are stored unscaled; their reduction applies alpha)
    const float alpha = __fmul_rn(*p.a_scale, *p.b_scale);
    // quantising epilogue: tensor scale s = amax_in / 2688 (1 if that is
    // zero); a negative or non-finite amax_in is reported and nothing is
    // encoded
    float s_dec = 1.0f;
    float rs = 0.0f;  // RN(1/s_dec) where the residual-corrected block-scale division applies
    bool q_live = true;
    uint32_t amax_bits = 0;
    if (QUANT) {
      const float a_in = *p.q_amax_in;
      const bool first = blockIdx.x == 0 && threadIdx.x == 64;  // warp 2, lane 0
      if (!(a_in >= 0.0f) || isinf(a_in)) {
        q_live = false;
        if (first) {
          ptx::set_status(p.status, kDevNonFinite);
          *p.q_tensor_scale = __uint_as_float(0x7FC00000u);
        }
      } else {
        s_dec = __fdiv_rn(fabsf(a_in), 2688.0f);
        if (s_dec == 0.0f) s_dec = 1.0f;
        rs = (s_dec >= 0x1p-70f && s_dec < 0x1p126f) ? __frcp_rn(s_dec) : 0.0f;
        if (first) *p.q_tensor_scale = s_dec;
      }
    }
    uint32_t acc_phase = 0;
    for (int unit = unit0; unit < p.num_units; unit += ustep) {
      int m_blk, n_blk, tile, kb_lo, kb_hi;
      int64_t d_off;
      bool part;
      unit_split<!QUANT && !LORA>(p, unit, tile, kb_lo, kb_hi, d_off, part);
      unit_coords<PAIR>(p, tile, rank, m_blk, n_blk);
      if (!warp_wait(&ctl->acc_full, acc_phase, abort_flag, lane)) {
        if (lane == 0) fail(&ctl->abort, p, 6);
        break;
      }
      ptx::tc_fence_after();
      if constexpr (QUANT) {
        if (q_live)
          epilogue_half<OUT_F32, PAIR, true>(p, &tmap_d, &tmap_q, stg, &ctl->acc_empty, tmem, m_blk, n_blk, q, half, lane, alpha, rank,
                                             s_dec, rs, amax_bits, d_off, part);
        else
          epilogue_half<OUT_F32, PAIR, false>(p, &tmap_d, &tmap_q, stg, &ctl->acc_empty, tmem, m_blk, n_blk, q, half, lane, alpha, rank,
                                              s_dec, rs, amax_bits, d_off, part);
      } else {
        epilogue_half<OUT_F32, PAIR, false>(p, &tmap_d, &tmap_q, stg, &ctl->acc_empty, tmem, m_blk, n_blk, q, half, lane, alpha, rank,
                                            s_dec, rs, amax_bits, d_off, part);
      }
      acc_phase ^= 1u;
    }
    // the staging buffer and the kernel's lifetime must outlast the stores
    if ((p.tma_store || QUANT) && lane == 0) ptx::bulk_wait_group0();
    if (QUANT && q_live) {
      // the lanes of a warp leave the loop above together (warp_wait is
      // warp-uniform), so the shuffles below see the whole warp
      if (amax_bits >= 0x7F800000u) ptx::set_status(p.status, kDevNonFinite);  // D overflowed
      if (p.q_amax_out) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xFFFFFFFFu, amax_bits, o));
        if (lane == 0) atomicMax(p.q_amax_out, amax_bits);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  // neither CTA of a pair leaves (or frees TMEM) while the other may still
  // write into it
  if (PAIR) ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (PAIR)
      ptx::tmem_dealloc_pair(tmem, kTmemCols);
    else
      ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Tensor map over packed codes [rows, K/2] bytes, box = 128 bytes x box_rows,
// 128-byte swizzle, out-of-range elements read as zero.
bool make_codes_map(CUtensorMap* map, const uint8_t* codes, int64_t rows, int64_t K, uint32_t box_rows) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kRowBytes), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map over BF16 D [M, N] (row stride ldd elements) for the staged
// output: box 32 columns x 32 rows, 64-byte swizzle.
bool make_d_map(CUtensorMap* map, void* d, int64_t M, int64_t N, int64_t ldd) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldd) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kEpiChunkCols), 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map over the quantised output's codes [M, N/2] bytes: box 64 bytes
// x 32 rows, 64-byte swizzle.
bool make_qcodes_map(CUtensorMap* map, uint8_t* codes, int64_t M, int64_t N) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N / 2), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N / 2)};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, codes, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Reduction of partial accumulators: D[m, n] = RN(alpha * (((P0 + P1) + P2)
// + ...)) over the `split` partial blocks of each output block, in that
// fixed order, alpha = RN(sA * sB); BF16 (round to nearest even) or FP32
// output, row stride ldd.  Every 128 x 256 output block h (blockIdx.z) has
// one column-major partial block per split s at part + (s * blocks + h) *
// BM * BN (element (r, c) at c * BM + r).  Split-K (single mode, M <= 128):
// block h is column block h.  Tail pieces (pair mode): block h is the half
// h & 1 of tail tile h >> 1, placed by the tile raster.  A CTA of 256
// threads sums a 32-row x 32-column piece: each thread reads four rows of
// one column from every split with 16-byte loads (eight splits in flight),
// and the sums leave along rows through a shared-memory transpose.
template <bool OUT_F32>
__global__ void __launch_bounds__(256) partial_reduce_kernel(const float* __restrict__ part, int split, int blocks,
                                                             const GParams p, void* d, int64_t ldd) {
  __shared__ float sm[32][33];  // [column][row]
  const int h = static_cast<int>(blockIdx.z);
  int m_blk = 0, n_blk = h;
  if (p.tail_tiles > 0) {
    int mp;
    tile_coords(p, p.tail_first + (h >> 1), p.tiles_mp, mp, n_blk);
    m_blk = 2 * mp + (h & 1);
  }
  const int r0 = static_cast<int>(blockIdx.y) * 32, c0 = static_cast<int>(blockIdx.x) * 32;
  const int64_t row0 = static_cast<int64_t>(m_blk) * BM + r0, col0 = static_cast<int64_t>(n_blk) * BN + c0;
  if (row0 >= p.M || col0 >= p.N) return;  // block-uniform
  ptx::griddep_wait();  // the GEMM grid's partials (launched as its programmatic dependent)
  const float alpha = __fmul_rn(*p.a_scale, *p.b_scale);
  const int t = static_cast<int>(threadIdx.x);
  const int cc = t >> 3, rq = (t & 7) * 4;  // column cc, rows rq .. rq + 3 of the piece
  const int64_t split_stride = static_cast<int64_t>(blocks) * BM * BN;
  const float* src = part + static_cast<int64_t>(h) * BM * BN + static_cast<int64_t>(c0 + cc) * BM + r0 + rq;
  float4 acc = __ldcg(reinterpret_cast<const float4*>(src));
  for (int s0 = 1; s0 < split; s0 += 8) {
    float4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (s0 + k < split) v[k] = __ldcg(reinterpret_cast<const float4*>(src + (s0 + k) * split_stride));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (s0 + k < split) {
        acc.x = __fadd_rn(acc.x, v[k].x);
        acc.y = __fadd_rn(acc.y, v[k].y);
        acc.z = __fadd_rn(acc.z, v[k].z);
        acc.w = __fadd_rn(acc.w, v[k].w);
      }
    }
  }
  sm[cc][rq] = acc.x;
  sm[cc][rq + 1] = acc.y;
  sm[cc][rq + 2] = acc.z;
  sm[cc][rq + 3] = acc.w;
  __syncthreads();
  // thread t writes row t / 8, columns (t % 8) * 4 .. + 3
  const int r = t >> 3, cs = (t & 7) * 4;
  const int64_t m = row0 + r, n = col0 + cs;
  if (m >= p.M || n >= p.N) return;
  float v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = __fmul_rn(alpha, sm[cs + k][r]);
  const bool whole = n + 4 <= p.N && p.vec_store;
  if (OUT_F32) {
    float* drow = static_cast<float*>(d) + m * ldd;
    if (whole) {
      *reinterpret_cast<float4*>(drow + n) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (n + k < p.N) drow[n + k] = v[k];
    }
  } else {
    __nv_bfloat16* drow = static_cast<__nv_bfloat16*>(d) + m * ldd;
    if (whole) {
      *reinterpret_cast<uint2*>(drow + n) = make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]));
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (n + k < p.N) drow[n + k] = __float2bfloat16_rn(v[k]);
    }
  }
}

// Launched right after the GEMM kernel as its programmatic dependent, so its
// launch overlaps the GEMM's last wave.
template <bool OUT_F32>
cudaError_t launch_partial_reduce(const GParams& p, int split, int blocks, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(BN / 32, BM / 32, static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, partial_reduce_kernel<OUT_F32>, static_cast<const float*>(p.part), split, blocks,
                            p, p.d, p.ldd);
}

// Tail split of a pair-mode GEMM run by `clusters` CTA pairs: when the tiles
// past the last whole wave would leave at least half the pairs idle, each is
// cut along K into `split` pieces of `kb` k-blocks (whole scale stages), one
// piece per pair, so the last wave ends after a fraction of a tile's
// k-blocks; the pieces' partial accumulators are then summed by a separate
// reduction.  Tiles [first, first + tiles) are the split ones.
struct TailPlan {
  int first, tiles, split, kb;
};

bool plan_tail(int units, int clusters, int num_kb, TailPlan* t) {
  if (units <= 0 || clusters < 2) return false;
  const int rem = units % clusters;
  if (rem == 0 || num_kb < 2 * kSfGroup) return false;
  int s = std::min(clusters / rem, num_kb / kSfGroup);
  if (s < 2) return false;
  int per = (num_kb + s - 1) / s;
  per = (per + kSfGroup - 1) / kSfGroup * kSfGroup;
  s = (num_kb + per - 1) / per;
  if (s < 2 || num_kb - per < kTailMinGainKb) return false;
  t->first = units - rem;
  t->tiles = rem;
  t->split = s;
  t->kb = per;
  return true;
}

// FP32 partial blocks of a tail split: two 128 x 256 blocks (one per CTA of
// the pair) per piece.
size_t tail_bytes(const TailPlan& t) {
  return static_cast<size_t>(t.tiles) * t.split * 2 * BM * BN * sizeof(float);
}

cudaLaunchAttribute pair_cluster_attr() {
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  return attr;
}

// One-time setup per device of one kernel instantiation (the shared-memory
// opt-in and, in pair mode, the number of co-resident clusters), safe against
// concurrent first calls; *max_clusters = co-resident CTA pairs (1 in single
// mode).
template <bool OUT_F32, bool PAIR, bool QUANT, bool LORA>
cudaError_t kernel_setup(int* max_clusters) {
  using L = Layout<PAIR>;
  auto kernel = gemm_kernel<OUT_F32, PAIR, QUANT, LORA>;
  static std::mutex setup_mutex;
  static int clusters_of_device[64] = {0};  // 0: not set up yet
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(setup_mutex);
  if (clusters_of_device[dev] == 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return e;
    int mc = 1;
    if (PAIR) {
      cudaLaunchConfig_t cfg{};
      cudaLaunchAttribute attr = pair_cluster_attr();
      cfg.gridDim = dim3(2 * device_sm_count());
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = L::kSmemBytes;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&mc, kernel, &cfg);
      if (e != cudaSuccess) return e;
      if (mc < 1) return cudaErrorInvalidConfiguration;
    }
    clusters_of_device[dev] = mc;
  }
  *max_clusters = clusters_of_device[dev];
  return cudaSuccess;
}

template <bool OUT_F32, bool PAIR, bool QUANT, bool LORA = false>
cudaError_t launch_typed(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md,
                         const CUtensorMap& mq, const CUtensorMap& mlu, const CUtensorMap& ml2, GParams p,
                         cudaStream_t stream, size_t part_bytes = 0) {
  using L = Layout<PAIR>;
  auto kernel = gemm_kernel<OUT_F32, PAIR, QUANT, LORA>;
  int max_clusters = 0;
  cudaError_t e = kernel_setup<OUT_F32, PAIR, QUANT, LORA>(&max_clusters);
  if (e != cudaSuccess) return e;
  if (!PAIR) {
    p.num_units = p.num_tiles * (p.split_k > 1 ? p.split_k : 1);
    const int grid = std::min(p.num_units, device_sm_count());
    kernel<<<grid, kThreads, L::kSmemBytes, stream>>>(ma, mb, md, mq, mlu, ml2, p);
    return cudaGetLastError();
  }
  p.num_units = p.tiles_mp * p.tiles_n;
  p.tail_tiles = 0;
  TailPlan tp;
  if (!QUANT && !LORA && p.part != nullptr && plan_tail(p.num_units, max_clusters, p.num_kb, &tp) &&
      tail_bytes(tp) <= part_bytes) {
    p.tail_first = tp.first;
    p.tail_tiles = tp.tiles;
    p.tail_kb = tp.kb;
    p.num_units = tp.first + tp.tiles * tp.split;
  }
  const int clusters = std::min(p.num_units, max_clusters);
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr = pair_cluster_attr();
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, ma, mb, md, mq, mlu, ml2, p);
  if (e != cudaSuccess || p.tail_tiles == 0) return e;
  // the tail tiles' D: their pieces summed in piece order
  return launch_partial_reduce<OUT_F32>(p, tp.split, 2 * tp.tiles, stream);
}

}  // namespace

int gemm_split_k(int64_t M, int64_t N, int64_t K, int* kb_per_split) {
  // Split-K only where the output has too few tiles to occupy the GPU: one
  // row block (single mode), fewer than half as many tiles as SMs, and at
  // least two scale stages (8 k-blocks) of K.  Splits are whole scale stages
  // (multiples of kSfGroup k-blocks).
  if (M <= 0 || N <= 0 || M > BM || K <= 0) return 1;
  const int num_kb = static_cast<int>((K + BK - 1) / BK);
  const int64_t tiles = (N + BN - 1) / BN;
  const int sms = device_sm_count();
  if (tiles * 2 > sms || num_kb < 2 * kSfGroup) return 1;
  int s = static_cast<int>(std::min<int64_t>(sms / tiles, num_kb / kSfGroup));
  if (s < 2) return 1;
  int per = (num_kb + s - 1) / s;
  per = (per + kSfGroup - 1) / kSfGroup * kSfGroup;
  s = (num_kb + per - 1) / per;
  if (s < 2) return 1;
  if (kb_per_split) *kb_per_split = per;
  return s;
}

size_t gemm_split_k_bytes(int64_t M, int64_t N, int split_k) {
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  return static_cast<size_t>(split_k) * tiles * BM * BN * sizeof(float);
}

cudaError_t gemm_plan(int64_t M, int64_t N, int64_t K, size_t partial_bytes, GemmPlan* g) {
  *g = GemmPlan{};
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  const int num_kb = static_cast<int>((K + BK - 1) / BK);
  const int tiles_m = static_cast<int>((M + BM - 1) / BM), tiles_n = static_cast<int>((N + BN - 1) / BN);
  g->split_k = 1;
  g->kb_per_unit = num_kb;
  if (tiles_m < 2) {
    int per = 0;
    const int sk = gemm_split_k(M, N, K, &per);
    g->pair = 0;
    g->units = tiles_m * tiles_n;
    g->partial_bytes_needed = sk > 1 ? gemm_split_k_bytes(M, N, sk) : 0;
    if (sk > 1 && partial_bytes >= g->partial_bytes_needed) {
      g->split_k = sk;
      g->kb_per_unit = per;
      g->units *= sk;
    }
    g->ctas = std::min(g->units, device_sm_count());
    return cudaSuccess;
  }
  int max_clusters = 0;
  const cudaError_t e = kernel_setup<false, true, false, false>(&max_clusters);
  if (e != cudaSuccess) return e;
  g->pair = 1;
  g->units = ((tiles_m + 1) / 2) * tiles_n;
  TailPlan tp;
  if (plan_tail(g->units, max_clusters, num_kb, &tp)) {
    g->partial_bytes_needed = tail_bytes(tp);
    if (partial_bytes >= g->partial_bytes_needed) {
      g->tail_tiles = tp.tiles;
      g->tail_split = tp.split;
      g->tail_kb = tp.kb;
      g->units = tp.first + tp.tiles * tp.split;
    }
  }
  g->ctas = 2 * std::min(g->units, max_clusters);
  return cudaSuccess;
}

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  if (a.K == 0) {
    const size_t esz = a.out_f32 ? 4 : 2;
    return cudaMemset2DAsync(a.d, a.ldd * esz, 0, a.N * esz, a.M, stream);
  }
  // Pair mode needs at least two row blocks.
  const bool pair = (a.M + BM - 1) / BM >= 2;
  CUtensorMap ma, mb;
  if (!make_codes_map(&ma, a.a_codes, a.M, a.K, BM) ||
      !make_codes_map(&mb, a.b_codes, a.N, a.K, pair ? Layout<true>::kBRows : Layout<false>::kBRows))
    return cudaErrorInvalidValue;
  GParams p{};
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.num_kb = static_cast<int>((a.K + BK - 1) / BK);
  p.tiles_m = static_cast<int>((a.M + BM - 1) / BM);
  p.tiles_n = static_cast<int>((a.N + BN - 1) / BN);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.tiles_mp = (p.tiles_m + 1) / 2;
  p.sf_katoms = (a.K / 16 + 3) / 4;
  p.a_sf = a.a_sf;
  p.b_sf = a.b_sf;
  p.a_scale = a.a_scale;
  p.b_scale = a.b_scale;
  p.d = a.d;
  p.ldd = a.ldd;
  p.status = a.status;
  p.skip_first_load = a.skip_first_load;
  {
    // DRAM operand traffic of the two rasters: a group holds as many panels
    // of its own operand (all of K for one row or column block) as fit in
    // kGroupL2Bytes, which stay in L2 while the other operand is swept past
    // them; the swept operand is read once per group.
    const double a_bytes = static_cast<double>(a.M) * a.K * 0.5625, b_bytes = static_cast<double>(a.N) * a.K * 0.5625;
    const int m_units = pair ? p.tiles_mp : p.tiles_m;
    const int g_m = static_cast<int>(std::max(1.0, std::min<double>(m_units, kGroupL2Bytes * m_units / a_bytes)));
    const int g_n = static_cast<int>(std::max(1.0, std::min<double>(p.tiles_n, kGroupL2Bytes * p.tiles_n / b_bytes)));
    const double by_m = a_bytes + b_bytes * ((m_units + g_m - 1) / g_m);
    const double by_n = b_bytes + a_bytes * ((p.tiles_n + g_n - 1) / g_n);
    p.group_n = by_n < by_m ? 1 : 0;
    p.group = p.group_n ? g_n : g_m;
  }
  const size_t esz = a.out_f32 ? 4 : 2;
  p.vec_store = (reinterpret_cast<uintptr_t>(a.d) % 16 == 0) && ((a.ldd * esz) % 16 == 0);
  CUtensorMap md{}, mq{}, mlu{}, ml2{};
  p.split_k = 1;
  p.kb_per_split = p.num_kb;
  if (!a.quant && a.lora_r == 0 && !pair && a.partial) {
    int per = 0;
    const int sk = gemm_split_k(a.M, a.N, a.K, &per);
    if (sk > 1 && a.partial_bytes >= gemm_split_k_bytes(a.M, a.N, sk)) {
      // partial accumulators [split_k, M, N] FP32 in the workspace, then a
      // fixed-order reduction that applies alpha and converts
      GParams q = p;
      q.split_k = sk;
      q.kb_per_split = per;
      q.part = a.partial;
      q.tma_store = 0;
      cudaError_t e = launch_typed<true, false, false>(ma, mb, md, mq, mlu, ml2, q, stream);
      if (e != cudaSuccess) return e;
      return a.out_f32 ? launch_partial_reduce<true>(q, sk, p.num_tiles, stream)
                       : launch_partial_reduce<false>(q, sk, p.num_tiles, stream);
    }
  }
  if (a.lora_r > 0) {
    // LoRA branch: two BF16 k-blocks (hi, lo) per 64 columns of U; boxes of
    // 64 columns x the code boxes' rows (reads past r are zero)
    if (a.quant) return cudaErrorInvalidValue;
    p.lora_kb = static_cast<int>(2 * (a.lora_rpad / 64));
    if (!make_lora_bf16_map(&mlu, a.lora_uhl, a.M, 2 * a.lora_rpad, 2 * a.lora_rpad, BM) ||
        !make_lora_bf16_map(&ml2, a.lora_l2, a.N, a.lora_r, a.lora_r,
                            pair ? Layout<true>::kBRows : Layout<false>::kBRows))
      return cudaErrorInvalidValue;
  }
  p.tma_store = !a.out_f32 && a.d != nullptr && p.vec_store;
  if (p.tma_store && !make_d_map(&md, a.d, a.M, a.N, a.ldd)) return cudaErrorInvalidValue;
  if (a.quant) {
    // BF16 output only; N % 32 == 0 and 16-byte aligned codes (checked by the caller)
    if (a.out_f32) return cudaErrorInvalidValue;
    p.q_codes = a.q_codes;
    p.q_sf = a.q_sf;
    p.q_tensor_scale = a.q_tensor_scale;
    p.q_amax_in = a.q_amax_in;
    p.q_amax_out = reinterpret_cast<uint32_t*>(a.q_amax_out);
    p.q_sf_mma = a.q_sf_mma;
    p.q_kb_count = a.N / 16;
    p.q_katoms = (p.q_kb_count + 3) / 4;
    if (!make_qcodes_map(&mq, a.q_codes, a.M, a.N)) return cudaErrorInvalidValue;
    return pair ? launch_typed<false, true, true>(ma, mb, md, mq, mlu, ml2, p, stream)
                : launch_typed<false, false, true>(ma, mb, md, mq, mlu, ml2, p, stream);
  }
  if (p.lora_kb > 0) {
    if (pair)
      return a.out_f32 ? launch_typed<true, true, false, true>(ma, mb, md, mq, mlu, ml2, p, stream)
                       : launch_typed<false, true, false, true>(ma, mb, md, mq, mlu, ml2, p, stream);
    return a.out_f32 ? launch_typed<true, false, false, true>(ma, mb, md, mq, mlu, ml2, p, stream)
                     : launch_typed<false, false, false, true>(ma, mb, md, mq, mlu, ml2, p, stream);
  }
  if (pair) {
    // the workspace past its header holds the tail split's partial blocks
    p.part = a.partial;
    return a.out_f32 ? launch_typed<true, true, false>(ma, mb, md, mq, mlu, ml2, p, stream, a.partial_bytes)
                     : launch_typed<false, true, false>(ma, mb, md, mq, mlu, ml2, p, stream, a.partial_bytes);
  }
  return a.out_f32 ? launch_typed<true, false, false>(ma, mb, md, mq, mlu, ml2, p, stream)
                   : launch_typed<false, false, false>(ma, mb, md, mq, mlu, ml2, p, stream);
}

}  // namespace nvfp4
