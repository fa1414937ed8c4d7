// LoRA-SVD projection forward, first half (sm_103a, tcgen05 kind::f16).
//
// "Full-Stack FP4: Stable LLM Pretraining with Quantized Projections,
// Optimizers, and Attention", section 2.1: the weight is W = W_res +
// beta L2 L1, with the residual W_res in NVFP4 and the principal low-rank
// part L2 [dout, r], L1 [r, din] in BF16 (section 3 calls the
// reparametrisation fusable).  Y = X W^T is then
//     Y = (NVFP4 GEMM of X and W_res) + beta U L2^T,   U = BF16(X L1^T).
//
// This kernel computes the branch's intermediate U [T, r] on the tensor cores
// (BF16 x BF16, FP32 accumulation in TMEM, rounded to BF16) and prepares it
// for the NVFP4 GEMM, which adds beta U L2^T into its own accumulator: that
// accumulator holds sum(eA sfA eB sfB) and is scaled by alpha = sA sB only in
// the epilogue, so the branch must enter it as (beta / alpha) U L2^T.  The
// product v = RN(U * RN(beta / alpha)) is not a BF16 value, so it is split
// into hi = BF16(v) and lo = BF16(v - hi) (v - hi is exact in FP32), which
// together carry v to about 2^-16 relative; the GEMM runs two BF16 k-blocks
// per 64 columns of U (hi and lo, each against the same 64 columns of L2).
// Layout of that buffer, uhl [T, 2 rpad] BF16 (rpad = r rounded up to 64):
// columns 128 c .. 128 c + 63 hold hi of U's columns 64 c .., the next 64
// hold lo; columns of U past r are zero.
//
// One CTA per 128 rows of X (cta_group::1, M = 128, N = rpad <= 256):
//   warp 0      TMA producer (X and L1 boxes of 64 BF16 columns, 128-byte
//               swizzle, out-of-range elements read as zero);
//   warp 1      TMEM allocation and MMA issue (K = 16 per instruction);
//   warps 4-7   epilogue, one TMEM lane quarter each (lane = row).
// Every mbarrier wait is bounded; on a timeout the CTA records
// NVFP4_ERR_TIMEOUT in the status word, drains what it issued, frees TMEM
// and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kRows = 128;                 // rows of X per CTA
constexpr int kKb = 64;                    // BF16 elements of K per stage (128 bytes per row)
constexpr int kABytes = kRows * 128;       // 16 KB
constexpr int kMaxN = 256;                 // rpad limit
constexpr int kBBytesMax = kMaxN * 128;    // 32 KB
constexpr int kStageBytes = kABytes + kBBytesMax;
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr int kFirstEpiWarp = 4;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*alignment*/;

struct DownParams {
  int64_t T, din, r, rpad;
  int num_kb;
  uint32_t b_bytes;      // bytes of one L1 box (rpad rows x 128 bytes)
  uint32_t idesc;        // kind::f16, BF16 x BF16 -> F32, M = 128, N = rpad
  uint32_t tmem_cols;    // power of two >= rpad
  float beta;
  const float* sx;       // tensor scales of the two NVFP4 operands of the GEMM
  const float* sw;
  uint16_t* u;           // [T, r]
  uint16_t* uhl;         // [T, 2 rpad]
  uint32_t* status;
};

struct __align__(8) DownCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint16_t bf16_bits_rn(float f) {
  const __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<const uint16_t*>(&b);
}

__device__ __forceinline__ float bf16_value(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

__global__ void __launch_bounds__(kThreads, 1)
    lora_down_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_l1,
                     const DownParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DownCtl ctl;
  volatile int* abort_flag = &ctl.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kRows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&ctl.full[s], 1);
      ptx::mbar_init(&ctl.empty[s], 1);
    }
    ptx::mbar_init(&ctl.acc_full, 1);
    ctl.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl.tmem_base, p.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmap_x);
      ptx::prefetch_tensormap(&tmap_l1);
      uint32_t issued_mask = 0, issued_parity = 0;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = static_cast<uint32_t>(kb / kStages) & 1u;
        if (!ptx::mbar_wait(&ctl.empty[s], ph ^ 1u, abort_flag)) {
          ptx::set_status(p.status, kDevTimeout | (21u << 8));
          ctl.abort = 1;
          break;
        }
        uint8_t* st = smem + s * kStageBytes;
        ptx::mbar_arrive_expect_tx(&ctl.full[s], kABytes + p.b_bytes);
        ptx::tma_load_2d(st, &tmap_x, &ctl.full[s], kb * kKb, static_cast<int32_t>(m0));
        ptx::tma_load_2d(st + kABytes, &tmap_l1, &ctl.full[s], kb * kKb, 0);
        issued_mask |= 1u << s;
        issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
      }
      // every copy issued must land before the CTA exits
      for (int s = 0; s < kStages; ++s) {
        if (issued_mask & (1u << s)) {
          volatile int never = 0;
          if (!ptx::mbar_wait(&ctl.full[s], (issued_parity >> s) & 1u, &never))
            ptx::set_status(p.status, kDevTimeout | (22u << 8));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint64_t a_desc0 = ptx::smem_desc(ptx::smem_u32(smem), 16, 1024, ptx::kSwizzle128B);
      const uint64_t b_desc0 = ptx::smem_desc(ptx::smem_u32(smem + kABytes), 16, 1024, ptx::kSwizzle128B);
      bool ok = true;
      int kb = 0;
      for (; kb < p.num_kb; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = static_cast<uint32_t>(kb / kStages) & 1u;
        if (!ptx::mbar_wait(&ctl.full[s], ph, abort_flag)) {
          ptx::set_status(p.status, kDevTimeout | (23u << 8));
          ctl.abort = 1;
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t off = static_cast<uint32_t>(s * kStageBytes) >> 4;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // K = 16 BF16 = 32 bytes per instruction
          ptx::tc_mma_f16(tmem, a_desc0 + off + 2 * kk, b_desc0 + off + 2 * kk, p.idesc, (kb | kk) != 0 ? 1u : 0u);
        ptx::tc_commit(&ctl.empty[s]);
      }
      // The accumulator is complete (or abandoned) once every MMA issued so
      // far has finished: the epilogue waits for this before it reads TMEM,
      // and TMEM is not freed before it.
      ptx::tc_commit(&ctl.acc_full);
      // TMEM is freed below only after every MMA issued here has finished,
      // whether or not the epilogue read the accumulator.
      volatile int never = 0;
      if (!ptx::mbar_wait(&ctl.acc_full, 0, &never)) ptx::set_status(p.status, kDevTimeout | (25u << 8));
      (void)ok;
    }
  } else if (warp >= kFirstEpiWarp) {
    const int q = warp & 3;
    uint32_t ok = 1;
    if (lane == 0) ok = ptx::mbar_wait(&ctl.acc_full, 0, abort_flag) ? 1u : 0u;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        ptx::set_status(p.status, kDevTimeout | (24u << 8));
        ctl.abort = 1;
      }
    } else if (ctl.abort == 0) {
      ptx::tc_fence_after();
      const float alpha = __fmul_rn(*p.sx, *p.sw);
      const float c = __fdiv_rn(p.beta, alpha);
      const int64_t row = m0 + q * 32 + lane;
      const bool row_ok = row < p.T;
      uint16_t* urow = p.u + row * p.r;
      uint16_t* hrow = p.uhl + row * 2 * p.rpad;
      for (int c32 = 0; c32 < p.rpad / 32; ++c32) {
        uint32_t acc[32];
        ptx::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c32 * 32, acc);
        ptx::tmem_ld_wait();
        ptx::tmem_ld_regs_ready(acc);
        if (!row_ok) continue;
        const int col0 = c32 * 32;
        const int hcol0 = (col0 / 64) * 128 + (col0 % 64);  // hi; lo is 64 further
        uint32_t uw[16], hw[16], lw[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          uint16_t uh[2], hh[2], lh[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool in = col0 + j + e < p.r;
            const uint16_t ub = bf16_bits_rn(__uint_as_float(acc[j + e]));
            const float v = __fmul_rn(bf16_value(ub), c);
            const uint16_t hb = bf16_bits_rn(v);
            const uint16_t lb = bf16_bits_rn(__fsub_rn(v, bf16_value(hb)));
            uh[e] = ub;
            hh[e] = in ? hb : 0;
            lh[e] = in ? lb : 0;
          }
          uw[j / 2] = uh[0] | (static_cast<uint32_t>(uh[1]) << 16);
          hw[j / 2] = hh[0] | (static_cast<uint32_t>(hh[1]) << 16);
          lw[j / 2] = lh[0] | (static_cast<uint32_t>(lh[1]) << 16);
        }
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          *reinterpret_cast<uint4*>(hrow + hcol0 + 8 * v4) =
              make_uint4(hw[4 * v4], hw[4 * v4 + 1], hw[4 * v4 + 2], hw[4 * v4 + 3]);
          *reinterpret_cast<uint4*>(hrow + hcol0 + 64 + 8 * v4) =
              make_uint4(lw[4 * v4], lw[4 * v4 + 1], lw[4 * v4 + 2], lw[4 * v4 + 3]);
        }
        // U itself: r is a multiple of 8, so whole 16-byte pieces
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          if (col0 + 8 * v4 < p.r)
            *reinterpret_cast<uint4*>(urow + col0 + 8 * v4) =
                make_uint4(uw[4 * v4], uw[4 * v4 + 1], uw[4 * v4 + 2], uw[4 * v4 + 3]);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, p.tmem_cols);
  }
}

// Tensor map over a BF16 matrix [rows, cols] (row stride ld elements): box
// 64 columns x box_rows rows, 128-byte swizzle, out-of-range reads as zero.
bool make_bf16_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult res = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS;
}

}  // namespace

bool make_lora_bf16_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                        uint32_t box_rows) {
  return make_bf16_map(map, base, rows, cols, ld, box_rows);
}

cudaError_t launch_lora_down(const LoraArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  static std::mutex setup_mutex;
  static bool ready[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(setup_mutex);
    if (!ready[dev]) {
      e = cudaFuncSetAttribute(lora_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
      ready[dev] = true;
    }
  }
  DownParams p{};
  p.T = a.T;
  p.din = a.din;
  p.r = a.r;
  p.rpad = (a.r + 63) / 64 * 64;
  if (p.rpad > kMaxN) return cudaErrorInvalidValue;
  p.num_kb = static_cast<int>((a.din + kKb - 1) / kKb);
  p.b_bytes = static_cast<uint32_t>(p.rpad * 128);
  p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(p.rpad >> 3) << 17) |
            (static_cast<uint32_t>(kRows >> 4) << 24);
  p.tmem_cols = p.rpad <= 64 ? 64u : (p.rpad <= 128 ? 128u : 256u);
  p.beta = a.beta;
  p.sx = a.sx;
  p.sw = a.sw;
  p.u = a.u;
  p.uhl = a.uhl;
  p.status = a.status;
  CUtensorMap mx, ml1;
  if (!make_bf16_map(&mx, a.x, a.T, a.din, a.ldx, kRows) ||
      !make_bf16_map(&ml1, a.l1, a.r, a.din, a.din, static_cast<uint32_t>(p.rpad)))
    return cudaErrorInvalidValue;
  const int grid = static_cast<int>((a.T + kRows - 1) / kRows);
  lora_down_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mx, ml1, p);
  return cudaGetLastError();
}

}  // namespace nvfp4
