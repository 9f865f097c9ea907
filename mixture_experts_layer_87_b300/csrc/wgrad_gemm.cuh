// Weight-gradient GEMM of the backward pass on the tcgen05 tensor cores
// (sm_103a): for every group g (an expert),
//
//   out[g][m][n] = sum over k in [0, len_g) of A[m][ka_g + k] * B[n][kb_g + k]     (fp32)
//
// A [M rows, *] and B [N rows, *] are K-major bf16: activations transposed so
// that the expert's tokens run along K (dW2 = dY^T H: A = dY^T, B = H^T;
// dW13 = dAB^T X: A = dAB^T, B = X^T).  The tokens of one expert are a K range
// whose start and length are multiples of 64 (the padded columns are zero).
// Weight gradients stay fp32 (ai.flicky.cc 3.3 item 1: weight gradients are
// kept in higher precision).
//
// One CTA per 128 x 256 output tile of one group: warp 0 issues the TMA loads
// (128-byte swizzle, 4-stage ring), one thread of warp 1 the kind::f16 MMAs
// (M = 128, N = 256, K = 16) into a 256-column TMEM accumulator, warps 2..5
// store it (one TMEM lane quarter each).  A group with no tokens gets zeros.
// Every wait is bounded, as in the other GEMMs.
#pragma once

#include <cuda_bf16.h>

#include "gemm.cuh"
#include "ptx.cuh"

namespace moe {

struct WgradGroup {
  int32_t ka, kb, len, pad;  // K offsets into A and B, K length (multiples of 64)
};

struct WgradArgs {
  const WgradGroup* groups;  // [n_groups], device
  int32_t M, N;              // output rows and columns per group
  float* out;                // [n_groups][M][N]
  int* status;
};

constexpr int kWgStages = 4;
constexpr size_t wgrad_smem_bytes() { return 1024 + size_t(kWgStages) * (128 * 128 + 256 * 128) + 256; }

__global__ void __launch_bounds__(192, 1)
    wgrad_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const WgradArgs args) {
  constexpr int BM = 128, BN = 256, BK = 64, STAGES = kWgStages;
  constexpr uint32_t A_BYTES = BM * 128, B_BYTES = BN * 128, TMEM_COLS = BN;
  const int n_idx = blockIdx.x, m_idx = blockIdx.y, g = blockIdx.z;
  const WgradGroup grp = args.groups[g];
  const int nk = grp.len / BK;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* mma_done = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0 && nk > 0) {  // TMA producer
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES && !mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, args.status)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
        tma_load_2d(sA + s * A_BYTES, &tmA, grp.ka + i * BK, m_idx * BM, &full[s]);
        tma_load_2d(sB + s * B_BYTES, &tmB, grp.kb + i * BK, n_idx * BN, &full[s]);
        issued = i + 1;
      }
      // copies in flight land before the CTA may exit (abnormal exit only)
      if (*abort_flag)
        for (int i = max(0, issued - STAGES); i < issued; ++i) mbar_wait(&full[i % STAGES], (i / STAGES) & 1, args.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      constexpr uint32_t idesc = idesc_make(1u, BM, BN);
      bool ok = true;
      for (int i = 0; i < nk && ok; ++i) {
        const int s = i % STAGES;
        ok = mbar_wait(&full[s], (i / STAGES) & 1, args.status);
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          mma_bf16(tmem_base, sdesc_k128(a0 + k * 32), sdesc_k128(b0 + k * 32), idesc, (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
      }
      mma_commit(acc_full);
      mma_commit(mma_done);  // every MMA has completed before TMEM is released
      mbar_wait(mma_done, 0, args.status);
    }
  } else {  // epilogue: warps 2..5, one TMEM lane quarter each
    const int quarter = warp & 3;
    const int m = m_idx * BM + quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool ok = mbar_wait(acc_full, 0, args.status);
    tc_fence_after();
    float* orow = args.out + ((int64_t)g * args.M + m) * args.N;
    const bool m_ok = m < args.M;
    if (nk == 0) {  // no tokens: a zero gradient
#pragma unroll 1
      for (int c = 0; c < BN; c += 4) {
        const int n = n_idx * BN + c;
        if (m_ok && n < args.N) *reinterpret_cast<float4*>(orow + n) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else if (__all_sync(0xffffffffu, ok && !*abort_flag)) {  // tcgen05.ld is warp-collective
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(t_lane + c * 32, v);
        const int n0 = n_idx * BN + c * 32;
        if (!m_ok || n0 >= args.N) continue;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          if (n0 + i < args.N) *reinterpret_cast<float4*>(orow + n0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace moe
