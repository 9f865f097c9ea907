// Shared pieces of the tcgen05 GEMMs of this library, and the router logits
// GEMM (sm_103a).
//
// Router logits (ai.flicky.cc 2.1.2: s_{i,t} = sigmoid(u_t^T e_i), computed in
// bf16 with fp32 accumulation -- section 3.3 keeps the router out of FP8):
//
//   z_split[t, e] = sum over the split's K range of u[t, k] * e[e, k]
//
// One CTA computes one 128 x 128 tile of one K split: warp 0 streams u and
// centroid tiles with TMA (128-byte swizzle, 4-stage ring), one thread of
// warp 1 issues kind::f16 MMAs (K = 16) into a TMEM accumulator, warps 2..5
// store it as fp32.  With few tokens (a decode step) the K dimension is
// split over several CTAs so the centroids stream through many SMs; the
// top-k kernel adds the splits in a fixed order, so the logits stay
// deterministic.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "ptx.cuh"

namespace moe {

enum class Epi : int { F32 = 0, BF16 = 1, SWIGLU = 2 };

// One expert's rows: A rows [a_row0, a_row0 + m), output rows [out_row0, ...),
// and the number of row chunks of the groups before it (mt_start).
struct GroupEntry {
  int32_t a_row0, out_row0, m, mt_start;
};

// Arguments of the FP8 expert GEMM (fp8_gemm.cuh).
struct GemmArgs {
  // Group description: either a device table (routed experts, sizes known
  // only on the device) or n_groups uniform groups of uni_m rows.
  const GroupEntry* groups;    // nullptr -> uniform groups
  const int32_t* mt_total;     // device: total 128-row tiles over the table
  const int32_t* chunk_group;  // device: group of every 128-row tile of the table
  int32_t n_groups;
  int32_t uni_m, uni_a_step, uni_out_step;
  int32_t N, K;
  int32_t b_rows_per_group;  // rows of B per group in its 2-D view
  int32_t a_rows_cap;        // rows allocated in A (bounds the scale reads)
  void* out;                 // bf16 y, or E4M3 codes of h (SWIGLU)
  int64_t out_ld;            // elements per output row
  const float* a_scale;      // [K/128][a_scale_ld]
  int64_t a_scale_ld;
  const float* b_scale;      // [G][b_rows_per_group/128][K/128]
  float* out_scale;          // SWIGLU: [N/256 = I/128][out_scale_ld]
  int64_t out_scale_ld;
  int* queue;                // item counter, zero at launch
  int* status;
#ifdef MOE_CHECK
  // extents the range-checked build checks against (absent from the normal
  // build: a larger argument block costs the 16-warp epilogue a register spill)
  int64_t b_rows;            // rows of B
  int32_t out_rows;          // rows allocated in out
#endif
};

struct TileCoord {
  int32_t g, m_idx, n_idx, a_row, out_row, rows_valid;
};

// SiLU(x) = x * sigmoid(x), with the fast reciprocal division (its result is
// rounded to bf16 or quantised to E4M3 next; for x -> -inf the denominator
// overflows and the quotient is the correct limit 0).
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Store 32 fp32 values as bf16 (64 contiguous bytes).
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float (&v)[32]) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    d4[q] = w;
  }
}

// UE8M0 scale (DeepSeek-V3.1's FP8 scales are bare powers of two,
// ai.flicky.cc in its continuation of section 3.5): the smallest power of two
// >= s for a positive finite fp32 s -- s itself when its mantissa bits are
// zero, else the next exponent; scales below 2^-126 become 2^-126.
__device__ __forceinline__ float pow2_ceil(float s) {
  constexpr float kMinNormal = 1.17549435e-38f;  // 2^-126
  if (!(s > kMinNormal)) return kMinNormal;
  const uint32_t b = __float_as_uint(s);
  return (b & 0x7FFFFFu) ? __uint_as_float((b & 0x7F800000u) + 0x00800000u) : s;
}

// Two fp32 -> two E4M3 codes, round-to-nearest-even, saturating (cvt.rn.satfinite).
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// ---------------------------------------------------------------------------
// Router logits GEMM.
struct LogitsArgs {
  int32_t T, E, K;
  int32_t kb_per_split;  // 64-wide K blocks per split
  float* z;              // [splits][T][E]
  int64_t split_stride;  // T * E
  int* status;
};

constexpr int kLogitsStages = 4;
constexpr size_t logits_smem_bytes() { return 1024 + size_t(kLogitsStages) * (128 * 128 + 128 * 128) + 256; }

__global__ void __launch_bounds__(192, 1)
    logits_gemm_kernel(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmC,
                       const LogitsArgs args) {
  constexpr int BM = 128, BN = 128, BK = 64, STAGES = kLogitsStages;
  constexpr uint32_t A_BYTES = BM * 128, B_BYTES = BN * 128, TMEM_COLS = BN;
  const int mt = (args.T + BM - 1) / BM, nt = (args.E + BN - 1) / BN;
  const int split = blockIdx.x / (mt * nt), t = blockIdx.x % (mt * nt);
  const int n_idx = t / mt, m_idx = t % mt;
  const int num_kb = (args.K + BK - 1) / BK;
  const int kb0 = split * args.kb_per_split, kb1 = min(num_kb, kb0 + args.kb_per_split);
  if (kb0 >= kb1) return;  // whole CTA: nothing to do
  const int nk = kb1 - kb0;

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
    tma_prefetch_desc(&tmU);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES && !mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, args.status)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
        tma_load_2d(sA + s * A_BYTES, &tmU, (kb0 + i) * BK, m_idx * BM, &full[s]);
        tma_load_2d(sB + s * B_BYTES, &tmC, (kb0 + i) * BK, n_idx * BN, &full[s]);
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
    const int row = m_idx * BM + quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool ok = mbar_wait(acc_full, 0, args.status);
    tc_fence_after();
    if (__all_sync(0xffffffffu, ok && !*abort_flag)) {  // tcgen05.ld is warp-collective
      float* zrow = args.z + split * args.split_stride + (int64_t)row * args.E;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(t_lane + c * 32, v);
        const int col0 = n_idx * BN + c * 32;
        if (row >= args.T || col0 >= args.E) continue;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (col0 + i < args.E) zrow[col0 + i] = v[i];
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
