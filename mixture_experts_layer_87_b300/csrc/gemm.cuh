// Grouped GEMM on the 5th-generation tensor cores (tcgen05) for sm_103a.
//
//   out[rows of group g] = epilogue( A[rows of group g] . B_g^T )
//
// A is [rows, K] (K-major), B_g is [N, K] (K-major, nn.Linear layout), both
// streamed by TMA with 128-byte swizzling into a STAGES-deep shared-memory
// ring; one thread issues tcgen05.mma into a TMEM accumulator; epilogue warps
// read TMEM with tcgen05.ld and write the output.  One CTA computes one
// 128 x BN tile.  Groups are the experts of the layer (ai.flicky.cc 2.1.2:
// routed experts see a variable, dropless number of rows; shared experts see
// every token), so the tile list is built on the device from the per-expert
// row offsets and never read back by the host.
//
// Precisions:
//   bf16: kind::f16 MMAs (K = 16 each), one fp32 accumulator in TMEM.
//   FP8 (ai.flicky.cc section 3.3 items 2-3): kind::f8f6f4 MMAs on E4M3
//   codes.  Every 128 elements of K (one pipeline stage) the MMAs write a
//   fresh fp32 partial sum into one of two TMEM buffers; the epilogue warps
//   multiply it by (activation tile scale x weight block scale) and add it
//   into fp32 registers -- the "promotion to FP32 every N_c = 128" of the
//   pages, done by the CUDA cores while the tensor cores fill the other buffer.
//
// Epilogues:
//   F32      store the fp32 accumulator (router logits).
//   BF16     store bf16 (down projection).
//   SWIGLU   B tiles hold 128 gate rows then the 128 matching up rows
//            (w13 interleave), so h = SiLU(gate) * up for 128 features is
//            finished inside the tile and stored as bf16, or (FP8) as E4M3
//            codes with a 1 x 128 scale per row: the input of the down GEMM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "ptx.cuh"

namespace moe {

enum class Epi : int { F32 = 0, BF16 = 1, SWIGLU = 2 };

// One expert's rows: A rows [a_row0, a_row0 + m), output rows [out_row0, ...),
// and the number of 128-row tiles of the groups before it (mt_start).
struct GroupEntry {
  int32_t a_row0, out_row0, m, mt_start;
};

struct GemmArgs {
  // Group description: either a device table (routed experts, sizes known
  // only on the device) or n_groups uniform groups of uni_m rows.
  const GroupEntry* groups;  // nullptr -> uniform groups
  const int32_t* mt_total;   // device: total 128-row tiles over the table
  int32_t n_groups;
  int32_t uni_m, uni_a_step, uni_out_step;
  int32_t N, K;
  int32_t b_rows_per_group;  // rows of B per group in its 2-D view
  int32_t a_rows_cap;        // rows allocated in A (bounds the scale reads)
  void* out;                 // F32 / BF16 / SWIGLU(bf16): element type per epilogue
  int64_t out_ld;            // elements per output row
  // FP8 only
  const float* a_scale;      // [K/128][a_scale_ld]
  int64_t a_scale_ld;
  const float* b_scale;      // [G][b_rows_per_group/128][K/128]
  float* out_scale;          // SWIGLU FP8: [N/256 ... = I/128][out_scale_ld]
  int64_t out_scale_ld;
  int* status;
};

template <bool FP8>
struct GemmShape {
  static constexpr int BM = 128;
  static constexpr int BK = FP8 ? 128 : 64;   // elements per stage: 128 bytes of K
  static constexpr int UK = FP8 ? 32 : 16;    // K of one MMA instruction
  static constexpr int EPI_WARPS = FP8 ? 8 : 4;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int STAGES = 4;
};

template <bool FP8, int BN>
constexpr size_t gemm_smem_bytes() {
  using S = GemmShape<FP8>;
  return 1024 /* alignment slack */ + size_t(S::STAGES) * (S::BM * 128 + BN * 128) + 256 /* barriers */ +
         2 * 128 * sizeof(float) /* amax exchange */;
}

struct TileCoord {
  int32_t g, m_idx, n_idx, a_row, out_row, rows_valid;
};

__device__ __forceinline__ bool decode_tile(const GemmArgs& a, int tile, int n_tiles, TileCoord& tc) {
  constexpr int BM = 128;
  if (a.groups == nullptr) {
    const int mt = (a.uni_m + BM - 1) / BM;
    const int per_group = mt * n_tiles;
    if (tile >= per_group * a.n_groups) return false;
    tc.g = tile / per_group;
    const int local = tile - tc.g * per_group;
    tc.n_idx = local / mt;
    tc.m_idx = local - tc.n_idx * mt;
    tc.a_row = tc.g * a.uni_a_step + tc.m_idx * BM;
    tc.out_row = tc.g * a.uni_out_step + tc.m_idx * BM;
    tc.rows_valid = min(BM, a.uni_m - tc.m_idx * BM);
    return true;
  }
  const int total = __ldg(a.mt_total) * n_tiles;
  if (tile >= total) return false;
  // last group whose first tile is <= tile (empty groups share the start of the next)
  int lo = 0, hi = a.n_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&a.groups[mid].mt_start) * n_tiles <= tile) lo = mid; else hi = mid - 1;
  }
  const GroupEntry G = a.groups[lo];
  const int mt = (G.m + BM - 1) / BM;
  const int local = tile - G.mt_start * n_tiles;
  tc.g = lo;
  tc.n_idx = local / mt;
  tc.m_idx = local - tc.n_idx * mt;
  tc.a_row = G.a_row0 + tc.m_idx * BM;
  tc.out_row = G.out_row0 + tc.m_idx * BM;
  tc.rows_valid = min(BM, G.m - tc.m_idx * BM);
  return true;
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + __expf(-x)); }

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

// Two fp32 -> two E4M3 codes, round-to-nearest-even, saturating (cvt.rn.satfinite).
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

template <bool FP8, int BN, Epi EPI>
__global__ void __launch_bounds__(GemmShape<FP8>::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs args) {
  using S = GemmShape<FP8>;
  constexpr int BM = S::BM, BK = S::BK, STAGES = S::STAGES;
  constexpr uint32_t A_BYTES = BM * 128, B_BYTES = BN * 128;
  constexpr uint32_t TMEM_COLS = FP8 ? 2 * BN : (BN < 32 ? 32 : BN);
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
  static_assert(EPI != Epi::SWIGLU || BN == 256, "SwiGLU tiles hold 128 gate + 128 up features");
  static_assert(!FP8 || BN == 256, "FP8 epilogue splits 256 columns over two warps per lane quarter");
  static_assert(!FP8 || EPI != Epi::F32, "router stays bf16");

  const int n_tiles = (args.N + BN - 1) / BN;
  TileCoord tc;
  if (!decode_tile(args, blockIdx.x, n_tiles, tc)) return;  // whole CTA: nothing to do

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment (in the shared window) of the swizzled operand tiles
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;   // [2]: FP8 partial buffers full; bf16 uses [0]
  uint64_t* acc_empty = acc_full + 2;    // [2]: FP8 partial buffers drained by the epilogue
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  float* amax_x = reinterpret_cast<float*>(smem + STAGES * (A_BYTES + B_BYTES) + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_kb = (args.K + BK - 1) / BK;
  const int b_row = tc.g * args.b_rows_per_group + tc.n_idx * BN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    mbar_init(&acc_empty[0], S::EPI_WARPS);
    mbar_init(&acc_empty[1], S::EPI_WARPS);
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % STAGES;
        if (kb >= STAGES && !mbar_wait(&empty[s], ((kb / STAGES) & 1) ^ 1, args.status)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
        tma_load_2d(sA + s * A_BYTES, &tmA, kb * BK, tc.a_row, &full[s]);
        tma_load_2d(sB + s * B_BYTES, &tmB, kb * BK, b_row, &full[s]);
        issued = kb + 1;
      }
      // Our copies must have landed before the CTA may exit (abnormal exit only:
      // normally the MMA thread already consumed every one of them).
      for (int kb = max(0, issued - STAGES); kb < issued; ++kb)
        mbar_wait(&full[kb % STAGES], (kb / STAGES) & 1, args.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_make(FP8 ? 0u : 1u, BM, BN);
      bool ok = true;
      for (int kb = 0; kb < num_kb && ok; ++kb) {
        const int s = kb % STAGES;
        ok = mbar_wait(&full[s], (kb / STAGES) & 1, args.status);
        uint32_t d_tmem = tmem_base;
        if (FP8) {
          const int b = kb & 1;
          if (ok && kb >= 2) ok = mbar_wait(&acc_empty[b], ((kb >> 1) & 1) ^ 1, args.status);
          d_tmem = tmem_base + b * BN;
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
        for (int k = 0; k < BK / S::UK; ++k) {
          const uint64_t ad = sdesc_k128(a0 + k * 32), bd = sdesc_k128(b0 + k * 32);
          if (FP8) mma_fp8(d_tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
          else mma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&empty[s]);
        if (FP8) mma_commit(&acc_full[kb & 1]);
      }
      if (!FP8) mma_commit(&acc_full[0]);
      // every MMA of this CTA has finished before TMEM is released
      mma_commit(mma_done);
      mbar_wait(mma_done, 0, args.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                 // 0 .. EPI_WARPS-1
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;       // row of the tile
    const bool row_ok = r < tc.rows_valid;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);

    if constexpr (!FP8) {
      const bool ok = mbar_wait(&acc_full[0], 0, args.status);
      tc_fence_after();
      // tcgen05.ld is warp-collective: the whole warp takes one decision
      if (__all_sync(0xffffffffu, ok && !*abort_flag)) {
        if constexpr (EPI == Epi::SWIGLU) {
          __nv_bfloat16* h = static_cast<__nv_bfloat16*>(args.out) + (int64_t)(tc.out_row + r) * args.out_ld +
                             tc.n_idx * 128;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float g[32], u[32];
            tmem_ld32(t_lane + c * 32, g);
            tmem_ld32(t_lane + 128 + c * 32, u);
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = silu(g[i]) * u[i];
            if (row_ok) store_bf16x32(h + c * 32, g);
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_ld32(t_lane + c * 32, v);
            const int col0 = tc.n_idx * BN + c * 32;
            if (!row_ok || col0 >= args.N) continue;
            if constexpr (EPI == Epi::F32) {
              float* o = static_cast<float*>(args.out) + (int64_t)(tc.out_row + r) * args.out_ld + col0;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (col0 + i < args.N) o[i] = v[i];
            } else {
              __nv_bfloat16* o =
                  static_cast<__nv_bfloat16*>(args.out) + (int64_t)(tc.out_row + r) * args.out_ld + col0;
              store_bf16x32(o, v);  // N is a multiple of 128 for bf16 outputs
            }
          }
        }
      }
    } else {
      // FP8: promote every 128-K partial into fp32 registers.
      const int half = ew >> 2;              // which 128 of the 256 columns
      // SwiGLU: half 0 -> gate [0,64) + up [128,192); half 1 -> gate [64,128) + up [192,256)
      // plain : half 0 -> cols [0,128);               half 1 -> cols [128,256)
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
      const int KB = args.K / 128;
      const int a_row = tc.a_row + r;
      const bool a_in = a_row < args.a_rows_cap;
      const float* sa_ptr = args.a_scale + a_row;
      const float* sb_ptr = args.b_scale + (int64_t)(b_row / 128) * KB;  // block row of this tile's first 128 rows
      // plain epilogue: the second 128 columns may lie beyond N (N a multiple of 128)
      const bool half_ok = EPI == Epi::SWIGLU || tc.n_idx * BN + half * 128 < args.N;
      float sa_next = a_in ? __ldg(sa_ptr) : 0.0f;
      bool ok = true;
#pragma unroll 1
      for (int kb = 0; kb < num_kb; ++kb) {
        const int b = kb & 1;
        const float sa = sa_next;
        if (kb + 1 < num_kb) sa_next = a_in ? __ldg(sa_ptr + (int64_t)(kb + 1) * args.a_scale_ld) : 0.0f;
        float s0, s1;  // scale of the first / second 32-column chunk pair
        if constexpr (EPI == Epi::SWIGLU) {
          s0 = sa * __ldg(sb_ptr + kb);        // gate block (rows b_row .. +128)
          s1 = sa * __ldg(sb_ptr + KB + kb);   // up block   (rows b_row+128 .. +256)
        } else {
          s0 = s1 = half_ok ? sa * __ldg(sb_ptr + (int64_t)half * KB + kb) : 0.0f;
        }
        ok = __all_sync(0xffffffffu, ok && mbar_wait(&acc_full[b], (kb >> 1) & 1, args.status));
        if (!ok) break;  // warp-uniform
        tc_fence_after();
        const uint32_t tb = t_lane + b * BN;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          int col;
          float sc;
          if constexpr (EPI == Epi::SWIGLU) {
            col = (c < 2) ? half * 64 + c * 32 : 128 + half * 64 + (c - 2) * 32;
            sc = (c < 2) ? s0 : s1;
          } else {
            col = half * 128 + c * 32;
            sc = s0;
          }
          float v[32];
          tmem_ld32(tb + col, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[c * 32 + i] = fmaf(v[i], sc, acc[c * 32 + i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[b]);
      }
      if (!ok) *abort_flag = 1;
      // all epilogue warps agree on abort before touching the output
      asm volatile("bar.sync 1, %0;" ::"r"(32 * S::EPI_WARPS) : "memory");
      const bool write = !*abort_flag;
      if constexpr (EPI == Epi::SWIGLU) {
        // h = SiLU(gate) * up for my 64 features, then one E4M3 scale per row per 128 features
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          acc[i] = silu(acc[i]) * acc[64 + i];
          amax = fmaxf(amax, fabsf(acc[i]));
        }
        amax_x[half * 128 + r] = amax;
        asm volatile("bar.sync 1, %0;" ::"r"(32 * S::EPI_WARPS) : "memory");
        amax = fmaxf(amax, amax_x[(half ^ 1) * 128 + r]);
        const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
        if (write && row_ok) {
          uint8_t* q = static_cast<uint8_t*>(args.out) + (int64_t)(tc.out_row + r) * args.out_ld +
                       tc.n_idx * 128 + half * 64;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint4 pk;
            uint32_t* p32 = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = w * 16 + j * 4;
              const uint32_t lo = e4m3x2(acc[i] / scale, acc[i + 1] / scale);
              const uint32_t hi = e4m3x2(acc[i + 2] / scale, acc[i + 3] / scale);
              p32[j] = lo | (hi << 16);
            }
            reinterpret_cast<uint4*>(q)[w] = pk;
          }
          if (half == 0) args.out_scale[(int64_t)tc.n_idx * args.out_scale_ld + tc.out_row + r] = scale;
        }
      } else {
        if (write && row_ok && half_ok) {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(args.out) + (int64_t)(tc.out_row + r) * args.out_ld +
                             tc.n_idx * BN + half * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = acc[c * 32 + i];
            store_bf16x32(o + c * 32, v);
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace moe
