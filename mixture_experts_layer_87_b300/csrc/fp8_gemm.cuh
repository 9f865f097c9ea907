// Persistent grouped FP8 expert GEMM on the tcgen05 tensor cores (sm_103a):
// the fine-grained FP8 scheme of ai.flicky.cc section 3.3 (items 2-3).
//
//   out[rows of group g] = epilogue( sum_kb  P_kb * s_x[row, kb] * s_w[block, kb] )
//   P_kb = X_q[rows, 128 kb .. 128 kb + 128) . W_q,g[cols, same K]^T   (E4M3 codes)
//
// Tokens sit on the 128 TMEM lanes (one row per lane) and weight rows on the
// columns, so the activation tile scale s_x of a lane is one number per
// 128-wide K block and the weight block scale s_w one number per 128 columns:
// the promotion of a 128-K partial into fp32 costs one FMA per element.
//
// Work item = (group g, 256-column weight block n, 128-row tile m), m
// fastest; one CTA per SM takes items from a shared queue (warp 2 fetches
// and decodes them, see the item ring of expert_gemm.cuh).  Warp 0
// issues TMA loads into a 4-stage ring (16 KB of tokens + 32 KB of weights
// per 128-K stage), one thread of warp 1 issues kind::f8f6f4 MMAs (K = 32)
// into one of two TMEM partial buffers (2 x 256 columns), and the epilogue
// warps (warps 4 .., two or four warpgroups) promote: each reads its lane
// quarter's share of the partial in 16-column slices, multiplies by
// s_x * s_w and adds into fp32 registers (packed fp32x2 FMAs), and frees the
// buffer for the MMA two K blocks ahead as soon as its last slice is in
// registers.  Warp 3 only lends its registers: the first warpgroup gives up
// most of its registers to the epilogue warpgroups (setmaxnreg), so that an
// epilogue warp can hold its 128 accumulators and four slices (64 more
// registers) at once and wait for TMEM twice per K block instead of four
// times.  Warps whose 32 rows all lie past the group's end keep the barrier
// phases in step without loading anything.
//
// Between items the MMA can run only two K blocks ahead of the epilogue, so
// the item tail is kept short: the scheduler warp stages the scales of an
// item's first K blocks in its ring slot (their memory latency is spent up to
// four items early), and the bf16 output rows leave through shared memory in
// coalesced stores.
//
// Epilogues:
//   SWIGLU  the weight block holds 128 gate rows then the 128 matching up
//           rows (w13 interleave): h = SiLU(gate) * up for 128 features,
//           quantised per row over those 128 features (scale = amax/448,
//           E4M3 codes, the 1 x 128 activation tile of the down GEMM).
//   BF16    y as bf16.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "expert_gemm.cuh"
#include "gemm.cuh"
#include "ptx.cuh"

namespace moe {

// EW epilogue warps, EW / 4 per TMEM lane quarter.  8: 128 accumulators per
// thread, TMEM read four slices per wait; 16: 64 accumulators per thread,
// one slice per wait, twice the warps on a quarter -- the better choice when
// few rows per tile are valid (a decode step: 8 tokens per expert on
// average) and all the work falls on one quarter.
//
// Registers: the block launches with LAUNCH_REGS per thread (the most that
// __launch_bounds__(THREADS, 1) allows, which the host checks against the
// compiled kernel); warpgroup 0 (producer, MMA, scheduler, lender) drops to
// CTRL_REGS and the epilogue warpgroups rise to EPI_REGS.
template <int EW>
struct F8Shape {
  static constexpr int BM = 128, BN = 256, BK = 128, UK = 32;
  static constexpr uint32_t A_BYTES = BM * 128, B_BYTES = BN * 128;
  static constexpr int STAGES = 4;
  static constexpr int EPI_WARPS = EW;
  static constexpr int CG = EW / 4;
  static constexpr int BATCH = CG == 2 ? 4 : 1;        // 16-column slices per TMEM wait
  static constexpr int THREADS = 32 * (4 + EW);        // producer, MMA, scheduler, lender, epilogue
  static constexpr int LAUNCH_REGS = 65536 / THREADS / 8 * 8;
  static constexpr int CTRL_REGS = 48;
  static constexpr int EPI_REGS = (LAUNCH_REGS * THREADS - 128 * CTRL_REGS) / (32 * EW) / 8 * 8;
  static_assert(CG == 2 || CG == 4, "column groups");
  static_assert(128 * CTRL_REGS + 32 * EW * EPI_REGS <= LAUNCH_REGS * THREADS, "register split");
  static_assert(EPI_REGS <= 256 && EPI_REGS >= LAUNCH_REGS, "register split");
  // promotion scales of the first AHEAD K blocks of an item, staged in its
  // ring slot by the scheduler warp: s_x of the 128 rows, then s_w of the
  // two 128-column weight blocks, per K block; later K blocks are loaded
  // AHEAD blocks before their use
  static constexpr int AHEAD = 3;
  static constexpr int SLOT_FLOATS = AHEAD * 128 + AHEAD * 2 + 2;
  // bf16 results of 8 epilogue warps (256 bytes per row and warp) leave
  // through a per-warp shared buffer, see warp_rows_out; the 64 code bytes
  // per row of the SwiGLU epilogue, and the 16-warp shapes, store directly
  template <Epi EPI>
  __host__ __device__ static constexpr bool stage_out() {
    return CG == 2 && EPI == Epi::BF16;
  }
};

// Row-per-lane results to global rows.  Lane l holds 64 contiguous bytes of
// row row0 + l; stored straight from the registers, each 16-byte store of the
// warp would touch 32 rows (32 cache lines).  The warp writes its 32 x 64
// bytes to a shared buffer instead (an 80-byte pitch puts the 16-byte writes
// of 8 consecutive lanes in distinct banks) and stores them back with 4 lanes
// per row: 8 rows, 8 lines, per instruction.  Rows at or past `rows` are not
// written; every lane of the warp calls this.
constexpr int kOutPitch = 80;
constexpr int kOutWarpBytes = 32 * kOutPitch;

__device__ __forceinline__ void warp_rows_out(uint8_t* wbuf, const uint4 (&v)[4], uint8_t* col0, int64_t ld_bytes,
                                              int row0, int rows, int lane) {
  uint4* mine = reinterpret_cast<uint4*>(wbuf + lane * kOutPitch);
#pragma unroll
  for (int q = 0; q < 4; ++q) mine[q] = v[q];
  __syncwarp();
  const int part = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = i * 8 + (lane >> 2);
    if (row < rows)
      *reinterpret_cast<uint4*>(col0 + (int64_t)(row0 + row) * ld_bytes + part * 16) =
          *reinterpret_cast<const uint4*>(wbuf + row * kOutPitch + part * 16);
  }
  __syncwarp();
}

template <Epi EPI, int EW>
constexpr size_t fp8_gemm_smem_bytes() {
  using S = F8Shape<EW>;
  return 1024 + size_t(S::STAGES) * (S::A_BYTES + S::B_BYTES) + 512 /* barriers, item ring */ +
         2 * S::CG * 128 * sizeof(float) /* amax exchange: 2 items x CG column groups x 128 rows */ +
         kQueueSlots * S::SLOT_FLOATS * sizeof(float) /* staged scales */ +
         (S::template stage_out<EPI>() ? size_t(EW) * kOutWarpBytes : 0) /* output staging */;
}

// Item -> (group, column block, row tile); the same ordering and table as
// the bf16 expert GEMM (chunks of 128 rows).
__device__ __forceinline__ bool f8decode(const GemmArgs& a, int tile, int items, int nb, TileCoord& tc) {
  constexpr int BM = 128;
  if (tile >= items) return false;
  if (a.groups == nullptr) {
    const int mt = (a.uni_m + BM - 1) / BM;
    const int per_group = mt * nb;
    tc.g = tile / per_group;
    const int local = tile - tc.g * per_group;
    tc.n_idx = local / mt;
    tc.m_idx = local - tc.n_idx * mt;
    tc.a_row = tc.g * a.uni_a_step + tc.m_idx * BM;
    tc.out_row = tc.g * a.uni_out_step + tc.m_idx * BM;
    tc.rows_valid = min(BM, a.uni_m - tc.m_idx * BM);
    return true;
  }
  const int cg = __ldg(a.chunk_group + tile / nb);  // group | the weights' expert << 16
  const int4 G = __ldg(reinterpret_cast<const int4*>(a.groups) + (cg & 0xFFFF));  // {a_row0, out_row0, m, mt_start}
  const int mt = (G.z + BM - 1) / BM;
  const int local = tile - G.w * nb;
  tc.g = cg >> 16;
  tc.n_idx = local / mt;
  tc.m_idx = local - tc.n_idx * mt;
  tc.a_row = G.x + tc.m_idx * BM;
  tc.out_row = G.y + tc.m_idx * BM;
  tc.rows_valid = min(BM, G.z - tc.m_idx * BM);
  return true;
}

// Promotion arithmetic on packed pairs: an accumulator pair is one 64-bit
// register (two fp32 lanes), so fma.rn.f32x2 -- two correctly rounded fp32
// FMAs, as fmaf -- needs no repacking of the accumulators.
__device__ __forceinline__ uint64_t pair_of(float s) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(s));
  return r;
}

// a += (v0, v1) * s2
__device__ __forceinline__ void fma2(uint64_t& a, uint32_t v0, uint32_t v1, uint64_t s2) {
  asm("{\n\t.reg .b64 val;\n\t"
      "mov.b64 val, {%1, %2};\n\t"
      "fma.rn.f32x2 %0, val, %3, %0;\n\t}"
      : "+l"(a)
      : "r"(v0), "r"(v1), "l"(s2));
}

__device__ __forceinline__ float lo_of(uint64_t a) { return __uint_as_float(static_cast<uint32_t>(a)); }
__device__ __forceinline__ float hi_of(uint64_t a) { return __uint_as_float(static_cast<uint32_t>(a >> 32)); }

// POW2: the SwiGLU epilogue quantises h with UE8M0 scales (amax/448 rounded up
// to a power of two); a template flag, since one more argument word costs the
// 16-warp epilogue a register spill.
template <Epi EPI, int EW, bool POW2 = false>
__global__ void __launch_bounds__(F8Shape<EW>::THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmArgs args) {
  using S = F8Shape<EW>;
  constexpr int BN = S::BN, STAGES = S::STAGES;
  constexpr uint32_t A_BYTES = S::A_BYTES, B_BYTES = S::B_BYTES;
  constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(EPI == Epi::SWIGLU || EPI == Epi::BF16, "FP8 epilogues");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;  // [2] partial buffer written
  uint64_t* acc_empty = acc_full + 2;   // [2] partial buffer drained (8 warps)
  uint64_t* quarter_bar = acc_empty + 2;  // [4] the CG warps of one lane quarter
  uint64_t* mma_done = quarter_bar + 4;
  ItemRing ring;
  ring.q_full = mma_done + 1;
  ring.q_empty = ring.q_full + kQueueSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring.q_empty + kQueueSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  ring.slot = reinterpret_cast<int*>(tmem_slot + 4);
  float* amax_x = reinterpret_cast<float*>(smem + STAGES * (A_BYTES + B_BYTES) + 512);  // [2][CG][128]
  float* slot_scales = amax_x + 2 * S::CG * 128;  // [kQueueSlots][SLOT_FLOATS]
  uint8_t* out_stage = reinterpret_cast<uint8_t*>(slot_scales + kQueueSlots * S::SLOT_FLOATS);  // [EW][32 x 80]
  constexpr int AHEAD = S::AHEAD, SLOT_FLOATS = S::SLOT_FLOATS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = (args.N + BN - 1) / BN;
  const int num_kb = args.K / S::BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], S::EPI_WARPS);
    }
    for (int q = 0; q < 4; ++q) mbar_init(&quarter_bar[q], S::CG);
    for (int q = 0; q < kQueueSlots; ++q) {
      mbar_init(&ring.q_full[q], 1);
      mbar_init(&ring.q_empty[q], 2 + S::EPI_WARPS);  // producer, MMA thread, epilogue warps
    }
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

  if (warp < 4) {
    // warpgroup 0: warp 3 only lends its registers to the epilogue warps
    regs_release<S::CTRL_REGS>();
    if (warp == 2) {
      // ------------------------------------------------------------ item scheduler
      // Lane 0 takes the items; the whole warp stages each item's first
      // scales in its slot before publishing it, so their memory latency is
      // spent up to kQueueSlots items ahead of the epilogue.
      const int items = args.groups == nullptr ? (args.uni_m + 127) / 128 * nb * args.n_groups
                                               : __ldg(args.mt_total) * nb;
      const int KB = args.K / S::BK;
      int item = blockIdx.x;
      for (uint32_t lt = 0;; ++lt) {
        TileCoord tc{-1, 0, 0, 0, 0, 0};
        const bool have = f8decode(args, item, items, nb, tc);  // item is warp-uniform
        if (have) {
          int next = 0;
          if (lane == 0) next = atomicAdd(args.queue, 1);  // the next one, while this one is staged
          item = gridDim.x + __shfl_sync(0xffffffffu, next, 0);
        }
        const uint32_t s = lt % kQueueSlots;
        if (lt >= kQueueSlots &&
            !__all_sync(0xffffffffu, xwait(&ring.q_empty[s], ((lt / kQueueSlots) & 1) ^ 1, args.status, abort_flag)))
          break;
        if (have) {
          float* ss = slot_scales + s * SLOT_FLOATS;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = tc.a_row + lane + 32 * i;
            const bool in = row < args.a_rows_cap;
#pragma unroll
            for (int kb = 0; kb < AHEAD; ++kb)
              ss[kb * 128 + lane + 32 * i] =
                  kb < num_kb && in ? __ldg(args.a_scale + (int64_t)kb * args.a_scale_ld + row) : 0.0f;
          }
          if (lane < 2 * AHEAD) {
            const int j = lane & 1, kb = lane >> 1;
            const int blk_row = (tc.g * args.b_rows_per_group + tc.n_idx * BN) / 128 + j;
            const bool blk_in = (EPI == Epi::SWIGLU || tc.n_idx * BN + j * 128 < args.N) &&
                                MOE_IN_RANGE(args.status, blk_row, args.b_rows / 128);
            ss[AHEAD * 128 + kb * 2 + j] =
                kb < num_kb && blk_in ? __ldg(args.b_scale + (int64_t)blk_row * KB + kb) : 0.0f;
          }
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) {
          volatile int* dst = ring.slot + s * 8;
          const int v[6] = {have ? tc.g : -1, tc.m_idx, tc.n_idx, tc.a_row, tc.out_row, tc.rows_valid};
#pragma unroll
          for (int i = 0; i < 6; ++i) dst[i] = v[i];
          mbar_arrive(&ring.q_full[s]);  // release: coordinates and scales
        }
        __syncwarp();
        if (!have) break;
      }
    } else if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        uint32_t it = 0, issued = 0;
        for (uint32_t lt = 0;; ++lt) {
          int v[6];
          if (!ring_take(ring, lt, v, args.status, abort_flag, false) || v[0] < 0) break;
          const int b_row = v[0] * args.b_rows_per_group + v[2] * BN, a_row = v[3];
          (void)MOE_IN_RANGE(args.status, b_row, args.b_rows);  // a tile starting outside its tensor
          (void)MOE_IN_RANGE(args.status, a_row, args.a_rows_cap);
          bool ok = true;
          for (int kb = 0; kb < num_kb; ++kb, ++it) {
            const uint32_t s = it % STAGES;
            if (it >= STAGES && !xwait(&empty[s], ((it / STAGES) & 1) ^ 1, args.status, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
            tma_load_2d(sA + s * A_BYTES, &tmA, kb * S::BK, a_row, &full[s]);
            tma_load_2d(sB + s * B_BYTES, &tmB, kb * S::BK, b_row, &full[s]);
            issued = it + 1;
          }
          if (!ok) break;
        }
        // Abnormal exit only: copies still in flight land before the CTA leaves.
        if (*abort_flag)
          for (uint32_t j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
            mbar_wait(&full[j % STAGES], (j / STAGES) & 1, args.status);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_make(0u, 128, BN);  // E4M3 x E4M3 -> fp32, M = 128, N = 256
        uint32_t it = 0;
        bool ok = true;
        // the MMAs need no item coordinates (the producer placed the operands),
        // only where the item stream ends
        for (uint32_t lt = 0; ok; ++lt) {
          int v[6];
          if (!ring_take(ring, lt, v, args.status, abort_flag, false)) {
            ok = false;
            break;
          }
          if (v[0] < 0) break;
          for (int kb = 0; kb < num_kb && ok; ++kb, ++it) {
            const uint32_t s = it % STAGES, b = it & 1, u = it >> 1;
            ok = xwait(&full[s], (it / STAGES) & 1, args.status, abort_flag);
            if (ok && u > 0) ok = xwait(&acc_empty[b], (u & 1) ^ 1, args.status, abort_flag);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
  #pragma unroll
            for (int k = 0; k < S::BK / S::UK; ++k)
              mma_fp8(tmem_base + b * BN, sdesc_k128(a0 + k * 32), sdesc_k128(b0 + k * 32), idesc, k > 0 ? 1u : 0u);
            mma_commit(&empty[s]);
            mma_commit(&acc_full[b]);
          }
        }
        if (!ok) *abort_flag = 1;
        mma_commit(mma_done);  // every MMA of this CTA has completed before TMEM is released
        mbar_wait(mma_done, 0, args.status);
      }
    }
  } else {
    // ------------------------------------------------------------ promotion + epilogue
    regs_claim<S::EPI_REGS>();
    // The CG warps of one TMEM lane quarter split the 256 columns into CG
    // groups of NCH 16-column chunks.  SWIGLU: a warp takes NCH/2 gate
    // chunks of columns [0, 128) and the matching up chunks of [128, 256)
    // (gate feature f and up feature f stay in one thread); plain: NCH
    // consecutive chunks, all inside one 128-column weight block.
    constexpr int CG = S::CG, NCH = 16 / CG, NP = NCH / 2, BATCH = S::BATCH;
    const int ew = warp - 4;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int cg = ew >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const int KB = args.K / 128;
    auto col_of = [&](int j) -> uint32_t {
      if constexpr (EPI == Epi::SWIGLU)
        return j < NP ? (cg * NP + j) * 16 : 128 + (cg * NP + j - NP) * 16;
      else
        return (cg * NCH + j) * 16;
    };
    const int blk = EPI == Epi::SWIGLU ? 0 : (cg * NCH * 16) / 128;  // plain: weight block of my columns
    uint32_t it = 0, qphase = 0;
    bool ok = true;
    for (uint32_t lt = 0;; ++lt) {
      // take item lt with its staged scales: (sa, sb0, sb1)[i] belong to the
      // i-th K block from now
      float sa[AHEAD], sb0[AHEAD], sb1[AHEAD];
      int v[6];
      {
        const uint32_t s = lt % kQueueSlots;
        ok = __all_sync(0xffffffffu, xwait(&ring.q_full[s], (lt / kQueueSlots) & 1, args.status, abort_flag));
        if (!ok) break;
        const volatile int* src = ring.slot + s * 8;
#pragma unroll
        for (int i = 0; i < 6; ++i) v[i] = src[i];
        const volatile float* ss = slot_scales + s * SLOT_FLOATS;
#pragma unroll
        for (int i = 0; i < AHEAD; ++i) {
          sa[i] = ss[i * 128 + r];
          sb0[i] = ss[AHEAD * 128 + i * 2 + (EPI == Epi::SWIGLU ? 0 : blk)];
          sb1[i] = ss[AHEAD * 128 + i * 2 + (EPI == Epi::SWIGLU ? 1 : blk)];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring.q_empty[s]);
      }
      if (v[0] < 0) break;
      const TileCoord tc{v[0], v[1], v[2], v[3], v[4], v[5]};
      const bool row_ok = r < tc.rows_valid;
      const bool warp_rows = quarter * 32 < tc.rows_valid;
      const int a_row = tc.a_row + r;
      const bool a_in = a_row < args.a_rows_cap;
      const int b_row = tc.g * args.b_rows_per_group + tc.n_idx * BN;
      // range-checked build: the scale rows read and the output rows written
      // lie inside their tensors (else skipped)
      const bool blk_ok = (EPI == Epi::SWIGLU || tc.n_idx * BN + blk * 128 < args.N) &&
                          MOE_IN_RANGE(args.status, b_row / 128 + (EPI == Epi::SWIGLU ? 1 : blk), args.b_rows / 128);
      const bool out_ok = MOE_IN_RANGE(args.status, tc.out_row, args.out_rows) &&
                          MOE_IN_RANGE(args.status, tc.out_row + max(tc.rows_valid, 1) - 1, args.out_rows);
      const float* sa_ptr = args.a_scale + a_row;
      const float* sb_ptr = args.b_scale + (int64_t)(b_row / 128) * KB;
      const float* sb0_ptr = sb_ptr + (int64_t)blk * KB;                          // gate / my block
      const float* sb1_ptr = sb_ptr + (EPI == Epi::SWIGLU ? KB : (int64_t)blk * KB);  // up / my block
      uint64_t acc2[NCH * 8];  // acc2[c] = columns (2c, 2c + 1) of my NCH * 16
#pragma unroll
      for (int i = 0; i < NCH * 8; ++i) acc2[i] = 0;
#pragma unroll 1
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const uint32_t b = it & 1, u = it >> 1;
        const float s0 = sa[0] * sb0[0], s1 = sa[0] * sb1[0];
#pragma unroll
        for (int i = 0; i + 1 < AHEAD; ++i) {
          sa[i] = sa[i + 1];
          sb0[i] = sb0[i + 1];
          sb1[i] = sb1[i + 1];
        }
        if (kb + AHEAD < num_kb) {
          sa[AHEAD - 1] = a_in ? __ldg(sa_ptr + (int64_t)(kb + AHEAD) * args.a_scale_ld) : 0.0f;
          sb0[AHEAD - 1] = blk_ok ? __ldg(sb0_ptr + kb + AHEAD) : 0.0f;
          sb1[AHEAD - 1] = blk_ok ? __ldg(sb1_ptr + kb + AHEAD) : 0.0f;
        }
        ok = __all_sync(0xffffffffu, xwait(&acc_full[b], u & 1, args.status, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tb = t_lane + b * BN;
        bool released = false;
        if (warp_rows) {
          const uint64_t s0p = pair_of(s0), s1p = pair_of(s1);
          // BATCH 16-column slices per wait; the partial buffer is released
          // as soon as the last batch has landed in registers, before its FMAs
#pragma unroll
          for (int j0 = 0; j0 < NCH; j0 += BATCH) {
            uint32_t c[BATCH][16];
#pragma unroll
            for (int q = 0; q < BATCH; ++q) tmem_ld16_nowait(tb + col_of(j0 + q), c[q]);
#pragma unroll
            for (int q = 0; q < BATCH; ++q) tmem_ld_wait(c[q]);
            if (j0 + BATCH == NCH) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[b]);
              released = true;
            }
#pragma unroll
            for (int q = 0; q < BATCH; ++q) {
              const uint64_t sc = (EPI == Epi::SWIGLU && j0 + q >= NP) ? s1p : s0p;
#pragma unroll
              for (int i = 0; i < 8; ++i) fma2(acc2[(j0 + q) * 8 + i], c[q][2 * i], c[q][2 * i + 1], sc);
            }
          }
        }
        if (!released) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
      }
      if (!ok) break;
      float acc[NCH * 16];
#pragma unroll
      for (int i = 0; i < NCH * 8; ++i) {
        acc[2 * i] = lo_of(acc2[i]);
        acc[2 * i + 1] = hi_of(acc2[i]);
      }
      if constexpr (EPI == Epi::SWIGLU) {
        // h = SiLU(gate) * up for my NP * 16 features; the row's 1 x 128 scale
        // needs the amax of the other CG - 1 warps of the quarter too.
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < NP * 16; ++i) {
          acc[i] = silu(acc[i]) * acc[NP * 16 + i];
          amax = fmaxf(amax, fabsf(acc[i]));
        }
        float* ax = amax_x + (lt & 1) * CG * 128;  // alternate slots: a partner may still read the last item's
        ax[cg * 128 + r] = amax;
        ok = group_sync(&quarter_bar[quarter], qphase, args.status, abort_flag);
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < CG; ++c) amax = fmaxf(amax, ax[c * 128 + r]);
        float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
        if constexpr (POW2) scale = pow2_ceil(scale);
        // h is a GEMM output known to fp32 accuracy: its codes are taken from
        // h * (1/scale), one correctly rounded reciprocal per row
        const float inv = 1.0f / scale;
        if (row_ok && out_ok) {
          uint8_t* q = static_cast<uint8_t*>(args.out) + (int64_t)(tc.out_row + r) * args.out_ld + tc.n_idx * 128 +
                       cg * NP * 16;
#pragma unroll
          for (int w = 0; w < NP; ++w) {
            uint4 pk;
            uint32_t* p32 = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = w * 16 + j * 4;
              const uint32_t lo = e4m3x2(acc[i] * inv, acc[i + 1] * inv);
              const uint32_t hi = e4m3x2(acc[i + 2] * inv, acc[i + 3] * inv);
              p32[j] = lo | (hi << 16);
            }
            reinterpret_cast<uint4*>(q)[w] = pk;
          }
          if (cg == 0) args.out_scale[(int64_t)tc.n_idx * args.out_scale_ld + tc.out_row + r] = scale;
        }
      } else if constexpr (S::template stage_out<EPI>()) {
        if (warp_rows && blk_ok && out_ok) {
          uint8_t* ycol = static_cast<uint8_t*>(args.out) + (int64_t)(tc.n_idx * BN + cg * NCH * 16) * 2;
#pragma unroll
          for (int c = 0; c < NCH / 2; ++c) {
            uint4 w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float* f = acc + c * 32 + q * 8;
              w[q] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                                pack_bf16x2(f[6], f[7]));
            }
            warp_rows_out(out_stage + ew * kOutWarpBytes, w, ycol + c * 64, (int64_t)args.out_ld * 2,
                          tc.out_row + quarter * 32, tc.rows_valid - quarter * 32, lane);
          }
        }
      } else {
        if (row_ok && blk_ok && out_ok) {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(args.out) + (int64_t)(tc.out_row + r) * args.out_ld +
                             tc.n_idx * BN + cg * NCH * 16;
#pragma unroll
          for (int c = 0; c < NCH / 2; ++c) {
            float vv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) vv[i] = acc[c * 32 + i];
            store_bf16x32(o + c * 32, vv);
          }
        }
      }
    }
    if (!ok) *abort_flag = 1;
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
