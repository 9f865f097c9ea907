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
// The kernel is bound by writing the fp32 gradients (4 bytes per weight, 45 GB
// for V3's routed experts), so it is built around the stores:
//   * persistent: one CTA per SM takes 128 x 256 output tiles (group-major,
//     so a group's operands stay in L2) from a shared queue (the item ring of
//     expert_gemm.cuh, fed by warp 2);
//   * warp 0 issues the TMA loads (128-byte swizzle, 4-stage ring that runs
//     on across tiles), one thread of warp 1 the kind::f16 MMAs (M = 128,
//     N = 256, K = 16) into one of two 256-column TMEM accumulators, so the
//     stores of tile i overlap the loads and MMAs of tile i + 1;
//   * warps 3..6 (one TMEM lane quarter each) read 32 x 32 fp32 blocks of
//     the accumulator into a 128-byte-swizzled shared-memory box (conflict
//     free) and write it with one TMA store each (a 3-D tensor map [G][M][N],
//     so a tile's rows past M or columns past N are clipped, never written
//     into the next group), double-buffered per warp.
// A group with no tokens gets zeros.  Every wait is bounded, as in the other
// GEMMs.
#pragma once

#include <cuda_bf16.h>

#include "expert_gemm.cuh"
#include "gemm.cuh"
#include "ptx.cuh"

namespace moe {

struct WgradGroup {
  int32_t ka, kb, len, pad;  // K offsets into A and B, K length (multiples of 64)
};

struct WgradArgs {
  const WgradGroup* groups;  // [n_groups], device
  int32_t n_groups;
  int32_t M, N;              // output rows and columns per group
  int32_t m_tiles, n_tiles;  // 128-row and 256-column tiles per group
  int* queue;                // item counter, zero at launch
  int* status;
};

constexpr int kWgStages = 4;
constexpr int kWgEpiWarps = 4;
constexpr int kWgThreads = 32 * (3 + kWgEpiWarps);
constexpr uint32_t kWgABytes = 128 * 128, kWgBBytes = 256 * 128;  // per stage: 64 K x (128 | 256) rows, bf16
constexpr uint32_t kWgBoxBytes = 32 * 32 * 4;                      // one 32 x 32 fp32 store box

constexpr size_t wgrad_smem_bytes() {
  return 1024 + size_t(kWgStages) * (kWgABytes + kWgBBytes) + size_t(kWgEpiWarps) * 2 * kWgBoxBytes +
         512 /* barriers, item ring */;
}

__global__ void __launch_bounds__(kWgThreads, 1)
    wgrad_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmOut, const WgradArgs args) {
  constexpr int BM = 128, BN = 256, BK = 64, STAGES = kWgStages, NACC = 2;
  constexpr uint32_t A_BYTES = kWgABytes, B_BYTES = kWgBBytes;
  constexpr uint32_t TMEM_COLS = NACC * BN;
  static_assert(TMEM_COLS == 512, "TMEM budget");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sOut = sB + STAGES * B_BYTES;  // [epilogue warp][2][32 x 128 bytes], 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + kWgEpiWarps * 2 * kWgBoxBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;  // [NACC]
  uint64_t* acc_empty = acc_full + NACC;
  uint64_t* mma_done = acc_empty + NACC;
  ItemRing ring;
  ring.q_full = mma_done + 1;
  ring.q_empty = ring.q_full + kQueueSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring.q_empty + kQueueSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  ring.slot = reinterpret_cast<int*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kWgEpiWarps);
    }
    for (int s = 0; s < kQueueSlots; ++s) {
      mbar_init(&ring.q_full[s], 1);
      mbar_init(&ring.q_empty[s], 2 + kWgEpiWarps);  // producer, MMA thread, epilogue warps
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 2) {
    // ------------------------------------------------------------ item scheduler
    if (lane == 0) {
      const int per_group = args.m_tiles * args.n_tiles;
      const int items = args.n_groups * per_group;
      int item = blockIdx.x;
      for (uint32_t lt = 0;; ++lt) {
        const bool have = item < items;
        int v[6] = {-1, 0, 0, 0, 0, 0};
        if (have) {
          const int g = item / per_group, local = item - g * per_group;
          const WgradGroup grp = args.groups[g];
          v[0] = g;
          v[1] = local / args.n_tiles;  // m tile
          v[2] = local - v[1] * args.n_tiles;
          v[3] = grp.ka;
          v[4] = grp.kb;
          v[5] = grp.len;
          item = gridDim.x + atomicAdd(args.queue, 1);
        }
        if (!ring_put(ring, lt, v, args.status, abort_flag) || !have) break;
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0, issued = 0;
      for (uint32_t lt = 0;; ++lt) {
        int v[6];
        if (!ring_take(ring, lt, v, args.status, abort_flag, false) || v[0] < 0) break;
        const int nk = v[5] / BK;
        bool ok = true;
        for (int i = 0; i < nk; ++i, ++it) {
          const uint32_t s = it % STAGES;
          if (it >= STAGES && !xwait(&empty[s], ((it / STAGES) & 1) ^ 1, args.status, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
          tma_load_2d(sA + s * A_BYTES, &tmA, v[3] + i * BK, v[1] * BM, &full[s]);
          tma_load_2d(sB + s * B_BYTES, &tmB, v[4] + i * BK, v[2] * BN, &full[s]);
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
      constexpr uint32_t idesc = idesc_make(1u, BM, BN);
      uint32_t it = 0;
      bool ok = true;
      for (uint32_t lt = 0; ok; ++lt) {
        int v[6];
        if (!ring_take(ring, lt, v, args.status, abort_flag, false)) {
          ok = false;
          break;
        }
        if (v[0] < 0) break;
        const int nk = v[5] / BK;
        const uint32_t b = lt % NACC, u = lt / NACC;
        if (u > 0) ok = xwait(&acc_empty[b], (u & 1) ^ 1, args.status, abort_flag);
        const uint32_t acc = tmem_base + b * BN;
        for (int i = 0; i < nk && ok; ++i, ++it) {
          const uint32_t s = it % STAGES;
          ok = xwait(&full[s], (it / STAGES) & 1, args.status, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16(acc, sdesc_k128(a0 + k * 32), sdesc_k128(b0 + k * 32), idesc, (i > 0 || k > 0) ? 1u : 0u);
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&acc_full[b]);  // with no tokens: arrives at once, the epilogue writes zeros
      }
      if (!ok) *abort_flag = 1;
      mma_commit(mma_done);  // every MMA of this CTA has completed before TMEM is released
      mbar_wait(mma_done, 0, args.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 3..6)
    const int ew = warp - 3;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    uint8_t* box0 = sOut + ew * 2 * kWgBoxBytes;
    uint32_t nstore = 0;
    bool ok = true;
    for (uint32_t lt = 0;; ++lt) {
      int v[6];
      if (!ring_take(ring, lt, v, args.status, abort_flag, true)) {
        ok = false;
        break;
      }
      if (v[0] < 0) break;
      const bool has_k = v[5] >= BK;
      const uint32_t b = lt % NACC, u = lt / NACC;
      ok = __all_sync(0xffffffffu, xwait(&acc_full[b], u & 1, args.status, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const int y = v[1] * BM + quarter * 32;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c, ++nstore) {
        float r[32];
        if (has_k) {
          tmem_ld32(t_lane + b * BN + c * 32, r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0.0f;
        }
        if (c == BN / 32 - 1) {  // the accumulator is in registers: the MMA may refill it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
        uint8_t* box = box0 + (nstore & 1) * kWgBoxBytes;
        if (lane == 0) bulk_wait_read<1>();  // the store that last used this box has read it
        __syncwarp();
        // row `lane` of the box; 16-byte chunk j sits at chunk j ^ (row % 8) (128-byte swizzle)
        uint4* row = reinterpret_cast<uint4*>(box + lane * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          row[j ^ (lane & 7)] = make_uint4(__float_as_uint(r[4 * j]), __float_as_uint(r[4 * j + 1]),
                                           __float_as_uint(r[4 * j + 2]), __float_as_uint(r[4 * j + 3]));
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tmOut, box, v[2] * BN + c * 32, y, v[0]);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait<0>();  // every store of this warp is complete before the CTA exits
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
