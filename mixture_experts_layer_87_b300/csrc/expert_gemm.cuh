// Persistent grouped bf16 expert GEMM on the tcgen05 tensor cores (sm_103a),
// weights as the 128-row MMA operand ("swap AB").
//
//   out[tokens of group g, features] = epilogue( X[tokens of g] . W_g^T )
//
// X is [rows, K] (K-major: permuted tokens, or h), W_g is [Nw, K] (K-major,
// nn.Linear layout).  The MMA computes D[feature, token] = W . X^T, so the
// features of a 256-row weight block sit on the TMEM lanes (two 128-lane
// halves, two MMAs per K step) and the tokens of a chunk on the TMEM columns.
// A group's token count therefore only has to be rounded up to the MMA's N
// granularity (16), not to a 128-row tile: an expert with 300 tokens costs
// chunks of N = 128, 128 and 48, where 128-row tiles would have computed 384
// rows.  Routed experts (ai.flicky.cc 2.1.2: a dropless, uneven number of
// tokens per expert) are exactly the case where that padding adds up.
//
// Work item = (group g, weight block fb of 256 rows, token chunk c of CH
// rows), chunks fastest so the items sharing one weight block run together
// and the block leaves HBM once.  One CTA per SM; items are handed out
// dynamically (the item ring below), so SMs that drew cheap items (short
// chunks) take more of them.  The shared-memory ring and the TMEM buffers
// carry on from one item to the next, so the loads of the next item overlap
// the epilogue of the current one.  Two shapes (XShape): narrow, CH = 128
// tokens with two TMEM buffers of 2 x 128 columns (the epilogue of item i
// overlaps the MMAs of item i + 1); wide, CH = 256 with one buffer of
// 2 x 256 columns and one weight stage feeding twice the MMAs.
//
// Warp roles: warp 0 issues the TMA loads, one thread of warp 1 issues the
// MMAs (kind::f16, K = 16; warp 1 also owns the TMEM allocation), warps 2..9
// drain the accumulators, warp 10 fetches and decodes the items.
//
// Epilogues: BF16 stores y as bf16; SWIGLU pairs gate feature f (half 0) with
// up feature f (half 1) -- the w13 interleave puts both in one weight block --
// and stores h = SiLU(gate) * up as bf16.
#pragma once

#include <cuda_bf16.h>

#include "gemm.cuh"
#include "ptx.cuh"

namespace moe {

struct XGemmArgs {
  // groups: a device table (routed experts: GroupEntry.mt_start counts CH-row
  // chunks) with the total chunk count in *ch_total, or (groups == nullptr)
  // n_groups uniform groups of uni_m rows.
  const GroupEntry* groups;
  const int32_t* ch_total;
  const int32_t* chunk_group;  // [*ch_total]: group of every chunk
  int32_t n_groups;
  int32_t uni_m, uni_a_step, uni_out_step;
  int32_t Nw, K;        // weight rows (output features) per group; reduction length
  int32_t x_rows;       // rows allocated in X
  void* out;            // bf16 [.., out_ld]
  int64_t out_ld;
  int* queue;           // item counter, zero at launch
  int* status;
#ifdef MOE_CHECK
  int64_t w_rows;       // rows of the weight tensor (range-checked build only)
  int32_t out_rows;     // rows allocated in out (range-checked build only)
#endif
};

// ---------------------------------------------------------------------------
// Helpers shared with the FP8 expert GEMM.

// Bounded wait that also gives up as soon as another role of the CTA has
// aborted (so a fault never turns into seconds of waiting per remaining item).
__device__ __forceinline__ bool xwait(uint64_t* bar, uint32_t parity, int* status, volatile int* abort_flag) {
#pragma unroll 1
  for (int i = 0; i < 256; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_status(status, ST_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// Barrier of `count` warps (one arrival per warp, mbarrier initialised with
// that count), bounded and abort-aware.  `phase` counts this warp's uses.
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& phase, int* status, volatile int* abort_flag) {
  __threadfence_block();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = __all_sync(0xffffffffu, xwait(bar, phase & 1, status, abort_flag));
  ++phase;
  return ok;
}

// Item ring: the scheduler warp takes items (first blockIdx.x, then
// gridDim.x + an atomic counter), decodes them and publishes the six
// coordinates in a ring of kQueueSlots shared-memory slots; the producer, the
// MMA thread and every epilogue warp read each slot once (q_empty counts
// their arrivals).  A slot whose first coordinate is -1 ends the item stream.
constexpr int kQueueSlots = 4;

struct ItemRing {
  int* slot;          // [kQueueSlots][8]
  uint64_t* q_full;   // [kQueueSlots], one arrival (the scheduler)
  uint64_t* q_empty;  // [kQueueSlots], one arrival per consumer
};

// Consumer side: wait for item lt, copy its coordinates, release the slot.
// whole_warp: the calling warp reads together and arrives once (lane 0);
// otherwise one thread reads and arrives.
__device__ __forceinline__ bool ring_take(const ItemRing& r, uint32_t lt, int (&v)[6], int* status,
                                          volatile int* abort_flag, bool whole_warp) {
  const uint32_t s = lt % kQueueSlots;
  bool ok = xwait(&r.q_full[s], (lt / kQueueSlots) & 1, status, abort_flag);
  if (whole_warp) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return false;
  const volatile int* src = r.slot + s * 8;
#pragma unroll
  for (int i = 0; i < 6; ++i) v[i] = src[i];
  if (whole_warp) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&r.q_empty[s]);
  } else {
    mbar_arrive(&r.q_empty[s]);
  }
  return true;
}

// Scheduler side (one thread): publish item lt (v[0] = -1: end of stream).
__device__ __forceinline__ bool ring_put(const ItemRing& r, uint32_t lt, const int (&v)[6], int* status,
                                         volatile int* abort_flag) {
  const uint32_t s = lt % kQueueSlots;
  if (lt >= kQueueSlots && !xwait(&r.q_empty[s], ((lt / kQueueSlots) & 1) ^ 1, status, abort_flag)) return false;
  volatile int* dst = r.slot + s * 8;
#pragma unroll
  for (int i = 0; i < 6; ++i) dst[i] = v[i];
  mbar_arrive(&r.q_full[s]);  // release: the coordinates are visible to whoever completes the wait
  return true;
}

// ---------------------------------------------------------------------------
constexpr int kXChunk = 128;   // token rows per chunk of the group tables (plan_kernel)
constexpr int kXEpiWarps = 8;
constexpr int kXThreads = 32 * (3 + kXEpiWarps);
constexpr uint32_t kXABytes = 256 * 128;      // weight tile per stage (256 rows x 128 bytes of K)

// Two shapes of the kernel.  Narrow: an item is one chunk of <= 128 tokens,
// 4 operand stages, two TMEM accumulator buffers (the epilogue of an item
// overlaps the MMAs of the next).  Wide: an item is two consecutive chunks
// of a group (<= 256 tokens, N up to 256), so each weight stage feeds twice
// the MMA work; 3 stages of 64 KB and one TMEM buffer of 2 x 256 columns.
// Which is faster depends on the GEMM (measured per launch site).
template <bool WIDE>
struct XShape {
  static constexpr int CH = WIDE ? 2 * kXChunk : kXChunk;  // token rows per item
  static constexpr int STAGES = WIDE ? 3 : 4;
  static constexpr int NACC = WIDE ? 1 : 2;
  static constexpr uint32_t B_BYTES = CH * 128;  // token tile per stage
};

template <bool WIDE>
constexpr size_t xgemm_smem_bytes() {
  return 1024 + size_t(XShape<WIDE>::STAGES) * (kXABytes + XShape<WIDE>::B_BYTES) + 512 /* barriers + item ring */;
}

struct XTile {
  int32_t g, fb, c, a_row, out_row, n_valid;  // n_valid 0: no work (the odd chunk of a wide pair)
};

// Items of the launch: n_groups uniform groups of CH-row items, or (table)
// *ch_total chunks, each times the nb weight blocks.
template <bool WIDE>
__device__ __forceinline__ int xitems(const XGemmArgs& a, int nb) {
  constexpr int ch = XShape<WIDE>::CH;
  if (a.groups == nullptr) return (a.uni_m + ch - 1) / ch * nb * a.n_groups;
  return __ldg(a.ch_total) * nb;
}

// Item `tile` -> (expert weights, weight block, chunk).  Items are ordered
// group by group, and inside a group weight block by weight block with the
// chunks fastest, so group g owns items [mt_start_g * nb, (mt_start_g +
// nch_g) * nb) and chunk_group[tile / nb] names its group (low 16 bits) and
// the expert whose weights the group uses (high 16 bits; plan_kernel fills
// both): two dependent loads per item.  The wide kernel keeps the table's
// 128-row chunks: an even chunk takes the odd one after it as well (up to
// 256 rows), and the odd chunk's item does nothing (n_valid 0).
template <bool WIDE>
__device__ __forceinline__ bool xdecode(const XGemmArgs& a, int tile, int items, int nb, XTile& t) {
  constexpr int ch = XShape<WIDE>::CH;
  if (tile >= items) return false;
  if (a.groups == nullptr) {
    const int nch = (a.uni_m + ch - 1) / ch;
    const int per_group = nch * nb;
    t.g = tile / per_group;
    const int local = tile - t.g * per_group;
    t.fb = local / nch;
    t.c = local - t.fb * nch;
    t.a_row = t.g * a.uni_a_step + t.c * ch;
    t.out_row = t.g * a.uni_out_step + t.c * ch;
    t.n_valid = min(ch, a.uni_m - t.c * ch);
    return true;
  }
  const int cg = __ldg(a.chunk_group + tile / nb);
  const int4 G = __ldg(reinterpret_cast<const int4*>(a.groups) + (cg & 0xFFFF));  // {a_row0, out_row0, m, mt_start}
  const int nch = (G.z + kXChunk - 1) / kXChunk;
  const int local = tile - G.w * nb;
  t.g = cg >> 16;  // the weights' expert
  t.fb = local / nch;
  t.c = local - t.fb * nch;
  t.a_row = G.x + t.c * kXChunk;
  t.out_row = G.y + t.c * kXChunk;
  t.n_valid = (WIDE && (t.c & 1)) ? 0 : min(ch, G.z - t.c * kXChunk);
  return true;
}

template <Epi EPI, bool WIDE>
__global__ void __launch_bounds__(kXThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const XGemmArgs args) {
  using S = XShape<WIDE>;
  constexpr int CH = S::CH, BK = 64, STAGES = S::STAGES, NACC = S::NACC;
  constexpr uint32_t A_BYTES = kXABytes, B_BYTES = S::B_BYTES;
  constexpr uint32_t BUF_COLS = 2 * CH;  // one accumulator buffer: half 0 | half 1
  constexpr uint32_t TMEM_COLS = NACC * BUF_COLS;
  static_assert(TMEM_COLS == 512, "TMEM budget");
  static_assert(EPI == Epi::SWIGLU || EPI == Epi::BF16, "expert epilogues");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
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
  const int nb = (args.Nw + 255) / 256;
  const int num_kb = args.K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kXEpiWarps);
    }
    for (int s = 0; s < kQueueSlots; ++s) {
      mbar_init(&ring.q_full[s], 1);
      mbar_init(&ring.q_empty[s], 2 + kXEpiWarps);  // producer, MMA thread, epilogue warps
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 10) {
    // ------------------------------------------------------------ item scheduler
    if (lane == 0) {
      const int items = xitems<WIDE>(args, nb);
      int item = blockIdx.x;
      for (uint32_t lt = 0;; ++lt) {
        XTile t{-1, 0, 0, 0, 0, 0};
        bool have;
        do {  // items with nothing to do (wide: odd chunks) are passed over
          have = xdecode<WIDE>(args, item, items, nb, t);
          if (have) item = gridDim.x + atomicAdd(args.queue, 1);  // the next one, while this one is published
        } while (have && t.n_valid <= 0);
        const int v[6] = {have ? t.g : -1, t.fb, t.c, t.a_row, t.out_row, t.n_valid};
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
        const int w_row = v[0] * args.Nw + v[1] * 256, a_row = v[3];
        // TMA fills rows past a tensor's end with zeros; a tile that starts
        // outside its tensor is still a wrong coordinate
        (void)MOE_IN_RANGE(args.status, w_row, args.w_rows);
        (void)MOE_IN_RANGE(args.status, a_row, args.x_rows);
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const uint32_t s = it % STAGES;
          if (it >= STAGES && !xwait(&empty[s], ((it / STAGES) & 1) ^ 1, args.status, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
          tma_load_2d(sA + s * A_BYTES, &tmW, kb * BK, w_row, &full[s]);
          tma_load_2d(sB + s * B_BYTES, &tmX, kb * BK, a_row, &full[s]);
          issued = it + 1;
        }
        if (!ok) break;
      }
      // Abnormal exit only: copies still in flight must land before the CTA
      // may leave (normally the MMA thread has consumed every one of them).
      if (*abort_flag)
        for (uint32_t j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
          mbar_wait(&full[j % STAGES], (j / STAGES) & 1, args.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (uint32_t lt = 0; ok; ++lt) {
        int v[6];
        if (!ring_take(ring, lt, v, args.status, abort_flag, false)) {
          ok = false;
          break;
        }
        if (v[0] < 0) break;
        const uint32_t n_mma = (static_cast<uint32_t>(v[5]) + 15u) & ~15u;  // tokens rounded up to N % 16
        const uint32_t idesc = idesc_make(1u, 128, static_cast<int>(n_mma));
        const uint32_t b = lt % NACC, u = lt / NACC;
        if (u > 0) ok = xwait(&acc_empty[b], (u & 1) ^ 1, args.status, abort_flag);
        const uint32_t acc_col = b * BUF_COLS;
        for (int kb = 0; kb < num_kb && ok; ++kb, ++it) {
          const uint32_t s = it % STAGES;
          ok = xwait(&full[s], (it / STAGES) & 1, args.status, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad0 = sdesc_k128(a0 + k * 32), ad1 = sdesc_k128(a0 + 128 * 128 + k * 32);
            const uint64_t bd = sdesc_k128(b0 + k * 32);
            const uint32_t accumulate = (kb > 0 || k > 0) ? 1u : 0u;
            mma_bf16(tmem_base + acc_col, ad0, bd, idesc, accumulate);
            mma_bf16(tmem_base + acc_col + CH, ad1, bd, idesc, accumulate);
          }
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&acc_full[b]);
      }
      if (!ok) *abort_flag = 1;
      // every MMA of this CTA has completed before TMEM is released
      mma_commit(mma_done);
      mbar_wait(mma_done, 0, args.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    const int ew = warp - 2;
    const int q = warp & 3;    // TMEM lane quarter this warp may access
    const int hg = ew >> 2;    // token half of the chunk
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    constexpr int TOK = CH / 2;  // tokens per warp group
    bool ok = true;
    for (uint32_t lt = 0;; ++lt) {
      int v[6];
      if (!ring_take(ring, lt, v, args.status, abort_flag, true)) {
        ok = false;
        break;
      }
      if (v[0] < 0) break;
      const int fb = v[1], out_row = v[4], n_valid = v[5];
      const int tok_lo = hg * TOK;
      // the item's output rows lie inside out (range-checked build; else skipped)
      const bool rows_ok = MOE_IN_RANGE(args.status, out_row, args.out_rows) &&
                           MOE_IN_RANGE(args.status, out_row + max(n_valid, 1) - 1, args.out_rows);
      const int tok_n = rows_ok ? max(0, min(TOK, n_valid - tok_lo)) : 0;  // valid tokens of my half
      const uint32_t b = lt % NACC, u = lt / NACC;
      ok = __all_sync(0xffffffffu, xwait(&acc_full[b], u & 1, args.status, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t col0 = t_lane + b * BUF_COLS + tok_lo;
      if constexpr (EPI == Epi::SWIGLU) {
        const int f = fb * 128 + q * 32 + lane;  // feature of h (I = Nw / 2)
        __nv_bfloat16* h = static_cast<__nv_bfloat16*>(args.out) + (int64_t)(out_row + tok_lo) * args.out_ld + f;
#pragma unroll 1
        for (int j = 0; j * 32 < tok_n; ++j) {
          float g[32], up[32];
          tmem_ld32(col0 + j * 32, g);
          tmem_ld32(col0 + CH + j * 32, up);
          const int nv = min(32, tok_n - j * 32);
          __nv_bfloat16* p = h + (int64_t)(j * 32) * args.out_ld;
#pragma unroll
          for (int i = 0; i < 32; ++i, p += args.out_ld)
            if (i < nv) *p = __float2bfloat16_rn(silu(g[i]) * up[i]);
        }
      } else {
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          const int f = fb * 256 + half * 128 + q * 32 + lane;
          const bool f_ok = f < args.Nw;
          __nv_bfloat16* y = static_cast<__nv_bfloat16*>(args.out) + (int64_t)(out_row + tok_lo) * args.out_ld + f;
#pragma unroll 1
          for (int j = 0; j * 32 < tok_n; ++j) {
            float vv[32];
            tmem_ld32(col0 + half * CH + j * 32, vv);
            const int nv = f_ok ? min(32, tok_n - j * 32) : 0;
            __nv_bfloat16* p = y + (int64_t)(j * 32) * args.out_ld;
#pragma unroll
            for (int i = 0; i < 32; ++i, p += args.out_ld)
              if (i < nv) *p = __float2bfloat16_rn(vv[i]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
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
