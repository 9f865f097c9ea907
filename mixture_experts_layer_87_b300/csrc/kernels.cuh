// Bandwidth- and latency-bound kernels of the layer: top-k routing, the
// dropless dispatch (histogram, scan, stable scatter, row gather with fused
// FP8 activation quantisation), the combine, the bias update and the offline
// weight helpers.  None of them waits on anything, so none can hang.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <climits>
#include <float.h>

#include "gemm.cuh"
#include "ptx.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Router top-k (ai.flicky.cc 2.1.2, the g'_{i,t} rule; xyznot.com Method 2).
// One warp per token.  Lane l holds experts l, l+32, ... (VPL of them):
// z = the sum of the logits GEMM's K splits in split order, s = sigmoid(z),
// score = s + b.  k rounds of a warp arg-max (score
// descending, ties to the lower index) pick the experts; the gates are the
// selected unbiased s divided by their sum.  Lane j keeps the j-th pick.
// A NaN score ranks as -inf.
// Node limit (the same section: a token is sent to at most 4 nodes): with
// group_size > 0 the experts sit on nodes of group_size consecutive experts,
// and once group_limit nodes are in use the arg-max only looks at experts on
// those nodes -- the k best experts on the group_limit nodes whose best expert
// scores highest.
template <int VPL>
__global__ void __launch_bounds__(256, 1) route_topk_kernel(const float* __restrict__ z, int splits,
                                                         int64_t split_stride, int T, int E, int k,
                                                         const float* __restrict__ bias, int32_t* __restrict__ idx_out,
                                                         float* __restrict__ gate_out, int32_t* __restrict__ counts,
                                                         uint32_t* __restrict__ mask, int W, int group_size,
                                                         int group_limit, int* status) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float sc[VPL], sv[VPL];
  uint32_t taken = 0;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    if (e < E) {
      float zz = z[(int64_t)t * E + e];
      for (int p = 1; p < splits; ++p) zz += z[p * split_stride + (int64_t)t * E + e];
      const float s = 1.0f / (1.0f + expf(-zz));
      float score = s + bias[e];
      if (isnan(score)) score = -INFINITY;
      sc[j] = score;
      sv[j] = s;
    } else {
      sc[j] = -INFINITY;
      sv[j] = 0.0f;
      taken |= 1u << j;  // not an expert
    }
  }
  int my_idx = -1;
  float my_s = 0.0f;
  uint32_t nodes = 0;           // nodes in use (group_size > 0; at most 32 nodes)
  uint32_t allowed = ~0u;       // bit j: expert lane + 32 j may still be picked
  bool restricted = false;
  for (int r = 0; r < k; ++r) {
    float best = -INFINITY, bs = 0.0f;
    int bi = INT_MAX;
    if (group_size > 0 && !restricted && __popc(nodes) >= group_limit) {
      // the node budget is spent: from now on only experts on the used nodes
      // (the set of nodes cannot change any more)
      restricted = true;
      allowed = 0;
#pragma unroll 1
      for (int j = 0; j < VPL; ++j) {
        const int e = lane + 32 * j;
        if (e < E && ((nodes >> (e / group_size)) & 1u)) allowed |= 1u << j;
      }
    }
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      if (!(((taken | ~allowed) >> j) & 1u) && (sc[j] > best || (sc[j] == best && e < bi))) {
        best = sc[j];
        bi = e;
        bs = sv[j];
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      const float os = __shfl_xor_sync(0xffffffffu, bs, off);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
        bs = os;
      }
    }
    if (bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (group_size > 0 && bi < E) nodes |= 1u << (bi / group_size);  // bi is the same in every lane
    if (lane == r) {
      my_idx = bi;
      my_s = bs;
    }
  }
  float sum = lane < k ? my_s : 0.0f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  float gate = lane < k ? my_s / sum : 0.0f;
  if (!(sum >= FLT_MIN)) {
    // Every selected affinity underflowed (all their logits below about -87):
    // s_j / sum_j' s_j' is still well defined, so take it in the log domain,
    // g_j = exp(log s_j - m) / sum_j' exp(log s_j' - m), m = max log s, with
    // log s = z - log(1 + e^z) from the selected expert's logit.  (sum is
    // warp-uniform, so the whole warp takes this branch.)
    float ls = -INFINITY;
    if (lane < k && my_idx >= 0 && my_idx < E) {
      float zz = z[(int64_t)t * E + my_idx];
      for (int p = 1; p < splits; ++p) zz += z[p * split_stride + (int64_t)t * E + my_idx];
      ls = zz < 0.0f ? zz - log1pf(expf(zz)) : -log1pf(expf(-zz));
    }
    float m = ls;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float w = lane < k ? expf(ls - m) : 0.0f;
    float wsum = w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    gate = w / wsum;
  }
  if (lane < k) {
    idx_out[(int64_t)t * k + lane] = my_idx;
    gate_out[(int64_t)t * k + lane] = gate;
    if (MOE_IN_RANGE(status, my_idx, E)) {
      atomicAdd(&counts[my_idx], 1);
      if (mask) atomicOr(&mask[(int64_t)my_idx * W + (t >> 5)], 1u << (t & 31));
    }
  }
}

// ---------------------------------------------------------------------------
// Dispatch layout.  mask[e][w] bit b says token 32w+b chose expert e, so the
// rank of token t among expert e's tokens is the popcount of the mask bits
// before it: a stable, deterministic counting sort with no sort at all.

// Token-expert bitmask from a [T, k] selection (moe_permute's own path; the
// router kernel writes the same bits directly inside moe_forward).
__global__ void build_mask_kernel(const int32_t* __restrict__ idx, int64_t n, int k, int E, uint32_t* mask, int W,
                                  int* status) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int e = idx[i];
  const int64_t t = i / k;
  if (e < 0 || e >= E) {
    record_status(status, ST_BAD_INDEX);
    return;
  }
  atomicOr(&mask[(int64_t)e * W + (t >> 5)], 1u << (t & 31));
}

// Block-wide exclusive scan (blockDim.x threads, multiple of 32, <= 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    if (lane < nw) warp_sums[lane] = s;  // inclusive
  }
  __syncthreads();
  const int warp_prefix = wid > 0 ? warp_sums[wid - 1] : 0;
  total = warp_sums[nw - 1];
  __syncthreads();
  return warp_prefix + x - v;
}

// One block per expert: exclusive prefix of mask-word popcounts (wprefix)
// and the expert's row count (cnt).
__global__ void __launch_bounds__(256) expert_scan_kernel(const uint32_t* __restrict__ mask, int W,
                                                          int32_t* __restrict__ wprefix, int32_t* __restrict__ cnt) {
  __shared__ int warp_sums[32];
  const int e = blockIdx.x;
  int carry = 0;
  for (int base = 0; base < W; base += blockDim.x) {
    const int w = base + threadIdx.x;
    const int v = w < W ? __popc(mask[(int64_t)e * W + w]) : 0;
    int total;
    const int ex = block_exclusive_scan(v, warp_sums, total);
    if (w < W) wprefix[(int64_t)e * W + w] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) cnt[e] = carry;
}

// One block (1024 threads): row offsets of the experts and the GEMM group
// table (chunks of `chunk` rows per expert, prefix of chunks).  With
// offs_in != nullptr the counts come from untrusted offsets
// (moe_grouped_ffn): they are made non-decreasing and clipped to
// [0, clamp_rows], flagging any repair.
// chunk_group (optional, cg_cap entries) receives, for every chunk, its group
// g in the low 16 bits and the expert whose weights the group uses in the
// high 16 bits -- group_weight[g] (checked against n_weights: an entry
// outside [0, n_weights) is flagged and replaced by 0), or g when group_weight
// is nullptr -- so a GEMM maps a chunk index to both with one load.  G <= 65535.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ cnt, const int32_t* __restrict__ offs_in,
                                                    int G, int clamp_rows, int chunk, int32_t* __restrict__ offsets_out,
                                                    GroupEntry* __restrict__ groups, int32_t* __restrict__ mt_total,
                                                    int32_t* __restrict__ chunk_group, int cg_cap,
                                                    const int32_t* __restrict__ group_weight, int n_weights,
                                                    int* status) {
  __shared__ int warp_sums[32];
  __shared__ int carry_rows, carry_mt;
  if (threadIdx.x == 0) {
    carry_rows = 0;
    carry_mt = 0;
  }
  __syncthreads();
  for (int base = 0; base < G; base += blockDim.x) {
    const int g = base + threadIdx.x;
    int rows = 0, a0 = 0;
    if (g < G) {
      if (offs_in) {
        int lo = offs_in[g], hi = offs_in[g + 1];
        const int clo = min(max(lo, 0), clamp_rows), chi = min(max(hi, clo), clamp_rows);
        if (clo != lo || chi != hi || (g == 0 && lo != 0)) record_status(status, ST_BAD_INDEX);
        a0 = clo;
        rows = chi - clo;
      } else {
        rows = cnt[g];
      }
    }
    const int mt = (rows + chunk - 1) / chunk;
    int tot_rows, tot_mt;
    const int ex_rows = block_exclusive_scan(rows, warp_sums, tot_rows);
    const int ex_mt = block_exclusive_scan(mt, warp_sums, tot_mt);
    if (g < G) {
      const int off = offs_in ? a0 : carry_rows + ex_rows;
      if (offsets_out) offsets_out[g] = off;
      groups[g] = GroupEntry{off, off, rows, carry_mt + ex_mt};
      if (chunk_group) {
        int w = g;
        if (group_weight) {
          w = group_weight[g];
          if (w < 0 || w >= n_weights || w > 0xFFFF) {
            record_status(status, ST_BAD_INDEX);
            w = 0;
          }
        }
        for (int j = carry_mt + ex_mt; j < carry_mt + ex_mt + mt && j < cg_cap; ++j) chunk_group[j] = g | (w << 16);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry_rows += tot_rows;
      carry_mt += tot_mt;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (offsets_out) offsets_out[G] = carry_rows;
    if (chunk_group && carry_mt > cg_cap) record_status(status, ST_BAD_INDEX);  // overlapping untrusted offsets
    *mt_total = chunk_group ? min(carry_mt, cg_cap) : carry_mt;
  }
}

// 8 bf16 (16 bytes) -> 8 fp32
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = __bfloat1622float2(h[i]);
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}

// One warp per token: the slot of every (t, j) pair, perm, and the row
// gather x_perm[slot] = u[t].  FP8: u is quantised once per 1 x 128 tile
// (scale = amax/448, codes = RNE-saturated E4M3 of u/scale, ai.flicky.cc 3.3
// item 2) and the codes are copied to every slot; uq/uq_scale (optional)
// receive the token's own quantised row for the shared experts.  With
// gridDim.y > 1 the row is split into gridDim.y column ranges (more warps for
// few tokens); every split recomputes the token's slots, split 0 writes them.
template <bool FP8>
__global__ void __launch_bounds__(256) dispatch_kernel(
    const int32_t* __restrict__ idx, int T, int k, int E, const uint32_t* __restrict__ mask,
    const int32_t* __restrict__ wprefix, int W, const int32_t* __restrict__ offsets, int32_t* __restrict__ slot,
    int32_t* __restrict__ perm, const __nv_bfloat16* __restrict__ u, int d, void* __restrict__ x_perm,
    float* __restrict__ x_scale, int64_t rows, uint8_t* __restrict__ uq, float* __restrict__ uq_scale, int* status,
    bool pow2) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int my_slot = -1;
  if (lane < k) {
    const int e = idx[(int64_t)t * k + lane];
    if (e >= 0 && e < E) {
      const int w = t >> 5, b = t & 31;
      const int rank = wprefix[(int64_t)e * W + w] + __popc(mask[(int64_t)e * W + w] & ((1u << b) - 1u));
      my_slot = offsets[e] + rank;
      if (!MOE_IN_RANGE(status, my_slot, rows)) my_slot = -1;
      if (blockIdx.y == 0) {
        slot[(int64_t)t * k + lane] = my_slot;
        if (my_slot >= 0) perm[my_slot] = t;
      }
    } else if (blockIdx.y == 0) {
      slot[(int64_t)t * k + lane] = -1;
    }
  }
  const int split = blockIdx.y, n_split = gridDim.y;
  const uint4* src = reinterpret_cast<const uint4*>(u + (int64_t)t * d);
  if constexpr (!FP8) {
    uint4* dst = reinterpret_cast<uint4*>(x_perm);
    const int nc = d / 8;
    // every lane runs every iteration (the shuffles need the whole warp);
    // lanes past the row's last 16-byte chunk only skip the copy
    for (int c0 = 32 * split; c0 < nc; c0 += 32 * n_split) {
      const int c = c0 + lane;
      const bool act = c < nc;
      const uint4 v = act ? src[c] : make_uint4(0, 0, 0, 0);
      for (int j = 0; j < k; ++j) {
        const int s = __shfl_sync(0xffffffffu, my_slot, j);
        if (act && s >= 0) dst[(int64_t)s * nc + c] = v;
      }
    }
  } else {
    // A quarter-warp (8 lanes) per 128-wide tile, 16 elements per lane: a
    // lane reads 32 contiguous bytes of u and writes its 16 codes with one
    // 16-byte store per destination row (a warp: 512 contiguous bytes).
    const int groups = d / 128;
    const int ql = lane & 7, qw = lane >> 3;
    for (int g0 = 4 * split; g0 < groups; g0 += 4 * n_split) {
      const int g = g0 + qw;
      const bool active = g < groups;
      float f0[8], f1[8];
      float amax = 0.0f;
      if (active) {
        unpack8(src[g * 16 + 2 * ql], f0);
        unpack8(src[g * 16 + 2 * ql + 1], f1);
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(f0[i]), fabsf(f1[i])));
      }
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
      if (pow2) scale = pow2_ceil(scale);  // UE8M0 scales
      uint4 code = make_uint4(0, 0, 0, 0);
      if (active) {
        uint32_t c8[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          c8[i] = e4m3x2(f0[2 * i] / scale, f0[2 * i + 1] / scale);
          c8[4 + i] = e4m3x2(f1[2 * i] / scale, f1[2 * i + 1] / scale);
        }
        code = make_uint4(c8[0] | (c8[1] << 16), c8[2] | (c8[3] << 16), c8[4] | (c8[5] << 16), c8[6] | (c8[7] << 16));
        if (uq) {
          reinterpret_cast<uint4*>(uq + (int64_t)t * d + g * 128)[ql] = code;
          if (ql == 0) uq_scale[(int64_t)g * T + t] = scale;
        }
      }
      for (int j = 0; j < k; ++j) {
        const int s = __shfl_sync(0xffffffffu, my_slot, j);
        if (active && s >= 0) {
          reinterpret_cast<uint4*>(static_cast<uint8_t*>(x_perm) + (int64_t)s * d + g * 128)[ql] = code;
          if (ql == 0) x_scale[(int64_t)g * rows + s] = scale;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Combine (ai.flicky.cc 2.1.2, the h'_t equation):
//   out_t = u_t + sum_s shared_y[s,t] + sum_j gate[t,j] * y[slot[t,j]]
// fp32 in this fixed order, one rounding to bf16.  One block per token (per
// token and column range when gridDim.y > 1, for few tokens), 16 bytes (8
// features) per thread per step.  Slots outside [0, rows) are skipped (and
// flagged).
__global__ void __launch_bounds__(128) combine_kernel(const __nv_bfloat16* __restrict__ u,
                                                      const __nv_bfloat16* __restrict__ ysh, int n_shared,
                                                      const __nv_bfloat16* __restrict__ y,
                                                      const int32_t* __restrict__ slot,
                                                      const float* __restrict__ gate, int T, int d, int k,
                                                      int64_t rows, __nv_bfloat16* __restrict__ out, int* status) {
  __shared__ int s_slot[32];
  __shared__ float s_gate[32];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    int s = slot[(int64_t)t * k + threadIdx.x];
    if (s < 0 || s >= rows) {
      record_status(status, ST_BAD_INDEX);
      s = -1;
    }
    s_slot[threadIdx.x] = s;
    s_gate[threadIdx.x] = gate[(int64_t)t * k + threadIdx.x];
  }
  __syncthreads();
  const int nc = d / 8;
  for (int c = blockIdx.y * blockDim.x + threadIdx.x; c < nc; c += gridDim.y * blockDim.x) {
    float acc[8];
    unpack8(reinterpret_cast<const uint4*>(u + (int64_t)t * d)[c], acc);
    for (int s = 0; s < n_shared; ++s) {
      float f[8];
      unpack8(reinterpret_cast<const uint4*>(ysh + ((int64_t)s * T + t) * d)[c], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
    }
    for (int j = 0; j < k; ++j) {
      const int s = s_slot[j];
      if (s < 0) continue;
      const float g = s_gate[j];
      float f[8];
      unpack8(reinterpret_cast<const uint4*>(y + (int64_t)s * d)[c], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, f[i], acc[i]);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(out + (int64_t)t * d)[c] = o;
  }
}

// ---------------------------------------------------------------------------
// Auxiliary-loss-free bias update (ai.flicky.cc 2.1.2; xyznot.com Method 2):
// b_i <- b_i + gamma * sign(T*k/E - load_i), in fp32.
__global__ void bias_update_kernel(int E, int64_t T, int k, const int32_t* __restrict__ counts, float gamma,
                                   float* __restrict__ bias) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= E) return;
  const float mean = (float)(T * k) / (float)E;
  const float load = (float)counts[i];
  const float sgn = mean > load ? 1.0f : (mean < load ? -1.0f : 0.0f);
  bias[i] = bias[i] + gamma * sgn;
}

// ---------------------------------------------------------------------------
// Offline: 128 x 128 block quantisation of bf16 weights to E4M3 (ai.flicky.cc
// 3.3 item 2).  One block of 256 threads per 128 x 128 block.  pow2: UE8M0
// scales (amax/448 rounded up to a power of two).
__global__ void __launch_bounds__(256) quantize_blocks_kernel(const __nv_bfloat16* __restrict__ w, int cols,
                                                              uint8_t* __restrict__ q, float* __restrict__ scale,
                                                              bool pow2) {
  __shared__ float red[8];
  const int bc = blockIdx.x, br = blockIdx.y;
  const int64_t row0 = (int64_t)br * 128;
  float f[8][8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = threadIdx.x + 256 * i;  // chunk of 8 elements: row c/16, cols (c%16)*8
    const int r = c >> 4, c8 = (c & 15) * 8;
    const uint4 v = *reinterpret_cast<const uint4*>(w + (row0 + r) * cols + bc * 128 + c8);
    unpack8(v, f[i]);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[i][j]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  float s = amax > 0.0f ? amax / 448.0f : 1.0f;
  if (pow2) s = pow2_ceil(s);
  if (threadIdx.x == 0) scale[(int64_t)br * (cols / 128) + bc] = s;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = threadIdx.x + 256 * i;
    const int r = c >> 4, c8 = (c & 15) * 8;
    uint2 code;
    code.x = e4m3x2(f[i][0] / s, f[i][1] / s) | (uint32_t(e4m3x2(f[i][2] / s, f[i][3] / s)) << 16);
    code.y = e4m3x2(f[i][4] / s, f[i][5] / s) | (uint32_t(e4m3x2(f[i][6] / s, f[i][7] / s)) << 16);
    *reinterpret_cast<uint2*>(q + (row0 + r) * cols + bc * 128 + c8) = code;
  }
}

// Offline: interleave W1 and W3 ([E, I, d] each) into w13 [E, 2I, d] in
// 128-row blocks (gate block j, then up block j).
__global__ void pack_gate_up_kernel(const uint4* __restrict__ w1, const uint4* __restrict__ w3, int64_t E, int I,
                                    int d, uint4* __restrict__ w13) {
  const int nc = d / 8;
  const int64_t total = E * 2 * I * (int64_t)nc;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int c = i % nc;
    const int64_t row = i / nc;  // row of w13
    const int64_t e = row / (2 * I);
    const int R = row % (2 * I);
    const int j = R / 256, within = R % 256;
    const uint4* src = within < 128 ? w1 : w3;
    const int64_t srow = e * I + 128 * j + (within & 127);
    w13[i] = src[srow * nc + c];
  }
}

// ---------------------------------------------------------------------------
// Redundant experts (ai.flicky.cc 3.5: popular experts are duplicated to even
// out the load).  Expert e has replica_count[e] copies, the physical slots
// replica_first[e] ...; the pair (t, j) goes to copy t mod replica_count[e]:
// idx[t, j] is rewritten in place from the expert to its physical slot and the
// token's bit is set in the slot's row of the dispatch mask.  A bad expert
// index or plan entry is flagged and the pair left out.
__global__ void assign_replicas_kernel(int32_t* __restrict__ idx, int64_t n, int k, int E,
                                       const int32_t* __restrict__ replica_first,
                                       const int32_t* __restrict__ replica_count, int P, uint32_t* __restrict__ mask,
                                       int W, int* status) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int e = idx[i];
  const int64_t t = i / k;
  if (e < 0 || e >= E) {
    record_status(status, ST_BAD_INDEX);
    return;
  }
  const int first = replica_first[e], copies = replica_count[e];
  const int p = copies > 0 ? first + static_cast<int>(t % copies) : -1;
  if (copies <= 0 || first < 0 || p >= P) {
    record_status(status, ST_BAD_INDEX);
    idx[i] = -1;  // dispatch skips it (and flags it again)
    return;
  }
  idx[i] = p;
  atomicOr(&mask[(int64_t)p * W + (t >> 5)], 1u << (t & 31));
}

// Self-test: one warp waits on an mbarrier nothing arrives on; the bounded
// wait gives up after limit_ns, records ST_TIMEOUT and the kernel returns.
__global__ void selftest_timeout_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, status, limit_ns);
  __syncthreads();
}

}  // namespace moe
