// Backward pass of the layer (bf16): the bandwidth-side kernels.  The GEMMs
// are the expert GEMM of expert_gemm.cuh (the forward recompute and the two
// data-gradient products, on transposed weights) and the weight-gradient GEMM
// of wgrad_gemm.cuh.
//
// What is differentiated (the layer equation of ai.flicky.cc 2.1.2,
// xyznot.com Method 2): h'_t = u_t + sum_s FFN_s(u_t) + sum_j g_{t,j}
// FFN_{e_j}(u_t), g = s / sum s, s = sigmoid(u . c), FFN(x) = W2 (SiLU(W1 x) *
// (W3 x)).  The selection is held fixed (the gradient flows through the gate
// values, not through the top-k choice) and the bias, which the pages update
// by a sign rule, gets no gradient.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "gemm.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Columns of the transposed activations for the weight-gradient GEMM: the rows
// of group g (offsets[g] .. offsets[g+1]) become columns pad_off[g] .., every
// group padded to a multiple of `gran` columns (64: one 64-wide K stage of the
// GEMM; 128 in the FP8 scheme, so that 128-token quantisation blocks start at
// every group's first token; the padding is zero).  row_of_col[col] = the row a
// column holds, or -1 for a padding column, for the live columns
// col < pad_off[G] (the columns past it are never read).  One block of 1024
// threads: the padded sizes are prefix-summed across the block (two groups a
// thread, G <= 2048), then each thread finds its columns' groups by bisection.
__global__ void __launch_bounds__(1024) pad_plan_kernel(const int32_t* __restrict__ offsets, int G, int n_cols,
                                                        int gran, int32_t* __restrict__ pad_off,
                                                        int32_t* __restrict__ row_of_col, int* status) {
  __shared__ int s_off[2049];
  __shared__ int s_warp[32];
  if (G > 2048) {  // not used by the library (G <= E + n_shared <= 2048)
    if (threadIdx.x == 0) record_status(status, ST_BAD_INDEX);
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int sz[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int g = 2 * tid + q;
    sz[q] = g < G ? (offsets[g + 1] - offsets[g] + gran - 1) / gran * gran : 0;
  }
  // inclusive scan of the thread's pair sums: within the warp, then across warps
  int incl = sz[0] + sz[1];
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += o;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int excl = incl - (sz[0] + sz[1]) + (warp > 0 ? s_warp[warp - 1] : 0);
  if (2 * tid < G) s_off[2 * tid] = excl;
  if (2 * tid + 1 < G) s_off[2 * tid + 1] = excl + sz[0];
  if (tid == 0) s_off[G] = s_warp[31];  // the padded total
  __syncthreads();
  for (int g = tid; g <= G; g += blockDim.x) pad_off[g] = s_off[g];
  const int live = s_off[G];
  if (tid == 0 && live > n_cols) record_status(status, ST_BAD_INDEX);
  const int end = min(live, n_cols);
  for (int col = tid; col < end; col += blockDim.x) {
    int lo = 0, hi = G;  // g with s_off[g] <= col < s_off[g + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= col) lo = mid;
      else hi = mid;
    }
    const int local = col - s_off[lo];
    row_of_col[col] = local < offsets[lo + 1] - offsets[lo] ? offsets[lo] + local : -1;
  }
}

// Transposed gather, batched over blockIdx.z (src/dst strides per batch):
//   dst[c][col] = f(src[row(col)][c])  for c < C and the live columns col,
// row(col) = perm[row_of_col[col]] when perm is given, else row_of_col[col]
// (-1: a zero column), or col itself while col < rows when row_of_col is null
// (zero beyond).  Live columns: col < n_cols, and col < *n_live when n_live is
// given (the padded total of the groups: the tiles past it are not written,
// since nothing reads them, and the columns past it in the last tile are zero).
//
// f is the identity (FQ = false), or (FQ = true) the FP8 quantisation of the
// weight-gradient operands (1 x 128 tiles along the tokens, ai.flicky.cc 3.3
// items 2 and 4) written back dequantised as bf16:
//   dst[c][col] = bf16( E4M3(x * (1/s)) * s ),  x = src[row(col)][c],
// s = amax/448 over the 128-column block of col (UE8M0: rounded up to a power
// of two; an all-zero block: 1), 1/s one correctly rounded fp32 reciprocal
// per block (the operands are intermediates known to bf16 accuracy; a
// division per element would cost more than the copy).  With power-of-two
// scales the bf16 value is the E4M3 value exactly.
//
// A block owns one 128-column tile (one quantisation block) and walks the c
// range in 64-wide slabs, blockIdx.x, blockIdx.x + gridDim.x, ...: it looks
// up its columns' rows once, and loads the next slab (16-byte loads along the
// src rows, held in registers) while it writes the current one out of shared
// memory (FQ: four lanes per dst row, 16-byte stores; else a warp per dst row,
// 4-byte bf16 pairs).  Needs C % 8 == 0, 16-byte aligned src rows, an even ldd
// and a 4-byte aligned dst; FQ also ldd % 8 == 0 and a 16-byte aligned dst.
template <bool FQ>
__global__ void __launch_bounds__(256, 6) transpose_cols_kernel(
    const __nv_bfloat16* __restrict__ src, int rows, int C, int64_t src_batch, const int32_t* __restrict__ row_of_col,
    const int32_t* __restrict__ perm, int n_cols, const int32_t* __restrict__ n_live, __nv_bfloat16* __restrict__ dst,
    int64_t ldd, int64_t dst_batch, bool pow2) {
  __shared__ __align__(16) uint16_t tile[64][130];  // [c - c0][col - col0]
  const int col0 = blockIdx.y * 128;
  const int live = n_live ? min(*n_live, n_cols) : n_cols;
  if (col0 >= live) return;
  src += blockIdx.z * src_batch;
  dst += blockIdx.z * dst_batch;
  const int tid = threadIdx.x, chunk = tid & 7;  // chunk: 8 c values of a src row
  int row[4];                                     // src rows of my 4 columns, -1: zero column
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int col = col0 + (tid >> 3) + 32 * i;
    int r = -1;
    if (col < live) {
      r = row_of_col ? row_of_col[col] : (col < rows ? col : -1);
      if (r >= 0 && perm) r = perm[r];
    }
    row[i] = r >= 0 && r < rows ? r : -1;
  }
  const int n_slab = (C + 63) >> 6;
  uint4 v[4];
  auto fetch = [&](int slab) {
    const int c = slab * 64 + chunk * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      v[i] = row[i] >= 0 && c < C ? *reinterpret_cast<const uint4*>(src + (int64_t)row[i] * C + c)
                                  : make_uint4(0, 0, 0, 0);
  };
  int slab = blockIdx.x;
  if (slab < n_slab) fetch(slab);
  const int warp = tid >> 5, lane = tid & 31;
  for (; slab < n_slab; slab += gridDim.x) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t* e = reinterpret_cast<const uint16_t*>(&v[i]);
      const int cl = (tid >> 3) + 32 * i;
#pragma unroll
      for (int j = 0; j < 8; ++j) tile[chunk * 8 + j][cl] = e[j];
    }
    __syncthreads();
    if (slab + (int)gridDim.x < n_slab) fetch(slab + gridDim.x);
    const int c0 = slab * 64;
    if constexpr (FQ) {
      // four lanes per dst row (lanes r, r + 8, r + 16, r + 24 of warp w: row
      // 8 w + r), lane quarter q holding columns 32 m + 8 q .. + 7 (m = 0..3):
      // the block's scale is computed once per 32 values, and each store is a
      // 16-byte piece of 64 contiguous bytes per row
      const int r = lane & 7, q = lane >> 3, cl = 8 * warp + r, c = c0 + cl;
      const uint16_t* row = &tile[cl][8 * q];  // + 32 m + 2 i: columns 32 m + 8 q + 2 i, + 1
      // amax (a first pass over the row): with the sign bits cleared, bf16
      // patterns order as their values
      uint32_t mx = 0;
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          mx = __vmaxu2(mx, *reinterpret_cast<const uint32_t*>(row + 32 * m + 2 * i) & 0x7FFF7FFFu);
      mx = max(mx & 0xFFFFu, mx >> 16);
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float amax = __uint_as_float(mx << 16);
      float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
      if (pow2) scale = pow2_ceil(scale);
      const float inv = 1.0f / scale;
      __nv_bfloat16* o = dst + (int64_t)c * ldd;
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t x = *reinterpret_cast<const uint32_t*>(row + 32 * m + 2 * i);
          const float f0 = __uint_as_float(x << 16), f1 = __uint_as_float(x & 0xFFFF0000u);
          const __nv_fp8x2_storage_t e = __nv_cvt_float2_to_fp8x2(make_float2(f0 * inv, f1 * inv), __NV_SATFINITE,
                                                                  __NV_E4M3);
          const float2 back = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(e, __NV_E4M3)));
          w[i] = pack_bf16x2(back.x * scale, back.y * scale);
        }
        const int col = col0 + 32 * m + 8 * q;
        if (c >= C) continue;
        if (col + 8 <= n_cols) {
          *reinterpret_cast<uint4*>(o + col) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int cc = col + 2 * i;
            if (cc + 1 < n_cols) *reinterpret_cast<uint32_t*>(o + cc) = w[i];
            else if (cc < n_cols) *reinterpret_cast<uint16_t*>(o + cc) = static_cast<uint16_t>(w[i] & 0xFFFFu);
          }
        }
      }
    } else {
#pragma unroll 2
      for (int i = 0; i < 8; ++i) {
        const int cl = warp + 8 * i, c = c0 + cl;  // lane: columns 2 lane, +1 and 64 + 2 lane, +1
        if (c >= C) continue;
        const uint32_t w[2] = {*reinterpret_cast<const uint32_t*>(&tile[cl][2 * lane]),
                               *reinterpret_cast<const uint32_t*>(&tile[cl][64 + 2 * lane])};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int col = col0 + 2 * lane + 64 * j;
          if (col >= n_cols) continue;
          __nv_bfloat16* o = dst + (int64_t)c * ldd + col;
          if (col + 1 < n_cols) *reinterpret_cast<uint32_t*>(o) = w[j];
          else *reinterpret_cast<uint16_t*>(o) = static_cast<uint16_t>(w[j] & 0xFFFFu);
        }
      }
    }
    __syncthreads();
  }
}

// 1 x 128 quantisation of bf16 rows (ai.flicky.cc 3.3 item 2): the operand
// of an FP8 GEMM whose K runs along the rows.  codes [rows, C] E4M3 and
// scales [C/128][scale_ld] fp32 (MN-major, the layout of the GEMMs' activation
// scales): scale = amax/448 (UE8M0: rounded up to a power of two; 1 for an
// all-zero tile), codes = E4M3 of x * (1/scale) in fp32 with one correctly
// rounded reciprocal per tile (the rows are intermediates known to bf16
// accuracy).  A warp per row, a quarter warp per tile.
__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows, int C,
                                                         uint8_t* __restrict__ codes, float* __restrict__ scales,
                                                         int64_t scale_ld, bool pow2) {
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + row * C);
  const int groups = C / 128, ql = lane & 7, qw = lane >> 3;
  for (int g0 = 0; g0 < groups; g0 += 4) {
    const int g = g0 + qw;
    const bool active = g < groups;
    float f0[8], f1[8];
    float amax = 0.0f;
    if (active) {
      unpack8(s4[g * 16 + 2 * ql], f0);
      unpack8(s4[g * 16 + 2 * ql + 1], f1);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(f0[i]), fabsf(f1[i])));
    }
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    if (pow2) scale = pow2_ceil(scale);
    const float inv = 1.0f / scale;
    if (active) {
      uint32_t c8[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        c8[i] = e4m3x2(f0[2 * i] * inv, f0[2 * i + 1] * inv);
        c8[4 + i] = e4m3x2(f1[2 * i] * inv, f1[2 * i + 1] * inv);
      }
      reinterpret_cast<uint4*>(codes + row * C + g * 128)[ql] =
          make_uint4(c8[0] | (c8[1] << 16), c8[2] | (c8[3] << 16), c8[4] | (c8[5] << 16), c8[6] | (c8[7] << 16));
      if (ql == 0) scales[(int64_t)g * scale_ld + row] = scale;
    }
  }
}

// dst[b][c][r] = src[b][r][c] for bytes (FP8 weight codes [rows, C] per
// expert -> [C, rows]): 64 x 64 tiles, 16-byte loads, 4-byte stores; rows and
// C multiples of 4, 16-byte aligned rows.
__global__ void __launch_bounds__(256) transpose_u8_kernel(const uint8_t* __restrict__ src, int rows, int C,
                                                           int64_t batch_stride, uint8_t* __restrict__ dst) {
  __shared__ __align__(16) uint8_t tile[64][80];  // [r - r0][c - c0]
  src += blockIdx.z * batch_stride;
  dst += blockIdx.z * batch_stride;
  const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64, tid = threadIdx.x;
  {
    const int rl = tid >> 2, cl = (tid & 3) * 16, r = r0 + rl, c = c0 + cl;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < rows && c < C) v = *reinterpret_cast<const uint4*>(src + (int64_t)r * C + c);
    *reinterpret_cast<uint4*>(&tile[rl][cl]) = v;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = tid + 256 * i, cl = idx >> 4, rl = (idx & 15) * 4, c = c0 + cl, r = r0 + rl;
    if (c >= C || r >= rows) continue;
    const uint32_t w = uint32_t(tile[rl][cl]) | (uint32_t(tile[rl + 1][cl]) << 8) |
                       (uint32_t(tile[rl + 2][cl]) << 16) | (uint32_t(tile[rl + 3][cl]) << 24);
    *reinterpret_cast<uint32_t*>(dst + (int64_t)c * rows + r) = w;
  }
}

// dst[b][j][i] = src[b][i][j] for a small fp32 grid [rows, cols] per batch
// entry (the block scales of a transposed weight).
__global__ void transpose_f32_kernel(const float* __restrict__ src, int rows, int cols, int batch,
                                     float* __restrict__ dst) {
  const int64_t n = int64_t(batch) * rows * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / (int64_t(rows) * cols);
    const int rem = static_cast<int>(i - b * rows * cols), r = rem / cols, c = rem - r * cols;
    dst[b * rows * cols + int64_t(c) * rows + r] = src[i];
  }
}

// Gate and up values of a row in the w13 interleave: features f of block
// f / 128 sit at columns 256 (f / 128) + f % 128 (gate) and + 128 (up).
__device__ __forceinline__ int64_t gate_col(int f) { return 256 * (f >> 7) + (f & 127); }

// 8 floats -> 8 bf16 (16 bytes); unpack8 (kernels.cuh) is the inverse
__device__ __forceinline__ uint4 pack8_bf16(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

// h = SiLU(a) * b from the stored pre-activations ab [rows, 2I] (bf16, w13
// interleave) -> h [rows, I] bf16; 8 features per thread (I % 8 == 0, so
// the 8 never straddle a 128-feature block).
__global__ void swiglu_fwd_kernel(const __nv_bfloat16* __restrict__ ab, int64_t rows, int I,
                                  __nv_bfloat16* __restrict__ h) {
  const int I8 = I / 8;
  const int64_t n = rows * I8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / I8;
    const int f = static_cast<int>(i - r * I8) * 8;
    const __nv_bfloat16* row = ab + r * 2 * I + gate_col(f);
    float a[8], b[8], o[8];
    unpack8(*reinterpret_cast<const uint4*>(row), a);
    unpack8(*reinterpret_cast<const uint4*>(row + 128), b);
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = silu(a[j]) * b[j];
    *reinterpret_cast<uint4*>(h + r * I + f) = pack8_bf16(o);
  }
}

// SwiGLU backward: with sg = sigmoid(a), h = a sg b:
//   da = dh b sg (1 + a (1 - sg)),  db = dh a sg
// written into dab [rows, 2I] in the w13 interleave (the layout of ab);
// 8 features per thread.
__global__ void swiglu_bwd_kernel(const __nv_bfloat16* __restrict__ ab, const __nv_bfloat16* __restrict__ dh,
                                  int64_t rows, int I, __nv_bfloat16* __restrict__ dab) {
  const int I8 = I / 8;
  const int64_t n = rows * I8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / I8;
    const int f = static_cast<int>(i - r * I8) * 8;
    const int64_t ca = r * 2 * I + gate_col(f);
    float a[8], b[8], g[8], da[8], db[8];
    unpack8(*reinterpret_cast<const uint4*>(ab + ca), a);
    unpack8(*reinterpret_cast<const uint4*>(ab + ca + 128), b);
    unpack8(*reinterpret_cast<const uint4*>(dh + r * I + f), g);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float sg = 1.0f / (1.0f + __expf(-a[j]));
      da[j] = g[j] * b[j] * sg * (1.0f + a[j] * (1.0f - sg));
      db[j] = g[j] * a[j] * sg;
    }
    *reinterpret_cast<uint4*>(dab + ca) = pack8_bf16(da);
    *reinterpret_cast<uint4*>(dab + ca + 128) = pack8_bf16(db);
  }
}

// Backward of the gates, the last part for one token (block of 128 threads):
// with dg_j = dL/dg_{t,j} in s_dg[j][warp] (per-warp partial sums):
//   ds_j = (dg_j - sum_j' g_j' dg_j') / S, S = sum_j s_j;  dz_j = ds_j s_j (1 - s_j)
//   du_t = G_t + sum_j dz_j c_{e_j}                    (fp32: the residual and the router's share)
// dz_row[slot] = dz_j feeds the centroid gradient.
struct GateShared {
  int slot[32], e[32];
  float g[32], s[32], dg[32][4], dz[32];
};

__device__ __forceinline__ void gates_tail(GateShared& sh, int t, int k, int d, const __nv_bfloat16* __restrict__ Gt,
                                           const __nv_bfloat16* __restrict__ cent, float* __restrict__ dz_row,
                                           float* __restrict__ du) {
  const int tid = threadIdx.x;
  __syncthreads();
  if (tid < 32) {
    const bool on = tid < k && sh.slot[tid] >= 0;
    const float dg = on ? sh.dg[tid][0] + sh.dg[tid][1] + sh.dg[tid][2] + sh.dg[tid][3] : 0.0f;
    float gdg = on ? sh.g[tid] * dg : 0.0f, S = on ? sh.s[tid] : 0.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      gdg += __shfl_xor_sync(0xffffffffu, gdg, off);
      S += __shfl_xor_sync(0xffffffffu, S, off);
    }
    float dz = 0.0f;
    if (on) {
      const float s = sh.s[tid];
      // (S underflows only when every selected logit is below about -87; the
      // gates then came from the log domain and the affinities' own
      // gradient, s (1 - s), vanishes with them)
      dz = S > 0.0f ? (dg - gdg) / S * s * (1.0f - s) : 0.0f;
      dz_row[sh.slot[tid]] = dz;
    }
    if (tid < k) sh.dz[tid] = dz;
  }
  __syncthreads();
  const int d8 = d / 8;
  for (int c8 = tid; c8 < d8; c8 += blockDim.x) {
    float acc[8];
    unpack8(reinterpret_cast<const uint4*>(Gt)[c8], acc);
    for (int j = 0; j < k; ++j) {
      if (sh.e[j] < 0) continue;
      float cv[8];
      unpack8(reinterpret_cast<const uint4*>(cent + (int64_t)sh.e[j] * d)[c8], cv);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(sh.dz[j], cv[i], acc[i]);
    }
    float4* o = reinterpret_cast<float4*>(du + (int64_t)t * d) + 2 * c8;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// The token's selection: slots, experts, gates and the affinities s_j
// recomputed from the router's logits z (the sum of the K splits, as the
// top-k kernel takes it).  A bad slot or expert is recorded and skipped.
__device__ __forceinline__ void gates_head(GateShared& sh, int t, int k, int E, int64_t rows,
                                           const int32_t* __restrict__ slot, const int32_t* __restrict__ idx,
                                           const float* __restrict__ gate, const float* __restrict__ z, int splits,
                                           int64_t split_stride, int* status) {
  const int tid = threadIdx.x;
  if (tid < k) {
    int sl = slot[(int64_t)t * k + tid], e = idx[(int64_t)t * k + tid];
    if (sl < 0 || sl >= rows || e < 0 || e >= E) {
      record_status(status, ST_BAD_INDEX);
      sl = -1;
      e = -1;
    }
    sh.slot[tid] = sl;
    sh.e[tid] = e;
    sh.g[tid] = gate[(int64_t)t * k + tid];
    float zz = 0.0f;
    if (e >= 0) {
      zz = z[(int64_t)t * E + e];
      for (int p = 1; p < splits; ++p) zz += z[p * split_stride + (int64_t)t * E + e];
    }
    sh.s[tid] = 1.0f / (1.0f + expf(-zz));
  }
  __syncthreads();
}

// Backward of the combine and of the gates, one block (128 threads) per token:
//   dy[slot(t,j)] = g_{t,j} G_t                       (the routed experts' output gradient, bf16)
//   dg_j = G_t . y[slot(t,j)]                         (fp32, block reduction)
// then gates_tail.  8 columns per thread per step (d % 8 == 0).
__global__ void __launch_bounds__(128) combine_bwd_kernel(
    const __nv_bfloat16* __restrict__ G, const __nv_bfloat16* __restrict__ y, const int32_t* __restrict__ slot,
    const int32_t* __restrict__ idx, const float* __restrict__ gate, const float* __restrict__ z, int splits,
    int64_t split_stride, const __nv_bfloat16* __restrict__ cent, int T, int d, int k, int E, int64_t rows,
    __nv_bfloat16* __restrict__ dy, float* __restrict__ dz_row, float* __restrict__ du, int* status) {
  __shared__ GateShared sh;
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  gates_head(sh, t, k, E, rows, slot, idx, gate, z, splits, split_stride, status);
  const __nv_bfloat16* Gt = G + (int64_t)t * d;
  const int d8 = d / 8;
  for (int j = 0; j < k; ++j) {
    const int sl = sh.slot[j];
    float part = 0.0f;
    if (sl >= 0) {
      const float gj = sh.g[j];
      for (int c8 = tid; c8 < d8; c8 += blockDim.x) {
        float gv[8], yv[8], o[8];
        unpack8(reinterpret_cast<const uint4*>(Gt)[c8], gv);
        unpack8(reinterpret_cast<const uint4*>(y + (int64_t)sl * d)[c8], yv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          o[i] = gj * gv[i];
          part = fmaf(gv[i], yv[i], part);
        }
        reinterpret_cast<uint4*>(dy + (int64_t)sl * d)[c8] = pack8_bf16(o);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (lane == 0) sh.dg[j][wid] = part;
  }
  gates_tail(sh, t, k, d, Gt, cent, dz_row, du);
}

// dy[slot(t,j)] = g_{t,j} G_t for every routed row (bf16), block per token.
__global__ void __launch_bounds__(128) scale_rows_kernel(const __nv_bfloat16* __restrict__ G,
                                                         const int32_t* __restrict__ slot,
                                                         const float* __restrict__ gate, int k, int d, int64_t rows,
                                                         __nv_bfloat16* __restrict__ dy) {
  const int t = blockIdx.x;
  const uint4* Gt = reinterpret_cast<const uint4*>(G + (int64_t)t * d);
  const int d8 = d / 8;
  for (int j = 0; j < k; ++j) {
    const int sl = slot[(int64_t)t * k + j];
    if (sl < 0 || sl >= rows) continue;
    const float gj = gate[(int64_t)t * k + j];
    uint4* o = reinterpret_cast<uint4*>(dy + (int64_t)sl * d);
    for (int c8 = threadIdx.x; c8 < d8; c8 += blockDim.x) {
      float gv[8];
      unpack8(Gt[c8], gv);
#pragma unroll
      for (int i = 0; i < 8; ++i) gv[i] *= gj;
      o[c8] = pack8_bf16(gv);
    }
  }
}

// The gates' backward without the experts' outputs y: since dh = dy W2 and
// dy = g G, the gradient of the gate is
//   dg_j = G_t . y_r = G_t . (W2 h_r) = (G_t W2) . h_r = (dh_r . h_r) / g_j
// (r = slot(t, j)), a dot product of two [I] rows the backward holds anyway
// (0 for a gate that underflowed to 0); then gates_tail.
__global__ void __launch_bounds__(128) gate_grad_kernel(
    const __nv_bfloat16* __restrict__ G, const __nv_bfloat16* __restrict__ dh, const __nv_bfloat16* __restrict__ h,
    int I, const int32_t* __restrict__ slot, const int32_t* __restrict__ idx, const float* __restrict__ gate,
    const float* __restrict__ z, int splits, int64_t split_stride, const __nv_bfloat16* __restrict__ cent, int d, int k,
    int E, int64_t rows, float* __restrict__ dz_row, float* __restrict__ du, int* status) {
  __shared__ GateShared sh;
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  gates_head(sh, t, k, E, rows, slot, idx, gate, z, splits, split_stride, status);
  const int i8 = I / 8;
  for (int j = 0; j < k; ++j) {
    const int sl = sh.slot[j];
    float part = 0.0f;
    if (sl >= 0) {
      const uint4* a = reinterpret_cast<const uint4*>(dh + (int64_t)sl * I);
      const uint4* b = reinterpret_cast<const uint4*>(h + (int64_t)sl * I);
      for (int c8 = tid; c8 < i8; c8 += blockDim.x) {
        float av[8], bv[8];
        unpack8(a[c8], av);
        unpack8(b[c8], bv);
#pragma unroll
        for (int i = 0; i < 8; ++i) part = fmaf(av[i], bv[i], part);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (lane == 0) sh.dg[j][wid] = sh.g[j] > 0.0f ? part / sh.g[j] : 0.0f;
  }
  gates_tail(sh, t, k, d, G + (int64_t)t * d, cent, dz_row, du);
}

// du_t += sum_j dx[slot(t,j)] + sum_s dx_shared[s T + t]   (fp32 accumulation,
// 8 columns per thread: d % 8 == 0)
__global__ void __launch_bounds__(128) gather_dx_kernel(const __nv_bfloat16* __restrict__ dx,
                                                        const int32_t* __restrict__ slot, int k, int64_t rows,
                                                        const __nv_bfloat16* __restrict__ dx_shared, int n_shared,
                                                        int T, int d, float* __restrict__ du) {
  __shared__ int s_slot[32];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    const int s = slot[(int64_t)t * k + threadIdx.x];
    s_slot[threadIdx.x] = s >= 0 && s < rows ? s : -1;
  }
  __syncthreads();
  const int d8 = d / 8;
  for (int c8 = threadIdx.x; c8 < d8; c8 += blockDim.x) {
    float4* o = reinterpret_cast<float4*>(du + (int64_t)t * d) + 2 * c8;
    const float4 lo = o[0], hi = o[1];
    float acc[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    for (int j = 0; j < k; ++j) {
      if (s_slot[j] < 0) continue;
      float v[8];
      unpack8(reinterpret_cast<const uint4*>(dx + (int64_t)s_slot[j] * d)[c8], v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
    }
    for (int s = 0; s < n_shared; ++s) {
      float v[8];
      unpack8(reinterpret_cast<const uint4*>(dx_shared + ((int64_t)s * T + t) * d)[c8], v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
    }
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// Centroid gradient: dcent[e][c] = sum over expert e's rows r of
// dz_row[r] * u[perm[r]][c] (fp32).  Grid (E, d / 256), one column per thread.
__global__ void __launch_bounds__(256) dcent_kernel(const float* __restrict__ dz_row, const int32_t* __restrict__ perm,
                                                    const int32_t* __restrict__ offsets,
                                                    const __nv_bfloat16* __restrict__ u, int d,
                                                    float* __restrict__ dcent) {
  const int e = blockIdx.x, c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c >= d) return;
  float acc = 0.0f;
  for (int r = offsets[e]; r < offsets[e + 1]; ++r)
    acc = fmaf(dz_row[r], __bfloat162float(u[(int64_t)perm[r] * d + c]), acc);
  dcent[(int64_t)e * d + c] = acc;
}

}  // namespace moe
