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

#include "gemm.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Columns of the transposed activations for the weight-gradient GEMM: the rows
// of group g (offsets[g] .. offsets[g+1]) become columns pad_off[g] .., every
// group padded to a multiple of 64 columns (one 64-wide K stage of the GEMM;
// the padding is zero).  One block: the prefix is serial (G is at most a few
// thousand), the row -> column map is grid-strided by the same block.
__global__ void __launch_bounds__(1024) pad_plan_kernel(const int32_t* __restrict__ offsets, int G, int rows,
                                                        int32_t* __restrict__ pad_off, int32_t* __restrict__ col_of_row,
                                                        int* status) {
  __shared__ int s_off[2049];
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int g = 0; g <= G; ++g) {
      if (g <= 2048) s_off[g] = acc;
      pad_off[g] = acc;
      if (g < G) acc += (offsets[g + 1] - offsets[g] + 63) / 64 * 64;
    }
  }
  __syncthreads();
  if (G > 2048) {  // not used by the library (G <= E + n_shared <= 2048)
    if (threadIdx.x == 0) record_status(status, ST_BAD_INDEX);
    return;
  }
  for (int r = threadIdx.x; r < rows; r += blockDim.x) {
    int lo = 0, hi = G;  // find g with offsets[g] <= r < offsets[g + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (offsets[mid] <= r) lo = mid;
      else hi = mid;
    }
    col_of_row[r] = s_off[lo] + (r - offsets[lo]);
  }
}

// dst[c][col_of_row[r]] = src[r][c] for r < rows, c < C (bf16), batched over
// blockIdx.z (src/dst strides per batch).  col_of_row == nullptr: the
// identity.  32 x 32 tiles through shared memory, both sides coalesced.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const __nv_bfloat16* __restrict__ src, int rows, int C,
                                                             int64_t src_batch, const int32_t* __restrict__ col_of_row,
                                                             __nv_bfloat16* __restrict__ dst, int64_t ldd,
                                                             int64_t dst_batch) {
  __shared__ __nv_bfloat16 tile[32][33];
  src += blockIdx.z * src_batch;
  dst += blockIdx.z * dst_batch;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    const int r = r0 + ty + i, c = c0 + tx;
    if (r < rows && c < C) tile[ty + i][tx] = src[(int64_t)r * C + c];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    const int c = c0 + ty + i, r = r0 + tx;
    if (r < rows && c < C) {
      const int col = col_of_row ? col_of_row[r] : r;
      dst[(int64_t)c * ldd + col] = tile[tx][ty + i];
    }
  }
}

// Gate and up values of a row in the w13 interleave: features f of block
// f / 128 sit at columns 256 (f / 128) + f % 128 (gate) and + 128 (up).
__device__ __forceinline__ int64_t gate_col(int f) { return 256 * (f >> 7) + (f & 127); }

// h = SiLU(a) * b from the stored pre-activations ab [rows, 2I] (bf16, w13
// interleave) -> h [rows, I] bf16.
__global__ void swiglu_fwd_kernel(const __nv_bfloat16* __restrict__ ab, int64_t rows, int I,
                                  __nv_bfloat16* __restrict__ h) {
  const int64_t n = rows * I;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / I;
    const int f = static_cast<int>(i - r * I);
    const __nv_bfloat16* row = ab + r * 2 * I;
    const float a = __bfloat162float(row[gate_col(f)]), b = __bfloat162float(row[gate_col(f) + 128]);
    h[i] = __float2bfloat16_rn(silu(a) * b);
  }
}

// SwiGLU backward: with sg = sigmoid(a), h = a sg b:
//   da = dh b sg (1 + a (1 - sg)),  db = dh a sg
// written into dab [rows, 2I] in the w13 interleave (the layout of ab).
__global__ void swiglu_bwd_kernel(const __nv_bfloat16* __restrict__ ab, const __nv_bfloat16* __restrict__ dh,
                                  int64_t rows, int I, __nv_bfloat16* __restrict__ dab) {
  const int64_t n = rows * I;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / I;
    const int f = static_cast<int>(i - r * I);
    const int64_t ca = r * 2 * I + gate_col(f);
    const float a = __bfloat162float(ab[ca]), b = __bfloat162float(ab[ca + 128]);
    const float g = __bfloat162float(dh[i]);
    const float sg = 1.0f / (1.0f + __expf(-a));
    dab[ca] = __float2bfloat16_rn(g * b * sg * (1.0f + a * (1.0f - sg)));
    dab[ca + 128] = __float2bfloat16_rn(g * a * sg);
  }
}

// Backward of the combine and of the gates, one block (128 threads) per token:
//   dy[slot(t,j)] = g_{t,j} G_t                       (the routed experts' output gradient, bf16)
//   dg_j = G_t . y[slot(t,j)]                         (fp32, block reduction)
//   ds_j = (dg_j - sum_j' g_j' dg_j') / S, S = sum_j s_j;  dz_j = ds_j s_j (1 - s_j)
//   du_t = G_t + sum_j dz_j c_{e_j}                  (fp32: the residual and the router's share)
// s_j is recomputed from the router's logits z (the sum of the K splits, as
// the top-k kernel takes it).  dz_row[slot] = dz_j feeds the centroid gradient.
__global__ void __launch_bounds__(128) combine_bwd_kernel(
    const __nv_bfloat16* __restrict__ G, const __nv_bfloat16* __restrict__ y, const int32_t* __restrict__ slot,
    const int32_t* __restrict__ idx, const float* __restrict__ gate, const float* __restrict__ z, int splits,
    int64_t split_stride, const __nv_bfloat16* __restrict__ cent, int T, int d, int k, int E, int64_t rows,
    __nv_bfloat16* __restrict__ dy, float* __restrict__ dz_row, float* __restrict__ du, int* status) {
  __shared__ int s_slot[32], s_e[32];
  __shared__ float s_g[32], s_s[32], s_dg[32][4], s_dz[32];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid < k) {
    int sl = slot[(int64_t)t * k + tid], e = idx[(int64_t)t * k + tid];
    if (sl < 0 || sl >= rows || e < 0 || e >= E) {
      record_status(status, ST_BAD_INDEX);
      sl = -1;
      e = -1;
    }
    s_slot[tid] = sl;
    s_e[tid] = e;
    s_g[tid] = gate[(int64_t)t * k + tid];
    float zz = 0.0f;
    if (e >= 0) {
      zz = z[(int64_t)t * E + e];
      for (int p = 1; p < splits; ++p) zz += z[p * split_stride + (int64_t)t * E + e];
    }
    s_s[tid] = 1.0f / (1.0f + expf(-zz));
  }
  __syncthreads();
  const __nv_bfloat16* Gt = G + (int64_t)t * d;
  for (int j = 0; j < k; ++j) {
    const int sl = s_slot[j];
    float part = 0.0f;
    if (sl >= 0) {
      const float gj = s_g[j];
      for (int c = tid; c < d; c += blockDim.x) {
        const float gv = __bfloat162float(Gt[c]);
        dy[(int64_t)sl * d + c] = __float2bfloat16_rn(gj * gv);
        part = fmaf(gv, __bfloat162float(y[(int64_t)sl * d + c]), part);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (lane == 0) s_dg[j][wid] = part;
  }
  __syncthreads();
  if (tid < 32) {
    const bool on = tid < k && s_slot[tid] >= 0;
    const float dg = on ? s_dg[tid][0] + s_dg[tid][1] + s_dg[tid][2] + s_dg[tid][3] : 0.0f;
    float gdg = on ? s_g[tid] * dg : 0.0f, S = on ? s_s[tid] : 0.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      gdg += __shfl_xor_sync(0xffffffffu, gdg, off);
      S += __shfl_xor_sync(0xffffffffu, S, off);
    }
    float dz = 0.0f;
    if (on) {
      const float s = s_s[tid];
      // (S underflows only when every selected logit is below about -87; the
      // gates then came from the log domain and the affinities' own
      // gradient, s (1 - s), vanishes with them)
      dz = S > 0.0f ? (dg - gdg) / S * s * (1.0f - s) : 0.0f;
      dz_row[s_slot[tid]] = dz;
    }
    if (tid < k) s_dz[tid] = dz;
  }
  __syncthreads();
  for (int c = tid; c < d; c += blockDim.x) {
    float acc = __bfloat162float(Gt[c]);
    for (int j = 0; j < k; ++j)
      if (s_e[j] >= 0) acc = fmaf(s_dz[j], __bfloat162float(cent[(int64_t)s_e[j] * d + c]), acc);
    du[(int64_t)t * d + c] = acc;
  }
}

// du_t += sum_j dx[slot(t,j)] + sum_s dx_shared[s T + t]   (fp32 accumulation)
__global__ void __launch_bounds__(128) gather_dx_kernel(const __nv_bfloat16* __restrict__ dx,
                                                        const int32_t* __restrict__ slot, int k, int64_t rows,
                                                        const __nv_bfloat16* __restrict__ dx_shared, int n_shared,
                                                        int T, int d, float* __restrict__ du) {
  const int t = blockIdx.x;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float acc = du[(int64_t)t * d + c];
    for (int j = 0; j < k; ++j) {
      const int s = slot[(int64_t)t * k + j];
      if (s >= 0 && s < rows) acc += __bfloat162float(dx[(int64_t)s * d + c]);
    }
    for (int s = 0; s < n_shared; ++s) acc += __bfloat162float(dx_shared[((int64_t)s * T + t) * d + c]);
    du[(int64_t)t * d + c] = acc;
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
