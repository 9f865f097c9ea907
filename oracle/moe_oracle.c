/*
 * CPU oracle of the DeepSeekMoE layer forward -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the bench
 * load this code.  It shares nothing with the CUDA library: no header, no
 * helper, no table.  It is plain, slow and written to be checked by eye
 * against the method's statement:
 *
 *   DeepSeek-V3 technical report as read on ai.flicky.cc ("06 - DeepSeek-V3
 *   reading", section 2.1.2 "DeepSeekMoE and auxiliary-loss-free balancing",
 *   the layer equation for h'_t and s_{i,t} and the g'_{i,t} selection rule)
 *   and on xyznot.com ("DeepSeek-V3 technical report", Method 2, the h'_t,
 *   s_{i,t}, g'_{i,t} equations and the normalisation of g').
 *   FP8: the ai.flicky.cc page, section 3.3 "FP8 training", items 1-4.
 *   Expert FFN: the ai.flicky.cc page, the practice exercise's expert_params
 *   docstring (an expert is a SwiGLU FFN of three d x d_expert matrices).
 *
 * Floating point: fp64 throughout, except where a float decides an integer
 * (an FP8 code) or where the method's state is fp32 (the bias), which are
 * computed in fp32 like the kernels.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* bf16 bit pattern -> exact double. */
static double bf16_to_f64(uint16_t h) {
  uint32_t b = (uint32_t)h << 16;
  float f;
  memcpy(&f, &b, 4);
  return (double)f;
}

void oracle_bf16_to_f64(int64_t n, const uint16_t* in, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_f64(in[i]);
}

/* ---------------------------------------------------------------------------
 * Router (ai.flicky.cc section 2.1.2; xyznot.com Method 2).
 *   s_{i,t} = sigmoid(u_t^T e_i)
 *   selection: the K_r experts with the largest s_{i,t} + b_i
 *   g'_{i,t} = s_{i,t} if selected else 0;  g_{i,t} = g'_{i,t} / sum_j g'_{j,t}
 * The bias enters the selection only, never the gate value.
 * Readings where the pages are silent: exact ties go to the lower expert
 * index; a NaN score ranks below every number; the k selected experts are
 * reported by biased score descending, then index ascending.
 *
 * Outputs per token t: idx[t*k+j], s_sel[t*k+j] (unbiased affinity of the
 * j-th selected expert), gate[t*k+j], and gap[t] = (k-th biased score) -
 * ((k+1)-th biased score), +inf when k == E: the distance to a change of
 * selection, used to flag near-ties.  s_all (may be NULL) receives every
 * affinity s_{i,t}, [T, E].
 */
static int better(double a, int ia, double b, int ib) {
  /* is (a, ia) ranked before (b, ib)?  NaN ranks last; ties -> lower index */
  int na = isnan(a), nb = isnan(b);
  if (na != nb) return nb;
  if (!na && a != b) return a > b;
  return ia < ib;
}

/*
 * Node-limited routing (ai.flicky.cc 2.1.2: a token is sent to at most 4
 * nodes).  The E experts sit on `groups` nodes of E / groups consecutive
 * experts; groups == 0 means no limit.  The pages fix only the limit, not how
 * the nodes are chosen; reading: the k experts are taken in biased-score
 * order, and an expert is skipped when its node is not yet in use and `limit`
 * nodes already are -- which keeps the `limit` nodes whose best expert scores
 * highest and takes the k best experts inside them.  With a binding limit the
 * near-tie distance also covers the choice of nodes: gap is at most the score
 * of the pick that brought in the last node minus the best score on a node
 * left out.
 */
void oracle_route_limited(int64_t T, int d, int E, int k, int groups, int limit, const uint16_t* u,
                          const uint16_t* cent, const float* bias, int32_t* idx, double* s_sel, double* gate,
                          double* gap, double* s_all) {
  const int gs = groups > 0 ? E / groups : E;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t t = 0; t < T; ++t) {
    double s[E], score[E];
    char taken[E];
    char used[groups > 0 ? groups : 1];
    int n_used = 0;
    double last_node_pick = INFINITY;
    for (int n = 0; n < (groups > 0 ? groups : 1); ++n) used[n] = 0;
    for (int i = 0; i < E; ++i) {
      double z = 0.0;
      for (int c = 0; c < d; ++c) z += bf16_to_f64(u[t * d + c]) * bf16_to_f64(cent[(int64_t)i * d + c]);
      s[i] = 1.0 / (1.0 + exp(-z));
      score[i] = s[i] + (double)bias[i];
      taken[i] = 0;
      if (s_all) s_all[t * E + i] = s[i];
    }
    double sum = 0.0, kth = 0.0;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int i = 0; i < E; ++i) {
        const int allowed = groups == 0 || used[i / gs] || n_used < limit;
        if (!taken[i] && allowed && (best < 0 || better(score[i], i, score[best], best))) best = i;
      }
      taken[best] = 1;
      if (groups > 0 && !used[best / gs]) {
        used[best / gs] = 1;
        ++n_used;
        last_node_pick = score[best];
      }
      idx[t * k + j] = best;
      s_sel[t * k + j] = s[best];
      sum += s[best];
      kth = score[best];
    }
    for (int j = 0; j < k; ++j) gate[t * k + j] = s_sel[t * k + j] / sum;
    int next = -1, out = -1;
    for (int i = 0; i < E; ++i) {
      if (taken[i]) continue;
      if (groups == 0 || used[i / gs] || n_used < limit) {
        if (next < 0 || better(score[i], i, score[next], next)) next = i;
      } else if (out < 0 || better(score[i], i, score[out], out)) {
        out = i;
      }
    }
    double g = next < 0 ? INFINITY : kth - score[next];
    if (out >= 0 && last_node_pick - score[out] < g) g = last_node_pick - score[out];
    gap[t] = g;
  }
}

void oracle_route(int64_t T, int d, int E, int k, const uint16_t* u, const uint16_t* cent,
                  const float* bias, int32_t* idx, double* s_sel, double* gate, double* gap,
                  double* s_all) {
  oracle_route_limited(T, d, E, k, 0, 0, u, cent, bias, idx, s_sel, gate, gap, s_all);
}

/* ---------------------------------------------------------------------------
 * FP8 E4M3 (ai.flicky.cc section 3.3 items 2 and 4; glossary: E4M3, max 448).
 * Format from its definition: 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * no infinities; S.1111.111 is NaN; largest finite 1.75 * 2^8 = 448;
 * exponent field 0 holds subnormals m/8 * 2^-6.
 */
double oracle_e4m3_decode(uint8_t q) {
  int sgn = q >> 7, e = (q >> 3) & 15, m = q & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sgn ? -v : v;
}

/* Round to nearest, ties to even; saturate to +-448; NaN -> 0x7F. */
uint8_t oracle_e4m3_encode(double x) {
  if (isnan(x)) return 0x7F;
  uint8_t sgn = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  if (a >= 448.0) return sgn | 0x7E;
  if (a < ldexp(1.0, -6)) {                 /* subnormal range: multiples of 2^-9 */
    double m = nearbyint(a * 512.0);       /* default rounding mode: ties to even */
    return sgn | (uint8_t)m;               /* m == 8 is the smallest normal, code 0x08 */
  }
  int ex;
  frexp(a, &ex);                           /* a = f * 2^ex, f in [0.5, 1) */
  int e = ex - 1;                          /* a in [2^e, 2^(e+1)) */
  double m = nearbyint((a / ldexp(1.0, e) - 1.0) * 8.0);
  if (m == 8.0) { m = 0.0; e += 1; }
  if (e + 7 > 15 || (e + 7 == 15 && m > 6.0)) return sgn | 0x7E;
  return sgn | (uint8_t)(((e + 7) << 3) | (int)m);
}

/* Scale of one group: amax / 448 in fp32; an all-zero group gets scale 1. */
static float group_scale(double amax) {
  if (!(amax > 0.0)) return 1.0f;
  return (float)amax / 448.0f;
}

/*
 * UE8M0 scales (ai.flicky.cc, continuation of section 3.5: DeepSeek-V3.1 moved
 * to FP8 with UE8M0 scales, a scale that is a bare 8-bit exponent).  The page
 * gives no rounding rule; reading: the amax/448 scale above rounded UP to a
 * power of two, so that no element of the group exceeds 448 after scaling.
 * frexpf splits s = f * 2^e with f in [0.5, 1); s is a power of two exactly
 * when f == 0.5.  Scales below 2^-126 (never met by bf16 data) become 2^-126.
 */
static float group_scale_pow2(double amax) {
  const float s = group_scale(amax);
  if (s <= ldexpf(1.0f, -126)) return ldexpf(1.0f, -126);
  int e;
  const float f = frexpf(s, &e);
  return f == 0.5f ? s : ldexpf(1.0f, e);
}

static float scale_of(double amax, int pow2) { return pow2 ? group_scale_pow2(amax) : group_scale(amax); }

/* Code of one element: x / scale rounded to fp32 (the kernels' precision), then E4M3. */
static uint8_t quant_elem(double x, float scale) { return oracle_e4m3_encode((double)((float)x / scale)); }

/* The same from x * (1 / scale): the fp32 reciprocal of the tile's scale
 * (correctly rounded), then the fp32 product, then E4M3. */
static uint8_t quant_elem_recip(double x, float inv) { return oracle_e4m3_encode((double)((float)x * inv)); }

/*
 * Activation tiles 1 x 128 (ai.flicky.cc 3.3 item 2): row r, columns
 * [128g, 128g+128) share scale[r * G + g], G = cols / 128.  recip != 0: codes
 * from x * (1/scale) (quant_elem_recip) instead of x / scale.
 */
void oracle_quant_1x128(int64_t rows, int cols, const double* x, uint8_t* q, float* scale, int pow2, int recip) {
  const int G = cols / 128;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int g = 0; g < G; ++g) {
      double amax = 0.0;
      for (int c = 128 * g; c < 128 * g + 128; ++c) amax = fmax(amax, fabs(x[r * cols + c]));
      float s = scale_of(amax, pow2);
      scale[r * G + g] = s;
      const float inv = 1.0f / s;
      for (int c = 128 * g; c < 128 * g + 128; ++c)
        q[r * cols + c] = recip ? quant_elem_recip(x[r * cols + c], inv) : quant_elem(x[r * cols + c], s);
    }
}

/*
 * Weight blocks 128 x 128 (ai.flicky.cc 3.3 item 2): block (br, bc) of a
 * [rows, cols] matrix shares scale[br * (cols/128) + bc].
 */
void oracle_quant_128x128(int64_t rows, int cols, const double* w, uint8_t* q, float* scale, int pow2) {
  const int64_t BR = rows / 128;
  const int BC = cols / 128;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t br = 0; br < BR; ++br)
    for (int bc = 0; bc < BC; ++bc) {
      double amax = 0.0;
      for (int64_t r = 128 * br; r < 128 * br + 128; ++r)
        for (int c = 128 * bc; c < 128 * bc + 128; ++c) amax = fmax(amax, fabs(w[r * cols + c]));
      float s = scale_of(amax, pow2);
      scale[br * BC + bc] = s;
      for (int64_t r = 128 * br; r < 128 * br + 128; ++r)
        for (int c = 128 * bc; c < 128 * bc + 128; ++c) q[r * cols + c] = quant_elem(w[r * cols + c], s);
    }
}

/*
 * Dequantisation (code value times its scale), fp64: 1 x 128 tiles of a
 * [rows, cols] matrix (scale [rows, cols/128]) or 128 x 128 blocks (scale
 * [rows/128, cols/128]).
 */
void oracle_dequant(int64_t rows, int cols, const uint8_t* q, const float* scale, int block_rows, double* out) {
  const int G = cols / 128;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int c = 0; c < cols; ++c)
      out[r * cols + c] = oracle_e4m3_decode(q[r * cols + c]) * (double)scale[(r / block_rows) * G + c / 128];
}

/* ---------------------------------------------------------------------------
 * One SwiGLU expert (ai.flicky.cc practice exercise: three d x d_expert
 * matrices), on n rows:  y = W2 (SiLU(W1 x) * (W3 x)),  SiLU(a) = a sigmoid(a).
 * x [n, d], w1 and w3 [I, d], w2 [d, I] (nn.Linear layout), y [n, d]; fp64.
 * h_quant != 0: h is replaced by its FP8 1 x 128 quantise-dequantise along I
 * (h_quant == 2: with UE8M0 scales)
 * before the down projection, as the FP8 scheme quantises the input of every
 * main GEMM (ai.flicky.cc 3.3 items 1-2).
 */
void oracle_swiglu(int64_t n, int d, int I, const double* x, const double* w1, const double* w3,
                   const double* w2, int h_quant, double* y) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n; ++r) {
    double h[I];
    const double* xr = x + r * d;
    for (int i = 0; i < I; ++i) {
      double g = 0.0, v = 0.0;
      for (int c = 0; c < d; ++c) {
        g += w1[(int64_t)i * d + c] * xr[c];
        v += w3[(int64_t)i * d + c] * xr[c];
      }
      h[i] = g / (1.0 + exp(-g)) * v;
    }
    if (h_quant) {
      for (int gi = 0; gi < I / 128; ++gi) {
        double amax = 0.0;
        for (int i = 128 * gi; i < 128 * gi + 128; ++i) amax = fmax(amax, fabs(h[i]));
        float s = scale_of(amax, h_quant == 2);
        for (int i = 128 * gi; i < 128 * gi + 128; ++i) h[i] = oracle_e4m3_decode(quant_elem(h[i], s)) * (double)s;
      }
    }
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int i = 0; i < I; ++i) acc += w2[(int64_t)c * I + i] * h[i];
      y[r * d + c] = acc;
    }
  }
}

/* ---------------------------------------------------------------------------
 * Auxiliary-loss-free bias update (ai.flicky.cc 2.1.2: after every step the
 * bias of an overloaded expert drops by gamma, that of an underloaded one
 * rises by gamma; xyznot.com Method 2 says the same with gamma = 0.001).
 * Reading: the load of expert i is counts[i] over the step's T*k selections;
 * overloaded / underloaded means above / below the mean load T*k/E; an expert
 * exactly at the mean keeps its bias.  The bias is fp32 state, so this runs
 * in fp32 like the kernel: b_i <- b_i + gamma * sign(mean - load_i).
 */
void oracle_bias_update(int E, int64_t T, int k, const int32_t* counts, float gamma, float* bias) {
  const float mean = (float)(T * k) / (float)E;
  for (int i = 0; i < E; ++i) {
    const float load = (float)counts[i];
    const float sgn = mean > load ? 1.0f : (mean < load ? -1.0f : 0.0f);
    bias[i] = bias[i] + gamma * sgn;
  }
}
