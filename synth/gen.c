/*
 * Seeded synthetic input generator (host, C).
 *
 * This file only draws numbers.  It holds none of the MoE layer's arithmetic
 * and is shared by both sides of every comparison: the CPU oracle and the CUDA
 * library receive byte-identical copies of what it writes.
 *
 * Uniforms: element i of a stream with 64-bit key K is the SplitMix64
 * finaliser applied to K + (i + 1) * 0x9E3779B97F4A7C15 (Steele, Lea and
 * Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014).
 * Being counter-based, any element can be drawn without the ones before it,
 * so the work splits over OpenMP threads with a result that does not depend
 * on the thread count.
 *
 * Normals: inverse-CDF sampling.  The central part p in [1/N, 1 - 1/N] of the
 * unit interval (N = 16384 table intervals) interpolates linearly in a table
 * of the standard normal quantile; the two tails (probability 2/N) solve
 * Phi(x) = p by bisection with erfc from libm.  The interpolation error is
 * below 1e-3 absolute even at the table's edge (|x| ~ 3.8), far below what
 * a synthetic weight needs.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define TAB_N 16384

static double g_tab[TAB_N + 1];
static int g_tab_ready = 0;

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1ULL) * 0x9E3779B97F4A7C15ULL);
}

/* Standard normal CDF. */
static double phi_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

/* Quantile by bisection: 200 halvings of [-40, 40] reach double resolution. */
static double quantile_bisect(double p) {
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 200; ++it) {
    double mid = 0.5 * (lo + hi);
    if (mid == lo || mid == hi) break;
    if (phi_cdf(mid) < p) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

static void build_table(void) {
  if (g_tab_ready) return;
  g_tab[0] = -INFINITY;
  g_tab[TAB_N] = INFINITY;
  for (int j = 1; j < TAB_N; ++j) g_tab[j] = quantile_bisect((double)j / TAB_N);
  g_tab_ready = 1;
}

/* p in (0,1) from the top 53 bits, never 0 or 1. */
static inline double unit_open(uint64_t r) {
  return ((double)(r >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double normal_from(uint64_t r) {
  double p = unit_open(r);
  double pos = p * TAB_N;
  int j = (int)pos;
  if (j < 1 || j >= TAB_N - 1) return quantile_bisect(p);
  double f = pos - j;
  return g_tab[j] + f * (g_tab[j + 1] - g_tab[j]);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  b += 0x7FFFu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

/* Combine a key with a tag: used to derive per-tensor / per-expert keys. */
uint64_t synth_key(uint64_t key, uint64_t tag) {
  return mix64(key ^ mix64(tag + 0x632BE59BD9B4E019ULL));
}

/* out[i] = std * N(0,1) element i of stream `key`, rounded to bf16 (RNE). */
void synth_normal_bf16(uint64_t key, int64_t n, float std, uint16_t* out) {
  build_table();
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float v = (float)(std * normal_from(draw(key, (uint64_t)i)));
    out[i] = f32_to_bf16_rne(v);
  }
}

/* out[i] = std * N(0,1) element i of stream `key`, as fp32. */
void synth_normal_f32(uint64_t key, int64_t n, float std, float* out) {
  build_table();
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(std * normal_from(draw(key, (uint64_t)i)));
}

/* out[i] = uniform in (0,1), fp64. */
void synth_uniform_f64(uint64_t key, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = unit_open(draw(key, (uint64_t)i));
}

/*
 * Clustered tokens: u[t,:] = sqrt(rho) * centre[z[t],:] + sqrt(1-rho) * eps[t,:],
 * eps drawn from stream `key`, centres given in fp32, result rounded to bf16.
 * (Input construction only: each coordinate stays close to N(0,1).)
 */
void synth_clustered_bf16(uint64_t key, int64_t T, int64_t d, const float* centres,
                          const int32_t* z, float rho, uint16_t* out) {
  build_table();
  const double a = sqrt((double)rho), b = sqrt(1.0 - (double)rho);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const float* c = centres + (int64_t)z[t] * d;
    for (int64_t j = 0; j < d; ++j) {
      double e = normal_from(draw(key, (uint64_t)(t * d + j)));
      out[t * d + j] = f32_to_bf16_rne((float)(a * c[j] + b * e));
    }
  }
}
