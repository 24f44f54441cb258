/* Seeded synthetic inputs for the NVFP4 KV-cache workloads.
 *
 * This module holds only random-number generation: no step of the method lives here. It is the
 * one piece shared by the CUDA path's tests and the CPU oracle, so both see identical inputs.
 *
 * Generator: a counter-based splitmix64 stream. A stream key is derived from (seed, stream id);
 * draw(key, n) = splitmix64 finaliser applied to key + (n + 1) * 0x9E3779B97F4A7C15, i.e. the
 * n-th output of the splitmix64 sequence started at `key` (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014). Every element is addressed by its
 * own counter, so any token row can be regenerated on its own.
 *
 * Normal values: Box-Muller in double from two uniforms, then one round-to-nearest-even to bf16.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed + GOLDEN) ^ mix64(stream * 0xD1B54A32D192ED03ULL + 1ULL));
}

uint64_t synth_draw(uint64_t key, uint64_t n) { return mix64(key + (n + 1ULL) * GOLDEN); }

/* Round a double to the nearest bf16 (ties to even) and return the bit pattern. Inputs are
 * finite and far inside the bf16 range. */
static inline uint16_t double_to_bf16_rne(double x) {
  uint64_t b;
  memcpy(&b, &x, 8);
  /* keep 1 + 7 significand bits: 45 of the 52 stored bits are dropped */
  const uint64_t drop = 45;
  const uint64_t half = 1ULL << (drop - 1);
  const uint64_t rem = b & ((1ULL << drop) - 1);
  uint64_t t = b >> drop;
  if (rem > half || (rem == half && (t & 1ULL))) t += 1;
  b = t << drop;
  double r;
  memcpy(&r, &b, 8);
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t fb;
  memcpy(&fb, &f, 4);
  return (uint16_t)(fb >> 16);
}

/* Fill out[n_tok][heads][dim] with bf16 N(0,1) draws for tokens pos0 .. pos0+n_tok-1 of sequence
 * `seq`. Element counter c = (seq << 40) | (pos << 16) | (h * dim + d); the two uniforms of that
 * element are draws 2c and 2c+1. Channels listed in `outliers` are multiplied by `outlier_mult`
 * (in double) before the bf16 rounding. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, int32_t seq, int32_t pos0, int32_t n_tok,
                       int32_t heads, int32_t dim, const int32_t* outliers, int32_t n_outliers,
                       double outlier_mult, uint16_t* out, int32_t nthreads) {
  const uint64_t key = synth_stream_key(seed, stream);
  const double two_pi = 6.283185307179586476925286766559;
  const double inv53 = 1.0 / 9007199254740992.0; /* 2^-53 */
  double mult[4096];
  for (int d = 0; d < dim && d < 4096; ++d) mult[d] = 1.0;
  for (int k = 0; k < n_outliers; ++k)
    if (outliers[k] >= 0 && outliers[k] < dim) mult[outliers[k]] = outlier_mult;
#ifdef _OPENMP
  const int nt_used = nthreads > 0 ? nthreads : omp_get_max_threads();  // global setting kept
#pragma omp parallel for num_threads(nt_used) schedule(static)
#endif
  for (int64_t t = 0; t < (int64_t)n_tok; ++t) {
    const uint64_t pos = (uint64_t)(pos0 + t);
    for (int32_t h = 0; h < heads; ++h) {
      for (int32_t d = 0; d < dim; ++d) {
        const uint64_t c = ((uint64_t)seq << 40) | (pos << 16) | (uint64_t)(h * dim + d);
        const double u1 = ((double)(synth_draw(key, 2 * c) >> 11) + 0.5) * inv53;
        const double u2 = (double)(synth_draw(key, 2 * c + 1) >> 11) * inv53;
        const double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
        out[(t * heads + h) * dim + d] = double_to_bf16_rne(z * mult[d]);
      }
    }
  }
}

/* Seeded Fisher-Yates permutation of 0..n-1. Step i (from n-1 down to 1) swaps element i with
 * element j = floor(r * (i+1) / 2^32), r = top 32 bits of draw(key, i). */
void synth_permutation(uint64_t seed, uint64_t stream, int32_t n, int32_t* out) {
  const uint64_t key = synth_stream_key(seed, stream);
  for (int32_t i = 0; i < n; ++i) out[i] = i;
  for (int32_t i = n - 1; i >= 1; --i) {
    const uint64_t r = synth_draw(key, (uint64_t)i) >> 32;
    const int32_t j = (int32_t)((r * (uint64_t)(i + 1)) >> 32);
    const int32_t tmp = out[i];
    out[i] = out[j];
    out[j] = tmp;
  }
}

/* n integers floor(exp(U(ln lo, ln hi))), U uniform in [0,1) from draw(key, i). */
void synth_loguniform_int(uint64_t seed, uint64_t stream, int32_t n, double lo, double hi,
                          int32_t* out) {
  const uint64_t key = synth_stream_key(seed, stream);
  const double inv53 = 1.0 / 9007199254740992.0;
  for (int32_t i = 0; i < n; ++i) {
    const double u = (double)(synth_draw(key, (uint64_t)i) >> 11) * inv53;
    out[i] = (int32_t)floor(exp(log(lo) + u * (log(hi) - log(lo))));
  }
}

/* n uniform integers in [0, m): floor(r * m / 2^32), r = top 32 bits of draw(key, i). */
void synth_uniform_int(uint64_t seed, uint64_t stream, int32_t n, int32_t m, int32_t* out) {
  const uint64_t key = synth_stream_key(seed, stream);
  for (int32_t i = 0; i < n; ++i) {
    const uint64_t r = synth_draw(key, (uint64_t)i) >> 32;
    out[i] = (int32_t)((r * (uint64_t)m) >> 32);
  }
}
