/*
 * Seeded synthetic-input generator shared by the tests, the benchmark and
 * the oracle's callers.  It draws random numbers only: no quantisation,
 * routing, FFN or cache arithmetic of the MoE layer lives here.
 *
 * Counter-based: value i of stream `key` is a pure function of (key, i), so
 * any slice of any tensor can be regenerated independently (by either side,
 * on any number of threads) without storing it.
 *
 *   draw(key, i) = splitmix64_finaliser(key + (i + 1) * golden_gamma)
 *
 * is the SplitMix64 generator (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) evaluated at position i.
 *
 * Approximately normal values use the Irwin-Hall construction: the four
 * 16-bit fields of one draw are summed (an exact integer), centred and
 * scaled by one fp32 multiply, so the result is bit-identical on every
 * IEEE-754 machine.  The sum of four uniforms has mean 0, unit variance
 * after scaling, support +-3.46 sigma and excess kurtosis -0.3.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL
/* standard deviation of the sum of four uniform 16-bit integers */
#define IH4_SD 37837.22723720648
#define IH4_MEAN 131070

static inline uint64_t fin64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_draw(uint64_t key, uint64_t i) { return fin64(key + (i + 1) * GAMMA); }

/* Stream key for (seed, tag, a, b, c): nested finaliser so that nearby
 * tuples give unrelated streams. */
uint64_t synth_key(uint64_t seed, uint64_t tag, uint64_t a, uint64_t b, uint64_t c) {
  uint64_t k = fin64(seed + GAMMA);
  k = fin64(k ^ (tag + 1) * GAMMA);
  k = fin64(k ^ (a + 1) * 0xD1B54A32D192ED03ULL);
  k = fin64(k ^ (b + 1) * 0xAEF17502108EF2D9ULL);
  k = fin64(k ^ (c + 1) * 0xDB4F0B9175AE2165ULL);
  return k;
}

static inline int32_t ih4(uint64_t u) {
  return (int32_t)(u & 0xFFFF) + (int32_t)((u >> 16) & 0xFFFF) +
         (int32_t)((u >> 32) & 0xFFFF) + (int32_t)(u >> 48) - IH4_MEAN;
}

/* fp32 -> bf16 bits, round to nearest even (NaN -> canonical quiet NaN). */
static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

typedef struct {
  uint64_t key, start;
  int64_t lo, hi;
  float mul;
  void* out;
  int kind; /* 0 = f32, 1 = bf16 */
} job_t;

static void* run_job(void* p) {
  job_t* j = (job_t*)p;
  if (j->kind == 0) {
    float* o = (float*)j->out;
    for (int64_t i = j->lo; i < j->hi; ++i)
      o[i] = (float)ih4(synth_draw(j->key, j->start + (uint64_t)i)) * j->mul;
  } else {
    uint16_t* o = (uint16_t*)j->out;
    for (int64_t i = j->lo; i < j->hi; ++i)
      o[i] = f32_to_bf16_rne((float)ih4(synth_draw(j->key, j->start + (uint64_t)i)) * j->mul);
  }
  return NULL;
}

static void run_parallel(uint64_t key, uint64_t start, int64_t n, float sigma, void* out, int kind,
                         int nthreads) {
  float mul = (float)((double)sigma / IH4_SD);
  if (n <= 0) return;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (n < ((int64_t)1 << 20)) nthreads = 1;
  job_t jobs[64];
  pthread_t th[64];
  int spawned[64];
  int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].key = key;
    jobs[t].start = start;
    jobs[t].lo = (int64_t)t * per < n ? (int64_t)t * per : n;
    jobs[t].hi = jobs[t].lo + per < n ? jobs[t].lo + per : n;
    jobs[t].mul = mul;
    jobs[t].out = out;
    jobs[t].kind = kind;
    spawned[t] = 0;
  }
  /* share 0 runs on the calling thread; a share whose thread cannot be
   * created runs inline too */
  for (int t = 1; t < nthreads; ++t) {
    if (jobs[t].lo >= jobs[t].hi) continue;
    if (pthread_create(&th[t], NULL, run_job, &jobs[t]) == 0) spawned[t] = 1;
    else run_job(&jobs[t]);
  }
  run_job(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (spawned[t]) pthread_join(th[t], NULL);
}

/* out[i] = sigma * N01(key, start + i), i in [0, n) */
void synth_normal_f32(uint64_t key, uint64_t start, int64_t n, float sigma, float* out, int nthreads) {
  run_parallel(key, start, n, sigma, out, 0, nthreads);
}

/* bf16 (round to nearest even) of the same values */
void synth_normal_bf16(uint64_t key, uint64_t start, int64_t n, float sigma, uint16_t* out,
                       int nthreads) {
  run_parallel(key, start, n, sigma, out, 1, nthreads);
}

/* uniform integer in [0, m) by 64x64->128 multiply-high (Lemire). */
static inline uint64_t below(uint64_t u, uint64_t m) {
  return (uint64_t)(((__uint128_t)u * m) >> 64);
}

/* Seeded permutation pi of [0, n) (Fisher-Yates, draws from `key`). */
void synth_permutation(uint64_t key, int32_t n, int32_t* pi) {
  for (int32_t i = 0; i < n; ++i) pi[i] = i;
  for (int32_t i = n - 1; i > 0; --i) {
    int32_t j = (int32_t)below(synth_draw(key, (uint64_t)i), (uint64_t)i + 1);
    int32_t t = pi[i];
    pi[i] = pi[j];
    pi[j] = t;
  }
}

/* Popularity bias: expert e gets rank r = pi[e] (0 = most popular) and
 * bias[e] = log p_r with p_r = (r+1)^-s / sum_q (q+1)^-s (a Zipf law). */
void synth_zipf_bias(uint64_t key, int32_t n, double s, float* bias, int32_t* rank_out) {
  int32_t* pi = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
  if (!pi) return;
  synth_permutation(key, n, pi);
  double z = 0.0;
  for (int32_t r = n; r >= 1; --r) z += pow((double)r, -s);
  for (int32_t e = 0; e < n; ++e) {
    double p = pow((double)(pi[e] + 1), -s) / z;
    bias[e] = (float)log(p);
    if (rank_out) rank_out[e] = pi[e];
  }
  free(pi);
}
