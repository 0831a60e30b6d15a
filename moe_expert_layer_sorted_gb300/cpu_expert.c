/* SwiGLU expert FFN on the host CPU, over one expert in the canonical int-b
 * group-quantised format, for T tokens: g = Wg x, u = Wu x, h = silu(g) * u,
 * o = Wd h (fp32 arithmetic, h kept in fp32).
 *
 * This is the measured comparison of "CPU compute of a host-resident expert"
 * against the GPU reading that expert in place over its host link (the CPU
 * fill-in for cache misses of "Running a 24k-expert MoE on a single 32 GB
 * card", section 2 "Tiering, not activation, makes it run", and the
 * CPU-computed expert layers of "125B sparse model on one 32 GB consumer
 * card", section "Conclusion first").  It is not a path of the library,
 * which has no CPU fallback; only the benchmark and its test call it.
 *
 * Codes: weight i of a [rows][cols] matrix (row-major) occupies bits
 * [i*b, i*b + b) of a little-endian bit stream and holds u = q + 2^(b-1).
 * cols is a multiple of the group size G, itself a multiple of 8, so every
 * row starts on a byte and every 8 consecutive weights fill exactly b bytes.
 * Scales: [rows][cols / G] as fp32, bf16 or fp16 (scale dtype 0, 1, 2); the
 * weight is q * s.
 *
 * Work is split over `threads` POSIX threads by output rows: first the I rows
 * of gate and up, then (after a join) the H rows of down.  Per row, codes are
 * decoded 8 at a time into fp32 and multiplied against the tokens in 8
 * independent partial sums per group (a shape the compiler vectorises without
 * reassociating any single sum); each group's sum is scaled once. */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define CPU_MAX_T 8

static float half_to_float(uint16_t h) {
  const uint32_t s = (uint32_t)(h >> 15) << 31, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  uint32_t bits;
  if (e == 0) {
    if (m == 0) {
      bits = s;
    } else {  /* subnormal: m * 2^-24 */
      float f = (float)m * (1.0f / 16777216.0f);
      memcpy(&bits, &f, 4);
      bits |= s;
    }
  } else if (e == 31) {
    bits = s | 0x7f800000u | (m << 13);
  } else {
    bits = s | ((e + 112) << 23) | (m << 13);
  }
  float f;
  memcpy(&f, &bits, 4);
  return f;
}

static float scale_at(const void* scales, int64_t i, int sdt) {
  if (sdt == 0) return ((const float*)scales)[i];
  const uint16_t h = ((const uint16_t*)scales)[i];
  if (sdt == 1) {
    const uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, 4);
    return f;
  }
  return half_to_float(h);
}

/* the `cols` weights of row r (without their scales) as q in fp32 */
static void decode_row(const uint8_t* codes, int r, int cols, int b, float* q) {
  const uint8_t* p = codes + (int64_t)r * cols / 8 * b;
  const uint32_t mask = (1u << b) - 1u;
  const int off = 1 << (b - 1);
  for (int c = 0; c < cols; c += 8, p += b) {
    uint32_t w = 0;
    for (int j = 0; j < b; ++j) w |= (uint32_t)p[j] << (8 * j);
    for (int j = 0; j < 8; ++j) q[c + j] = (float)((int)((w >> (b * j)) & mask) - off);
  }
}

/* acc[t] = sum over the row of s * q * x[t] for T token rows x [T][cols] */
static void row_dot(const float* q, const void* scales, int64_t srow, int cols, int G, int sdt,
                    const float* x, int T, float* acc) {
  for (int t = 0; t < T; ++t) acc[t] = 0.0f;
  for (int c0 = 0; c0 < cols; c0 += G) {
    const float s = scale_at(scales, srow + c0 / G, sdt);
    for (int t = 0; t < T; ++t) {
      const float* xt = x + (int64_t)t * cols + c0;
      float part[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int c = 0; c < G; c += 8)
        for (int j = 0; j < 8; ++j) part[j] += q[c0 + c + j] * xt[c + j];
      const float sum = ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
      acc[t] += s * sum;
    }
  }
}

typedef struct {
  const uint8_t* codes[3];
  const void* scales[3];
  int H, I, b, G, sdt, T;
  const float* x;  /* [T][H] */
  float* h;        /* [T][I] */
  float* o;        /* [T][H] */
  int phase, r0, r1;
} job_t;

static void* worker(void* arg) {
  job_t* j = (job_t*)arg;
  const int cols = j->phase == 0 ? j->H : j->I;
  float* q = (float*)malloc(sizeof(float) * (size_t)cols);
  float a0[CPU_MAX_T], a1[CPU_MAX_T];
  for (int r = j->r0; r < j->r1; ++r) {
    if (j->phase == 0) {  /* gate and up row r -> h[t][r] */
      decode_row(j->codes[0], r, cols, j->b, q);
      row_dot(q, j->scales[0], (int64_t)r * (cols / j->G), cols, j->G, j->sdt, j->x, j->T, a0);
      decode_row(j->codes[1], r, cols, j->b, q);
      row_dot(q, j->scales[1], (int64_t)r * (cols / j->G), cols, j->G, j->sdt, j->x, j->T, a1);
      for (int t = 0; t < j->T; ++t) {
        const float g = a0[t];
        j->h[(int64_t)t * j->I + r] = g / (1.0f + expf(-g)) * a1[t];
      }
    } else {  /* down row r -> o[t][r] */
      decode_row(j->codes[2], r, cols, j->b, q);
      row_dot(q, j->scales[2], (int64_t)r * (cols / j->G), cols, j->G, j->sdt, j->h, j->T, a0);
      for (int t = 0; t < j->T; ++t) j->o[(int64_t)t * j->H + r] = a0[t];
    }
  }
  free(q);
  return NULL;
}

static void run_phase(job_t* base, int phase, int rows, int threads) {
  pthread_t tid[256];
  job_t jobs[256];
  int n = threads < 1 ? 1 : (threads > 256 ? 256 : threads);
  if (n > rows) n = rows;
  for (int i = 0; i < n; ++i) {
    jobs[i] = *base;
    jobs[i].phase = phase;
    jobs[i].r0 = (int)((int64_t)rows * i / n);
    jobs[i].r1 = (int)((int64_t)rows * (i + 1) / n);
  }
  for (int i = 1; i < n; ++i) pthread_create(&tid[i], NULL, worker, &jobs[i]);
  worker(&jobs[0]);
  for (int i = 1; i < n; ++i) pthread_join(tid[i], NULL);
}

/* x_bf16 [T][H] (bf16 bits), out [T][H] fp32.  Returns 0, or -1 for bad
 * arguments (T outside [1, 8], b outside {2, 3, 4}, G not a positive
 * multiple of 8 dividing both H and I). */
int cpu_expert_ffn(const void* const codes[3], const void* const scales[3], int H, int I, int b, int G,
                   int sdt, const uint16_t* x_bf16, int T, float* out, int threads) {
  if (T < 1 || T > CPU_MAX_T || b < 2 || b > 4 || G < 8 || G % 8 || H % G || I % G || sdt < 0 || sdt > 2)
    return -1;
  float* x = (float*)malloc(sizeof(float) * (size_t)T * H);
  float* h = (float*)malloc(sizeof(float) * (size_t)T * I);
  for (int64_t i = 0; i < (int64_t)T * H; ++i) {
    const uint32_t bits = (uint32_t)x_bf16[i] << 16;
    memcpy(&x[i], &bits, 4);
  }
  job_t base;
  memset(&base, 0, sizeof(base));
  for (int m = 0; m < 3; ++m) {
    base.codes[m] = (const uint8_t*)codes[m];
    base.scales[m] = scales[m];
  }
  base.H = H;
  base.I = I;
  base.b = b;
  base.G = G;
  base.sdt = sdt;
  base.T = T;
  base.x = x;
  base.h = h;
  base.o = out;
  run_phase(&base, 0, I, threads);
  run_phase(&base, 1, H, threads);
  free(x);
  free(h);
  return 0;
}
