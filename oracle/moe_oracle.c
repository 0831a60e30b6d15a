/*
 * CPU oracle for the tiered MoE layer.  TEST INFRASTRUCTURE ONLY: it is
 * called by tests/, by __graft_entry__.smoke() and by the benchmark's CPU
 * baseline leg, never by the library.  It shares no code with the CUDA path.
 *
 * Plain, slow and written to be checked by eye against the definitions:
 *  - the MoE layer of "763B MoE in two 96 GB cards", section "Where the VRAM
 *    gap comes from" (routed experts per layer, top-k per token) and the
 *    per-expert split of its "Same idea, native vLLM fails" side-box;
 *  - low-bit group quantisation ("763B ...", EXL3 side-box; "125B sparse
 *    model on one 32 GB consumer card", header; "Running a 24k-expert MoE on
 *    a single 32 GB card", section 2), read as symmetric int-b with one
 *    scale per group of G weights along the reduction axis;
 *  - SwiGLU expert FFN: h = silu(Wg x) * (Wu x), o = Wd h;
 *  - the adaptive frequency-admitted expert cache of "Running a 24k-expert
 *    MoE ...", sections 2 and 3.
 *
 * Precision: quantisation and routing decisions are taken in fp32 (the
 * precision the integer results depend on); the FFN, the routing weights
 * and the combine are evaluated in fp64.
 *
 * Parity pins: every function here is pinned by tests/test_oracle_*.py
 * (worked examples, brute force, invariants, closed forms); none is
 * "parity unpinned" except the realised Zipf shape of the synthetic router,
 * which is reported, not asserted.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { SC_F32 = 0, SC_BF16 = 1, SC_F16 = 2 };

/* ---------------------------------------------------------------- numbers */

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint16_t f32_to_bf16(float f) { /* round to nearest even */
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static float f16_to_f32(uint16_t h) {
  _Float16 v;
  memcpy(&v, &h, 2);
  return (float)v;
}

static uint16_t f32_to_f16(float f) { /* the compiler's IEEE conversion: RNE */
  _Float16 v = (_Float16)f;
  uint16_t h;
  memcpy(&h, &v, 2);
  return h;
}

static int scale_bytes(int dtype) { return dtype == SC_F32 ? 4 : 2; }

/* The scale as stored: fp32 rounded (RNE) to the scale dtype. */
static float round_scale(float s, int dtype) {
  if (dtype == SC_BF16) return bf16_to_f32(f32_to_bf16(s));
  if (dtype == SC_F16) return f16_to_f32(f32_to_f16(s));
  return s;
}

static void put_scale(void* sc, int64_t i, float s, int dtype) {
  if (dtype == SC_F32) ((float*)sc)[i] = s;
  else if (dtype == SC_BF16) ((uint16_t*)sc)[i] = f32_to_bf16(s);
  else ((uint16_t*)sc)[i] = f32_to_f16(s);
}

static float get_scale(const void* sc, int64_t i, int dtype) {
  if (dtype == SC_F32) return ((const float*)sc)[i];
  if (dtype == SC_BF16) return bf16_to_f32(((const uint16_t*)sc)[i]);
  return f16_to_f32(((const uint16_t*)sc)[i]);
}

/* ------------------------------------------------------- canonical codes */
/* Weight i of a matrix (row-major index) occupies bits [i*b, i*b + b) of a
 * little-endian bit stream; the stored value is offset binary u = q + 2^(b-1). */

static void put_code(uint8_t* codes, int64_t i, int bits, uint32_t u) {
  for (int k = 0; k < bits; ++k) {
    int64_t bit = i * bits + k;
    if ((u >> k) & 1u) codes[bit >> 3] |= (uint8_t)(1u << (bit & 7));
    else codes[bit >> 3] &= (uint8_t)~(1u << (bit & 7));
  }
}

static uint32_t get_code(const uint8_t* codes, int64_t i, int bits) {
  uint32_t u = 0;
  for (int k = 0; k < bits; ++k) {
    int64_t bit = i * bits + k;
    u |= (uint32_t)((codes[bit >> 3] >> (bit & 7)) & 1u) << k;
  }
  return u;
}

/* -------------------------------------------------------- quantisation */

static int shape_ok(int rows, int cols, int bits, int group, int dtype) {
  if (rows <= 0 || cols <= 0 || group <= 0 || cols % group) return 0;
  if (bits < 2 || bits > 8) return 0;
  if (dtype < SC_F32 || dtype > SC_F16) return 0;
  if (((int64_t)rows * cols * bits) % 8) return 0;
  return 1;
}

/* Symmetric int-b group quantisation of w [rows][cols], groups of `group`
 * consecutive weights along cols (the reduction axis):
 *   amax = max |w| over the group, s = round_dtype(amax / qmax) with
 *   qmax = 2^(b-1) - 1, q = clamp(rint(w / s), -qmax, qmax), q = 0 if s = 0.
 * rint is round-half-even; both divides are IEEE fp32.
 * Returns 0 on success, -1 on a bad shape, -2 on a non-finite scale. */
int oracle_quantize(const float* w, int rows, int cols, int bits, int group, int dtype,
                    uint8_t* codes, void* scales) {
  if (!shape_ok(rows, cols, bits, group, dtype)) return -1;
  const int qmax = (1 << (bits - 1)) - 1;
  const uint32_t off = 1u << (bits - 1);
  const int ng = cols / group;
  for (int r = 0; r < rows; ++r) {
    for (int g = 0; g < ng; ++g) {
      const float* wg = w + (int64_t)r * cols + (int64_t)g * group;
      float amax = 0.0f;
      for (int j = 0; j < group; ++j) {
        float a = fabsf(wg[j]);
        if (a > amax) amax = a;
      }
      float s = round_scale(amax / (float)qmax, dtype);
      if (!isfinite(s)) return -2;
      put_scale(scales, (int64_t)r * ng + g, s, dtype);
      for (int j = 0; j < group; ++j) {
        int q = 0;
        if (s != 0.0f) {
          float v = rintf(wg[j] / s);
          if (v > (float)qmax) v = (float)qmax;
          if (v < (float)-qmax) v = (float)-qmax;
          q = (int)v;
        }
        put_code(codes, (int64_t)r * cols + (int64_t)g * group + j, bits, (uint32_t)(q + (int)off));
      }
    }
  }
  return 0;
}

/* w_hat = q * s in fp32 (q = u - 2^(b-1)). */
int oracle_dequantize(const uint8_t* codes, const void* scales, int rows, int cols, int bits,
                      int group, int dtype, float* out) {
  if (!shape_ok(rows, cols, bits, group, dtype)) return -1;
  const int off = 1 << (bits - 1);
  const int ng = cols / group;
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < cols; ++c) {
      int64_t i = (int64_t)r * cols + c;
      int q = (int)get_code(codes, i, bits) - off;
      out[i] = (float)q * get_scale(scales, (int64_t)r * ng + c / group, dtype);
    }
  return 0;
}

/* -------------------------------------------------------------- routing */

/* Router logits in fp32, in the fixed summation order that the routing
 * contract names (so that the top-k decision is reproducible bit for bit):
 * 32 partial sums p_j, j in [0,32); p_j accumulates, starting from +0,
 * fmaf(x[i], w[i], p_j) over i = 256m + 8j + r in (m ascending, r ascending);
 * then five pairwise levels p_j <- p_j + p_(j xor d), d = 16, 8, 4, 2, 1;
 * then one fp32 add of the bias.  Requires H % 256 == 0. */
int oracle_router_logits(const uint16_t* x, int T, int H, const uint16_t* wr, int E,
                         const float* bias, float* logits) {
  if (H % 256) return -1;
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      const uint16_t* xt = x + (int64_t)t * H;
      const uint16_t* we = wr + (int64_t)e * H;
      float p[32], q[32];
      for (int j = 0; j < 32; ++j) {
        float acc = 0.0f;
        for (int m = 0; m < H / 256; ++m)
          for (int r = 0; r < 8; ++r) {
            int i = 256 * m + 8 * j + r;
            acc = fmaf(bf16_to_f32(xt[i]), bf16_to_f32(we[i]), acc);
          }
        p[j] = acc;
      }
      for (int d = 16; d >= 1; d >>= 1) {
        for (int j = 0; j < 32; ++j) q[j] = p[j] + p[j ^ d];
        memcpy(p, q, sizeof p);
      }
      float l = p[0];
      if (bias) l = l + bias[e];
      logits[(int64_t)t * E + e] = l;
    }
  return 0;
}

/* Top-k by (logit descending, expert index ascending); -0 and +0 compare
 * equal.  Weights: softmax over all E followed by renormalisation over the k
 * selected experts, which equals exp(l_j - l_max) / sum_sel exp(l_i - l_max);
 * evaluated in fp64. */
void oracle_topk(const float* logits, int T, int E, int k, int32_t* idx, double* w) {
  char* taken = (char*)malloc((size_t)E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* ties keep the lower index */
      }
      taken[best] = 1;
      idx[(int64_t)t * k + j] = best;
    }
    double lmax = l[idx[(int64_t)t * k]];
    double z = 0.0;
    for (int j = 0; j < k; ++j) z += exp((double)l[idx[(int64_t)t * k + j]] - lmax);
    for (int j = 0; j < k; ++j)
      w[(int64_t)t * k + j] = exp((double)l[idx[(int64_t)t * k + j]] - lmax) / z;
  }
  free(taken);
}

/* Group by expert: counts[e], exclusive prefix offsets[0..E], and the stable
 * order perm of slot ids s = t*k + j sorted by (expert asc, token asc);
 * inv[s] = position of s in perm. */
void oracle_permute(const int32_t* idx, int T, int E, int k, int32_t* counts, int32_t* offsets,
                    int32_t* perm, int32_t* inv) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t s = 0; s < (int64_t)T * k; ++s) counts[idx[s]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t pos = 0;
  for (int e = 0; e < E; ++e)
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (idx[(int64_t)t * k + j] == e) {
          perm[pos] = t * k + j;
          inv[t * k + j] = pos;
          ++pos;
        }
}

/* ------------------------------------------------------------------ FFN */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* One expert on one token, fp64: g = Wg x, u = Wu x (Wg, Wu [I][H]),
 * h = silu(g) * u, o = Wd h (Wd [H][I]).  Weights are the dequantised fp32
 * values, widened exactly. */
void oracle_expert_ffn(const float* wg, const float* wu, const float* wd, int H, int I,
                       const double* x, double* o) {
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < H; ++c) {
      g += (double)wg[(int64_t)i * H + c] * x[c];
      u += (double)wu[(int64_t)i * H + c] * x[c];
    }
    h[i] = silu(g) * u;
  }
  for (int r = 0; r < H; ++r) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += (double)wd[(int64_t)r * I + i] * h[i];
    o[r] = acc;
  }
  free(h);
}

/* The oracle's view of one expert: canonical codes and scales of
 * gate [I][H], up [I][H] and down [H][I]. */
typedef struct {
  const uint8_t* codes[3];
  const void* scales[3];
} oracle_expert;

/* Whole layer: logits -> top-k -> permutation -> per routed (token, expert)
 * FFN -> y[t] = sum_j w_j o_j (fp64, j ascending).  Only the experts that
 * are routed are dequantised.  Any output pointer may be NULL except y. */
int oracle_layer_forward(const oracle_expert* ex, int E, int H, int I, int k, int bits, int group,
                         int dtype, const uint16_t* x, int T, const uint16_t* wr,
                         const float* bias, float* logits_out, int32_t* idx_out, double* w_out,
                         int32_t* counts_out, int32_t* offsets_out, int32_t* perm_out,
                         int32_t* inv_out, double* y) {
  if (T < 0 || k < 1 || k > E) return -1;
  if (T == 0) return 0;
  float* logits = (float*)malloc(sizeof(float) * (size_t)T * E);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
  int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  int32_t* inv = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  float* wg = (float*)malloc(sizeof(float) * (size_t)I * H);
  float* wu = (float*)malloc(sizeof(float) * (size_t)I * H);
  float* wd = (float*)malloc(sizeof(float) * (size_t)I * H);
  double* xd = (double*)malloc(sizeof(double) * (size_t)H);
  double* o = (double*)malloc(sizeof(double) * (size_t)T * k * H); /* per slot s */
  int rc = 0;
  if (!logits || !idx || !w || !counts || !offsets || !perm || !inv || !wg || !wu || !wd || !xd ||
      !o) {
    rc = -3;
    goto done;
  }
  if (oracle_router_logits(x, T, H, wr, E, bias, logits)) { rc = -1; goto done; }
  oracle_topk(logits, T, E, k, idx, w);
  oracle_permute(idx, T, E, k, counts, offsets, perm, inv);
  for (int e = 0; e < E; ++e) {
    if (!counts[e]) continue;
    if (oracle_dequantize(ex[e].codes[0], ex[e].scales[0], I, H, bits, group, dtype, wg) ||
        oracle_dequantize(ex[e].codes[1], ex[e].scales[1], I, H, bits, group, dtype, wu) ||
        oracle_dequantize(ex[e].codes[2], ex[e].scales[2], H, I, bits, group, dtype, wd)) {
      rc = -1;
      goto done;
    }
    for (int p = offsets[e]; p < offsets[e + 1]; ++p) {
      int s = perm[p], t = s / k;
      for (int c = 0; c < H; ++c) xd[c] = (double)bf16_to_f32(x[(int64_t)t * H + c]);
      oracle_expert_ffn(wg, wu, wd, H, I, xd, o + (int64_t)s * H);
    }
  }
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < H; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += w[(int64_t)t * k + j] * o[((int64_t)t * k + j) * H + c];
      y[(int64_t)t * H + c] = acc;
    }
  if (logits_out) memcpy(logits_out, logits, sizeof(float) * (size_t)T * E);
  if (idx_out) memcpy(idx_out, idx, sizeof(int32_t) * (size_t)T * k);
  if (w_out) memcpy(w_out, w, sizeof(double) * (size_t)T * k);
  if (counts_out) memcpy(counts_out, counts, sizeof(int32_t) * (size_t)E);
  if (offsets_out) memcpy(offsets_out, offsets, sizeof(int32_t) * (size_t)(E + 1));
  if (perm_out) memcpy(perm_out, perm, sizeof(int32_t) * (size_t)T * k);
  if (inv_out) memcpy(inv_out, inv, sizeof(int32_t) * (size_t)T * k);
done:
  free(logits); free(idx); free(w); free(counts); free(offsets); free(perm); free(inv);
  free(wg); free(wu); free(wd); free(xd); free(o);
  return rc;
}

/* Selected-token variant used at full sizes: the same layer, but the FFN and
 * combine are evaluated only for the tokens listed in `tok` (n of them);
 * y is [n][H].  Routing is computed for all T tokens. */
int oracle_layer_forward_tokens(const oracle_expert* ex, int E, int H, int I, int k, int bits,
                                int group, int dtype, const uint16_t* x, int T,
                                const uint16_t* wr, const float* bias, const int32_t* tok, int n,
                                double* y) {
  float* logits = (float*)malloc(sizeof(float) * (size_t)T * E);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
  float* wg = (float*)malloc(sizeof(float) * (size_t)I * H);
  float* wu = (float*)malloc(sizeof(float) * (size_t)I * H);
  float* wd = (float*)malloc(sizeof(float) * (size_t)I * H);
  double* xd = (double*)malloc(sizeof(double) * (size_t)H);
  double* o = (double*)malloc(sizeof(double) * (size_t)H);
  int rc = 0;
  if (!logits || !idx || !w || !wg || !wu || !wd || !xd || !o) { rc = -3; goto done; }
  if (oracle_router_logits(x, T, H, wr, E, bias, logits)) { rc = -1; goto done; }
  oracle_topk(logits, T, E, k, idx, w);
  for (int a = 0; a < n; ++a) {
    int t = tok[a];
    if (t < 0 || t >= T) { rc = -1; goto done; }
    for (int c = 0; c < H; ++c) {
      xd[c] = (double)bf16_to_f32(x[(int64_t)t * H + c]);
      y[(int64_t)a * H + c] = 0.0;
    }
    for (int j = 0; j < k; ++j) {
      int e = idx[(int64_t)t * k + j];
      if (oracle_dequantize(ex[e].codes[0], ex[e].scales[0], I, H, bits, group, dtype, wg) ||
          oracle_dequantize(ex[e].codes[1], ex[e].scales[1], I, H, bits, group, dtype, wu) ||
          oracle_dequantize(ex[e].codes[2], ex[e].scales[2], H, I, bits, group, dtype, wd)) {
        rc = -1;
        goto done;
      }
      oracle_expert_ffn(wg, wu, wd, H, I, xd, o);
      for (int c = 0; c < H; ++c) y[(int64_t)a * H + c] += w[(int64_t)t * k + j] * o[c];
    }
  }
done:
  free(logits); free(idx); free(w); free(wg); free(wu); free(wd); free(xd); free(o);
  return rc;
}

/* --------------------------------------------------------- expert cache */
/* Frequency-admitted HBM expert cache ("Running a 24k-expert MoE ...",
 * section 2: the cache adapts to what is used; section 3: ~70% of experts
 * give 97.8-99.7% hits).  One global pool of C slots, empty at start.
 *
 * access[(s*L + l)*maxd + i] lists the distinct experts (ids in [0, E),
 * -1 = unused entry) touched by layer l in step s.  Global id g = l*E + e.
 *
 * Per access: hit iff g is resident at the start of the step;
 * count[g] += 1; last[g] = s; a miss is queued.
 * At the end of step s, the queued misses are processed in (layer, expert)
 * ascending order: a free slot (lowest index) admits the miss; otherwise the
 * victim is the resident expert not accessed in step s with the smallest
 * (count, last, g), and the miss is admitted into the victim's slot iff
 * count[miss] > count[victim] (ties keep the incumbent).  When aging_period
 * > 0, every count is halved after each aging_period-th step.
 *
 * Outputs (any may be NULL): per-(step, layer) hits and misses, totals of
 * admissions and evictions, and the final owner of each slot (-1 = free). */
int oracle_cache_sim(int L, int E, int64_t C, int steps, const int32_t* access, int maxd,
                     int aging_period, int32_t* hits_sl, int32_t* misses_sl, int64_t* admissions,
                     int64_t* evictions, int32_t* slot_owner_out) {
  const int64_t G = (int64_t)L * E;
  int64_t* slot_of = (int64_t*)malloc(sizeof(int64_t) * (size_t)G);
  int64_t* count = (int64_t*)calloc((size_t)G, sizeof(int64_t));
  int64_t* last = (int64_t*)malloc(sizeof(int64_t) * (size_t)G);
  int64_t* owner = (int64_t*)malloc(sizeof(int64_t) * (size_t)(C > 0 ? C : 1));
  int64_t* missq = (int64_t*)malloc(sizeof(int64_t) * (size_t)L * (maxd > 0 ? maxd : 1));
  int rc = 0;
  if (!slot_of || !count || !last || !owner || !missq) { rc = -3; goto done; }
  for (int64_t g = 0; g < G; ++g) { slot_of[g] = -1; last[g] = -1; }
  for (int64_t c = 0; c < C; ++c) owner[c] = -1;
  int64_t adm = 0, evi = 0;
  for (int s = 0; s < steps; ++s) {
    int64_t nm = 0;
    for (int l = 0; l < L; ++l) {
      int32_t h = 0, m = 0;
      for (int i = 0; i < maxd; ++i) {
        int32_t e = access[((int64_t)s * L + l) * maxd + i];
        if (e < 0) continue;
        if (e >= E) { rc = -1; goto done; }
        int64_t g = (int64_t)l * E + e;
        if (slot_of[g] >= 0) ++h;
        else { ++m; missq[nm++] = g; }
        count[g] += 1;
        last[g] = s;
      }
      if (hits_sl) hits_sl[(int64_t)s * L + l] = h;
      if (misses_sl) misses_sl[(int64_t)s * L + l] = m;
    }
    /* (layer, expert) ascending == global id ascending; insertion sort */
    for (int64_t a = 1; a < nm; ++a) {
      int64_t v = missq[a], b = a - 1;
      while (b >= 0 && missq[b] > v) { missq[b + 1] = missq[b]; --b; }
      missq[b + 1] = v;
    }
    for (int64_t a = 0; a < nm; ++a) {
      int64_t g = missq[a];
      if (slot_of[g] >= 0) continue; /* already admitted (repeated access) */
      int64_t freec = -1;
      for (int64_t c = 0; c < C; ++c)
        if (owner[c] < 0) { freec = c; break; }
      if (freec >= 0) {
        owner[freec] = g;
        slot_of[g] = freec;
        ++adm;
        continue;
      }
      int64_t victim = -1;
      for (int64_t c = 0; c < C; ++c) {
        int64_t v = owner[c];
        if (last[v] == s) continue; /* accessed this step: not evictable */
        if (victim < 0 || count[v] < count[victim] ||
            (count[v] == count[victim] && last[v] < last[victim]) ||
            (count[v] == count[victim] && last[v] == last[victim] && v < victim))
          victim = v;
      }
      if (victim < 0) continue;
      if (count[g] > count[victim]) {
        int64_t c = slot_of[victim];
        slot_of[victim] = -1;
        owner[c] = g;
        slot_of[g] = c;
        ++adm;
        ++evi;
      }
    }
    if (aging_period > 0 && (s + 1) % aging_period == 0)
      for (int64_t g = 0; g < G; ++g) count[g] >>= 1;
  }
  if (admissions) *admissions = adm;
  if (evictions) *evictions = evi;
  if (slot_owner_out)
    for (int64_t c = 0; c < C; ++c) slot_owner_out[c] = (int32_t)owner[c];
done:
  free(slot_of); free(count); free(last); free(owner); free(missq);
  return rc;
}
