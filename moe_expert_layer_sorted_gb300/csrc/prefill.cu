// Prefill-batch forward (T > 8 tokens), the shape of "763B MoE in two 96 GB
// cards" (section "Where the VRAM gap comes from": each token routed to k of
// E experts, the layer output the routing-weighted sum of the experts'
// SwiGLU FFNs), as a chain of launches on the caller's stream:
//
//   1. routing, the top-k of the router logits in the library's fixed
//      summation order (lane j of a warp owns elements 256m + 8j + r;
//      xor-butterfly; bias last), ties -> lower expert index, softmax
//      renormalised over the k:
//      - a bf16 cuBLAS GEMM for approximate logits, then pf_select_kernel (one
//        warp per token): a rigorous bound on each approximate logit's
//        distance to the fixed-order one, the fixed-order logits of the
//        experts that can still reach the top-k only, the top-k over those
//        (see "bounded router" below);
//      - or, when the caller asks for the logits, pf_router_kernel (every
//        logit in the fixed order, tiled 32 tokens x 16 experts per CTA,
//        8 x 8 per warp, operands staged as bf16 with cp.async in a
//        four-block ring) and pf_topk_kernel.
//   2. pf_bucket_count / pf_bucket_scan / pf_bucket_place
//                         grouping by expert: a stable counting sort of the
//                         slots (per-block expert histograms, one prefix over
//                         (expert, block), placement in slot order) giving
//                         per-expert counts, offsets and the (expert, token)
//                         order perm / inv.
//   3. pf_gather_kernel   the layer input's rows copied into grouped
//                         (expert, token) order, columns in the GEMMs' stage
//                         K order.
//   4. pf_gemm_kernel<gate/up>  for every routed (expert, 128 of its tokens,
//                         128 rows of I): gate and up projections on tcgen05
//                         tensor cores (M = 128 tokens, N = 128 gate + 128 up
//                         rows) with fp32 accumulators in TMEM; the epilogue
//                         writes h = silu(g) * u (bf16) per (token, expert) slot.
//   5. pf_gemm_kernel<down>  o = Wd h per (expert, 128 tokens, 256 rows of H),
//                         times the slot's routing weight, bf16 per slot.
//   6. pf_combine_kernel  y[t] = sum over j ascending of the slot outputs, bf16.
//   7. pf_stats_kernel    the forward's accounting.
//
// GEMM kernel layout (one CTA of 23 warps per SM, persistent over work units,
// consecutive units of an expert sharing its token tile):
//   warps 0-15  dequantise: warp w turns 16 weight rows x 64 columns per stage
//               (int-b codes in the library's fragment-ordered device layout ->
//               bf16 s*q) into a 128-byte-swizzled K-major shared-memory tile;
//   warp 20     per stage the 128 token rows x 64 columns (one 2-D tensor
//               copy, 128-byte swizzle);
//   warp 21     per 256-column code block the unit's codes and scales (bulk
//               copies from HBM, 16-byte cp.async from pinned host memory);
//   warp 22     allocates TMEM and (lane 0) issues tcgen05.mma (K = 16 per
//               instruction) per stage, releasing both stage buffers by
//               tcgen05.commit; two accumulators of 256 columns alternate
//               between units;
//   warps 16-19 epilogue: tcgen05.ld of the accumulator (warp 16+q reads TMEM
//               lanes 32q..32q+31, i.e. tokens), activation / scaling, 16-byte
//               global stores.
// Stages and the accumulator hand-off are tracked by mbarriers; every wait is
// bounded and latches the plan's error word.
#include <stdio.h>

#include <cuda.h>

#include <algorithm>

#include "internal.h"

using namespace moe;

namespace {

#include "device_common.cuh"

// ------------------------------------------------------------------ router

constexpr int kRtTok = 32, kRtExp = 16;  // tokens and experts per router CTA (8 warps of 8 x 8)
constexpr int kRtStages = 4;             // 256-column blocks in flight (cp.async ring)
constexpr size_t kRtStageBytes = (size_t)(kRtTok + kRtExp) * 32 * 16;
constexpr size_t kRtSmem = kRtStages * kRtStageBytes;

// acc + x * w for the low (or high) bf16 halves of x and w, widened to fp32:
// the product of two bf16 values is exact in fp32, so the one rounding of this
// mixed-precision fma equals that of fmaf on the widened operands (bit for bit)
// without the two widening instructions.
__device__ __forceinline__ float fma_bf16_lo(uint32_t x, uint32_t w, float c) {
  asm("{\n .reg .b16 xl, xh, wl, wh;\n mov.b32 {xl, xh}, %1;\n mov.b32 {wl, wh}, %2;\n"
      " fma.rn.f32.bf16 %0, xl, wl, %0;\n}"
      : "+f"(c)
      : "r"(x), "r"(w));
  return c;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t x, uint32_t w, float c) {
  asm("{\n .reg .b16 xl, xh, wl, wh;\n mov.b32 {xl, xh}, %1;\n mov.b32 {wl, wh}, %2;\n"
      " fma.rn.f32.bf16 %0, xh, wh, %0;\n}"
      : "+f"(c)
      : "r"(x), "r"(w));
  return c;
}

// Operands staged as bf16: row r of a 256-column block m holds, at uint4
// index j, the elements 256m + 8j .. 256m + 8j + 7 (lane j's share in the
// fixed order), so a lane's 16-byte reads are conflict-free.  A ring of
// kRtStages blocks: block m + kRtStages - 1 is requested (cp.async) while
// block m is used; one barrier per block.
__global__ void __launch_bounds__(256) pf_router_kernel(const uint16_t* __restrict__ x, int T, int H,
                                                        const uint16_t* __restrict__ wr,
                                                        const float* __restrict__ bias, int E,
                                                        float* __restrict__ logits) {
  extern __shared__ __align__(16) uint4 rsm[];  // [stage][kRtTok + kRtExp rows][32]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kRtTok, e0 = blockIdx.y * kRtExp;
  const int tw = (warp & 3) * 8, ew = (warp >> 2) * 8;  // warp tile: 8 tokens x 8 experts
  const int nm = H / 256;
  // 48 rows x 32 pieces of 16 bytes per block, 6 per thread; rows past T or E read as zero
  auto stage = [&](int m) {
    uint4* buf = rsm + (size_t)(m % kRtStages) * (kRtTok + kRtExp) * 32;
#pragma unroll
    for (int i = 0; i < 6; ++i) {
      const int c = tid + i * 256, row = c >> 5, j = c & 31;
      const bool isx = row < kRtTok;
      const int g = isx ? t0 + row : e0 + row - kRtTok;
      uint4* dst = buf + row * 32 + j;
      if (g < (isx ? T : E)) cp_async16(dst, (isx ? x : wr) + (int64_t)g * H + m * 256 + j * 8);
      else *dst = make_uint4(0, 0, 0, 0);
    }
  };
  float acc[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
#pragma unroll
  for (int m = 0; m < kRtStages - 1; ++m) {  // one commit group per block (empty past the end)
    if (m < nm) stage(m);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int m = 0; m < nm; ++m) {
    asm volatile("cp.async.wait_group %0;" ::"n"(kRtStages - 2) : "memory");  // block m has landed
    __syncthreads();  // ... for every thread, and block m - 1's buffer is free
    if (m + kRtStages - 1 < nm) stage(m + kRtStages - 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const uint4* xs = rsm + (size_t)(m % kRtStages) * (kRtTok + kRtExp) * 32;
    const uint4* ws = xs + kRtTok * 32;
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // elements 4h .. 4h+3 of the lane's eight
      uint2 xv[8], wv[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) xv[a] = reinterpret_cast<const uint2*>(&xs[(tw + a) * 32 + lane])[h];
#pragma unroll
      for (int b = 0; b < 8; ++b) wv[b] = reinterpret_cast<const uint2*>(&ws[(ew + b) * 32 + lane])[h];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const uint32_t wu = (r < 2) ? wv[b].x : wv[b].y;
#pragma unroll
          for (int a = 0; a < 8; ++a) {
            const uint32_t xu = (r < 2) ? xv[a].x : xv[a].y;
            acc[a][b] = (r & 1) ? fma_bf16_hi(xu, wu, acc[a][b]) : fma_bf16_lo(xu, wu, acc[a][b]);
          }
        }
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      float v = acc[a][b];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
      const int t = t0 + tw + a, e = e0 + ew + b;
      if (lane == ((a * 8 + b) & 31) && t < T && e < E) logits[(int64_t)t * E + e] = v + bias[e];
    }
}

// Order-preserving key of a logit (-0 and +0 equal): a > b  <=>  key(a) > key(b).
__device__ __forceinline__ uint32_t logit_key(float v) {
  const uint32_t ub = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (ub & 0x80000000u) ? ~ub : (ub | 0x80000000u);
}

// The k largest entries of a token's logit row l[0..E) (one warp): k rounds of
// (lane's best untaken logit, warp max by key, warp min of the index among the
// lanes holding it); lanes scan experts lane, lane+32, ... so ties resolve to
// the lower index.  chosen[j], cv[j]: expert and logit of rank j, every lane.
__device__ void row_topk(const float* l, int E, int k, int lane, int* chosen, float* cv) {
  if (E <= 16 * 32) {  // the lane's logits (experts lane, lane + 32, ...) held in registers
    float vb[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) vb[q] = q * 32 + lane < E ? l[q * 32 + lane] : 0.0f;
    uint32_t taken = 0u;
    for (int j = 0; j < k; ++j) {
      uint32_t best = 0u;
      float bv = 0.0f;
      int bq = -1;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float v = vb[q];
        const uint32_t key = logit_key(v);
        if (q * 32 + lane < E && !((taken >> q) & 1u) && (bq < 0 || key > best)) {  // ascending e: ties keep the lower
          best = key;
          bv = v;
          bq = q;
        }
      }
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, bq < 0 ? 0u : best);
      const uint32_t mine = (bq >= 0 && best == kmax) ? (uint32_t)(bq * 32 + lane) : 0xffffffffu;
      const int win = (int)__reduce_min_sync(0xffffffffu, mine);
      if (bq >= 0 && bq * 32 + lane == win) taken |= 1u << bq;
      chosen[j] = win;
      cv[j] = __shfl_sync(0xffffffffu, bv, win & 31);
    }
    return;
  }
  for (int j = 0; j < k; ++j) {
    uint32_t best = 0u;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      bool taken = false;
      for (int q = 0; q < j; ++q) taken |= chosen[q] == e;
      if (taken) continue;
      const uint32_t key = logit_key(l[e]);
      if (bi == 0x7fffffff || key > best) {  // ascending e: ties keep the lower index
        best = key;
        bi = e;
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bi == 0x7fffffff ? 0u : best);
    const uint32_t mine = (bi != 0x7fffffff && best == kmax) ? (uint32_t)bi : 0xffffffffu;
    const int win = (int)__reduce_min_sync(0xffffffffu, mine);
    chosen[j] = win;
    cv[j] = l[win];
  }
}

// Lane 0: the token's experts and their weights, the softmax of the k chosen
// logits renormalised over the k.
__device__ __forceinline__ void write_routing(int64_t t, int k, int lane, const int* chosen, const float* cv,
                                              int32_t* idx, float* wout) {
  if (lane != 0) return;
  float ex[kMaxTopK];
  float z = 0.0f;
  for (int j = 0; j < k; ++j) {
    ex[j] = expf(cv[j] - cv[0]);
    z += ex[j];
  }
  for (int j = 0; j < k; ++j) {
    idx[t * k + j] = chosen[j];
    wout[t * k + j] = ex[j] / z;
  }
}

// One warp per token: top-k of the exact logit row, then the weights.
__global__ void pf_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                               int32_t* __restrict__ idx, float* __restrict__ wout) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  int chosen[kMaxTopK];
  float cv[kMaxTopK];
  row_topk(logits + (int64_t)t * E, E, k, lane, chosen, cv);
  write_routing(t, k, lane, chosen, cv, idx, wout);
}

// ------------------------------------------------------------------ bounded router
// Routing with the router logits on tensor cores.  A bf16 GEMM (cuBLAS, fp32
// accumulation, any internal order) gives approximate logits a[t][e]; the
// top-k must be that of the library's fixed-order fp32 logits F[t][e] (the
// order of pf_router_kernel), so a rigorous bound |a + b_e - F| <= d[t][e]
// decides which experts can still be among the k largest F, and only those
// are recomputed in the fixed order.
//
// The bound.  Every product x_i w_i of two bf16 values is exact in fp32.  An
// fp32 accumulation that adds blocks of n products to a running sum, aligning
// the n + 1 terms to the largest exponent and dropping the bits below it (no
// guard bits, truncation: the weakest tensor-core adder model), errs per
// block by less than (n + 1) ulp of its largest term, so over H / n blocks by
// less than H (n + 1) / n 2^-23 sum|x_i w_i| <= H 2^-22 sum|x_i w_i|; the
// fixed-order sum (chains of H / 32 fmas and five butterfly adds, round to
// nearest) errs by at most (H / 32 + 5) 2^-24 sum|x_i w_i|; adding the bias on
// either side rounds once more (2^-24 of |a| + |b|).  With
// sum|x_i w_i| <= ||x|| ||w|| (Cauchy-Schwarz),
//     d[t][e] = H 2^-20 ||x_t|| ||w_e|| + 2^-21 |b_e| + 2^-100
// (norms rounded up, products and sums rounded up) is four times the sum of
// those terms; the 2^-100 covers products flushed to zero on the tensor cores.
// With lo = a + b - d, hi = a + b + d (rounded down / up) and tau the k-th
// largest lo, an expert with hi < tau lies strictly below k experts whose
// F >= lo >= tau, so it is not among the k largest nor tied with them; the
// rest (the candidates, at least k) get their fixed-order logit, and the k
// rounds of the top-k over the candidates take exactly the choices the rounds
// over all E would.  A token whose bounds are not all finite and below 1e37,
// or with more than kCand candidates, has all E logits recomputed.

constexpr int kCand = 64;  // candidates per token held by the warp (two per lane)

// Upper bound of the 2-norm of a bf16 row of length H (H a multiple of 256), one warp.
__device__ __forceinline__ float row_norm_ru(const uint16_t* __restrict__ r, int H, int lane) {
  float s = 0.0f;
#pragma unroll 4
  for (int c = lane * 8; c < H; c += 256) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(r + c));
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = __uint_as_float(u[i] << 16), hi = __uint_as_float(u[i] & 0xffff0000u);
      s = __fmaf_ru(lo, lo, s);
      s = __fmaf_ru(hi, hi, s);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) s = __fadd_ru(s, __shfl_xor_sync(0xffffffffu, s, o));
  return __fsqrt_ru(s);
}

__global__ void __launch_bounds__(256) router_norm_kernel(const uint16_t* __restrict__ wr, int E, int H,
                                                          float* __restrict__ out) {
  const int lane = threadIdx.x & 31, e = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e >= E) return;
  const float v = row_norm_ru(wr + (int64_t)e * H, H, lane);
  if (lane == 0) out[e] = v;
}

// Fixed-order router logits of experts e4[0..3] for the token row xr: lane j
// accumulates elements 256m + 8j + r (m, then r ascending) with one rounding
// per fma, the xor butterfly, then the bias -- the arithmetic of
// pf_router_kernel, so the results are the same bits.
__device__ __forceinline__ void exact_logits4(const uint16_t* __restrict__ xr, const uint16_t* __restrict__ wr,
                                              const float* __restrict__ bias, int H, int lane, const int (&e4)[4],
                                              float (&v4)[4]) {
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 2
  for (int c = lane * 8; c < H; c += 256) {
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xr + c));
    uint4 wv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) wv[j] = __ldg(reinterpret_cast<const uint4*>(wr + (int64_t)e4[j] * H + c));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[j] = fma_bf16_lo(xv.x, wv[j].x, acc[j]);
      acc[j] = fma_bf16_hi(xv.x, wv[j].x, acc[j]);
      acc[j] = fma_bf16_lo(xv.y, wv[j].y, acc[j]);
      acc[j] = fma_bf16_hi(xv.y, wv[j].y, acc[j]);
      acc[j] = fma_bf16_lo(xv.z, wv[j].z, acc[j]);
      acc[j] = fma_bf16_hi(xv.z, wv[j].z, acc[j]);
      acc[j] = fma_bf16_lo(xv.w, wv[j].w, acc[j]);
      acc[j] = fma_bf16_hi(xv.w, wv[j].w, acc[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float v = acc[j];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
    v4[j] = v + bias[e4[j]];
  }
}

// One warp per token.  NQ > 0: the lane's bounds (experts lane, lane + 32, ...)
// held in registers, E <= 32 NQ; NQ = 0: recomputed from memory (any E).
// lg [T][E] holds the approximate dot products on entry (the bias not yet
// added); rows of tokens that take the full path are overwritten with their
// exact logits.  exact_count += fixed-order logits computed.
template <int NQ>
__global__ void __launch_bounds__(256) pf_select_kernel(const uint16_t* __restrict__ x, int T, int H,
                                                        const uint16_t* __restrict__ wr,
                                                        const float* __restrict__ bias,
                                                        const float* __restrict__ wnorm, int E, int k,
                                                        float* __restrict__ lg, int32_t* __restrict__ idx,
                                                        float* __restrict__ wout,
                                                        unsigned long long* __restrict__ exact_count) {
  __shared__ int cand_e[8][kCand];
  __shared__ float cand_v[8][kCand], cand_h[8][kCand];
  __shared__ int nexact[8];
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + wp;
  if (lane == 0) nexact[wp] = 0;
  if (t < T) {
    const uint16_t* xr = x + (int64_t)t * H;
    float* row = lg + (int64_t)t * E;
    const float nx = row_norm_ru(xr, H, lane);
    const float dx = __fmul_ru((float)H * 0x1p-20f, nx);
    auto bounds = [&](int e, float& lo, float& hi) -> bool {
      const float b = bias[e], nw = wnorm[e];
      const float a = row[e] + b;
      const float d = __fmaf_ru(dx, nw, __fmaf_ru(0x1p-21f, fabsf(b), 0x1p-100f));
      lo = __fsub_rd(a, d);
      hi = __fadd_ru(a, d);
      return __fmul_ru(nx, nw) < 1e37f && fabsf(b) < 1e37f && fabsf(a) < 1e37f && d < 1e37f;
    };
    constexpr bool R = NQ > 0;
    float lo_r[R ? NQ : 1], hi_r[R ? NQ : 1];
    bool ok = true;
    if constexpr (R) {
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        lo_r[q] = hi_r[q] = 0.0f;
        if (q * 32 + lane < E) ok &= bounds(q * 32 + lane, lo_r[q], hi_r[q]);
      }
    } else {
      for (int e = lane; e < E; e += 32) {
        float lo, hi;
        ok &= bounds(e, lo, hi);
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    int n = kCand + 1;  // candidates; > kCand: the full path
    if (ok) {
      // tau = the k-th largest lo, counted with multiplicity: rounds of (largest
      // key below the previous round's, how many experts hold it)
      uint32_t cur = 0xffffffffu, tau = 0u;
      int need = k;
      for (int r = 0; r < k; ++r) {
        uint32_t best = 0u;
        if constexpr (R) {
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            const uint32_t key = logit_key(lo_r[q]);
            if (q * 32 + lane < E && key < cur && key > best) best = key;
          }
        } else {
          for (int e = lane; e < E; e += 32) {
            float lo, hi;
            bounds(e, lo, hi);
            const uint32_t key = logit_key(lo);
            if (key < cur && key > best) best = key;
          }
        }
        const uint32_t m = __reduce_max_sync(0xffffffffu, best);
        uint32_t c = 0;
        if constexpr (R) {
#pragma unroll
          for (int q = 0; q < NQ; ++q) c += (q * 32 + lane < E && logit_key(lo_r[q]) == m) ? 1u : 0u;
        } else {
          for (int e = lane; e < E; e += 32) {
            float lo, hi;
            bounds(e, lo, hi);
            c += logit_key(lo) == m ? 1u : 0u;
          }
        }
        c = __reduce_add_sync(0xffffffffu, c);
        tau = m;
        if ((int)c >= need) break;
        need -= (int)c;
        cur = m;
      }
      // candidates hi >= tau, in ascending expert order
      n = 0;
      const int nq = R ? NQ : (E + 31) / 32;
#pragma unroll
      for (int q = 0; q < nq; ++q) {
        const int e = q * 32 + lane;
        float hi = 0.0f;
        if constexpr (R) {
          hi = hi_r[q];
        } else if (e < E) {
          float lo;
          bounds(e, lo, hi);
        }
        const bool in = e < E && logit_key(hi) >= tau;
        const uint32_t bal = __ballot_sync(0xffffffffu, in);
        const int pos = n + __popc(bal & ((1u << lane) - 1u));
        if (in && pos < kCand) {
          cand_e[wp][pos] = e;
          cand_h[wp][pos] = hi;
        }
        n += __popc(bal);
      }
      if (n < k) n = kCand + 1;  // cannot happen (the k experts defining tau are candidates)
    }
    __syncwarp();
    int chosen[kMaxTopK];
    float cv[kMaxTopK];
    int nev = n;  // fixed-order logits computed for this token
    if (n <= kCand) {
      // Fixed-order logits in rounds, the candidates with the largest upper
      // bounds first, until every candidate not computed has an upper bound
      // below the k-th largest computed logit: such a candidate lies strictly
      // below k computed experts, so the top-k over the computed ones is the
      // top-k over all (same choices, same order).  Slots lane and lane + 32.
      const bool s0 = lane < n, s1 = lane + 32 < n;
      const uint32_t hk0 = s0 ? logit_key(cand_h[wp][lane]) : 0u;
      const uint32_t hk1 = s1 ? logit_key(cand_h[wp][lane + 32]) : 0u;
      uint64_t evm = 0;  // slots computed (the same in every lane)
      int batch = min(8, (k + 5) & ~3);
      nev = 0;
      while (true) {
        int pick[8];
        int np = 0;
        for (int b = 0; b < batch && nev + np < n; ++b) {  // largest bound first, ties: lower slot
          const bool a0 = s0 && !((evm >> lane) & 1ull), a1 = s1 && !((evm >> (lane + 32)) & 1ull);
          uint32_t best = 0u;
          int bs = -1;
          if (a0) {
            best = hk0;
            bs = lane;
          }
          if (a1 && (bs < 0 || hk1 > best)) {
            best = hk1;
            bs = lane + 32;
          }
          const uint32_t km = __reduce_max_sync(0xffffffffu, bs < 0 ? 0u : best);
          const int win = (int)__reduce_min_sync(0xffffffffu, (bs >= 0 && best == km) ? (uint32_t)bs : 0xffffffffu);
          pick[np++] = win;
          evm |= 1ull << win;
        }
        for (int c = 0; c < np; c += 4) {
          int e4[4], s4[4];
          float v4[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            s4[j] = pick[min(c + j, np - 1)];
            e4[j] = cand_e[wp][s4[j]];
          }
          exact_logits4(xr, wr, bias, H, lane, e4, v4);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (lane == j && c + j < np) cand_v[wp][s4[j]] = v4[j];
        }
        nev += np;
        __syncwarp();
        if (nev >= n) break;
        // the k-th largest computed logit, counted with multiplicity (nev >= k)
        const bool c0 = s0 && ((evm >> lane) & 1ull), c1 = s1 && ((evm >> (lane + 32)) & 1ull);
        const uint32_t vk0 = c0 ? logit_key(cand_v[wp][lane]) : 0u, vk1 = c1 ? logit_key(cand_v[wp][lane + 32]) : 0u;
        uint32_t cur = 0xffffffffu, kth = 0u;
        int need = k;
        for (int r = 0; r < k; ++r) {
          uint32_t best = 0u;
          if (c0 && vk0 < cur && vk0 > best) best = vk0;
          if (c1 && vk1 < cur && vk1 > best) best = vk1;
          const uint32_t m = __reduce_max_sync(0xffffffffu, best);
          const uint32_t cnt = __reduce_add_sync(0xffffffffu, (c0 && vk0 == m ? 1u : 0u) + (c1 && vk1 == m ? 1u : 0u));
          kth = m;
          if ((int)cnt >= need) break;
          need -= (int)cnt;
          cur = m;
        }
        // the largest upper bound among the candidates not computed
        uint32_t hu = 0u;
        if (s0 && !c0) hu = hk0;
        if (s1 && !c1 && hk1 > hu) hu = hk1;
        hu = __reduce_max_sync(0xffffffffu, hu);
        if (hu < kth) break;
        batch = 4;
      }
      // top-k over the computed candidates (slot lane, then lane + 32: ascending expert)
      const bool h0 = s0 && ((evm >> lane) & 1ull), h1 = s1 && ((evm >> (lane + 32)) & 1ull);
      const int e0 = h0 ? cand_e[wp][lane] : 0, e1 = h1 ? cand_e[wp][lane + 32] : 0;
      const float v0 = h0 ? cand_v[wp][lane] : 0.0f, v1 = h1 ? cand_v[wp][lane + 32] : 0.0f;
      bool tk0 = false, tk1 = false;
      for (int j = 0; j < k; ++j) {
        uint32_t best = 0u;
        int be = -1, bs = 0;
        float bv = 0.0f;
        if (h0 && !tk0) {
          best = logit_key(v0);
          be = e0;
          bv = v0;
        }
        if (h1 && !tk1 && (be < 0 || logit_key(v1) > best)) {  // ties keep the lower expert
          best = logit_key(v1);
          be = e1;
          bv = v1;
          bs = 1;
        }
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, be < 0 ? 0u : best);
        const uint32_t mine = (be >= 0 && best == kmax) ? (uint32_t)be : 0xffffffffu;
        const int win = (int)__reduce_min_sync(0xffffffffu, mine);
        const bool own = be >= 0 && be == win;
        if (own) (bs ? tk1 : tk0) = true;
        const int wl = __ffs(__ballot_sync(0xffffffffu, own)) - 1;
        chosen[j] = win;
        cv[j] = __shfl_sync(0xffffffffu, bv, wl);
      }
    } else {  // the full path: every logit in the fixed order, then the plain top-k
      n = E;
      for (int c = 0; c < E; c += 4) {
        int e4[4];
        float v4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) e4[j] = min(c + j, E - 1);
        exact_logits4(xr, wr, bias, H, lane, e4, v4);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (lane == j && c + j < E) row[c + j] = v4[j];
      }
      __syncwarp();
      row_topk(row, E, k, lane, chosen, cv);
      nev = E;
    }
    write_routing(t, k, lane, chosen, cv, idx, wout);
    if (lane == 0) nexact[wp] = nev;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long s = 0;
    for (int w = 0; w < 8; ++w) s += (unsigned long long)nexact[w];
    atomicAdd(exact_count, s);
  }
}

// ------------------------------------------------------------------ grouping
// A stable counting sort of the n = T*k slots by expert, in blocks of
// kGroupChunk consecutive slots:
//   pf_bucket_count  per block, the number of its slots routed to each expert;
//   pf_bucket_scan   exclusive prefix over (expert, block), expert-major: the
//                    first perm position of block b's slots of expert e; the
//                    per-expert counts and offsets;
//   pf_bucket_place  per block, warp w takes slots 256w..256w+255 of the block
//                    in 32-slot rounds; a slot's position = its block's base
//                    for its expert + the earlier warps' count + the slots of
//                    its expert before it in its warp (match_any / popc).
// Every slot lands in ascending (expert, slot) order: the order the oracle's
// stable grouping defines.

__global__ void __launch_bounds__(256) pf_bucket_count(const int32_t* __restrict__ idx, int n, int E,
                                                       int32_t* __restrict__ bucket) {
  extern __shared__ int32_t hist[];  // [E]
  const int nb = gridDim.x, b = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int s0 = b * kGroupChunk, s1 = min(n, s0 + kGroupChunk);
  for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) atomicAdd(&hist[idx[s]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) bucket[(int64_t)e * nb + b] = hist[e];
}

__global__ void __launch_bounds__(1024) pf_bucket_scan(int32_t* __restrict__ bucket, int E, int nb,
                                                       int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  __shared__ int32_t part[1024];
  const int tid = threadIdx.x;
  const int64_t len = (int64_t)E * nb;
  const int64_t per = (len + 1023) / 1024;
  const int64_t i0 = tid * per, i1 = min(len, i0 + per);
  int32_t sum = 0;
  for (int64_t i = i0; i < i1; ++i) sum += bucket[i];
  part[tid] = sum;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {  // inclusive scan of the 1024 partial sums
    const int32_t v = tid >= o ? part[tid - o] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int32_t run = tid ? part[tid - 1] : 0;
  for (int64_t i = i0; i < i1; ++i) {  // counts -> exclusive bases
    const int32_t c = bucket[i];
    bucket[i] = run;
    run += c;
  }
  __syncthreads();
  for (int e = tid; e < E; e += 1024) {
    const int32_t first = bucket[(int64_t)e * nb];
    const int32_t next = e + 1 < E ? bucket[(int64_t)(e + 1) * nb] : part[1023];
    offsets[e] = first;
    counts[e] = next - first;
  }
  if (tid == 0) offsets[E] = part[1023];
}

__global__ void __launch_bounds__(256) pf_bucket_place(const int32_t* __restrict__ idx, int n, int E,
                                                       const int32_t* __restrict__ bucket,
                                                       int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  extern __shared__ int32_t wcnt[];  // [8 warps][E]
  const int nb = gridDim.x, b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int w0 = b * kGroupChunk + warp * (kGroupChunk / 8);
  const int w1 = min(n, w0 + kGroupChunk / 8);
  int32_t* mine = wcnt + warp * E;
  for (int s0 = w0; s0 < w1; s0 += 32) {  // this warp's count per expert
    const int s = s0 + lane;
    const int e = s < w1 ? idx[s] : -1;
    const unsigned m = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (m & lt) == 0) mine[e] += __popc(m);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {  // -> each warp's first position per expert
    int32_t run = bucket[(int64_t)e * nb + b];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int32_t c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int s0 = w0; s0 < w1; s0 += 32) {
    const int s = s0 + lane;
    const int e = s < w1 ? idx[s] : -1;
    const unsigned m = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int pos = mine[e] + __popc(m & lt);
      perm[pos] = s;
      inv[s] = pos;
    }
    __syncwarp();
    if (e >= 0 && (m & lt) == 0) mine[e] += __popc(m);
    __syncwarp();
  }
}

// ------------------------------------------------------------------ token rows in (expert, token) order

// K order of the GEMM operands within each 64-column stage.  Word w (columns
// 2w, 2w+1) of a stage's half h (columns 32h..32h+31) is written as
// w = 8 kk1 + 4 m + j with j < 4, kk1, m < 2 -- MMA step 2h + kk1 and, within
// the step, columns 2j + 8m, 2j + 8m + 1; it is placed at physical word
// 8 j + 4 h + 2 kk1 + m of the stage.  So physical 16-byte chunk 2j + h holds
// exactly what dequantising lane j (tig = j) produces for its row in MMA steps
// 2h and 2h+1 (its mma.m16n8k16 A-fragment columns), one 16-byte store, and a
// quarter warp's eight stores hit eight different chunks of the swizzled rows.
// The token rows (pf_gather_kernel) and h (the gate/up epilogue, the down
// GEMM's token operand) take the same order, so every product pairs the same
// column of both operands.  In words of one half: a 4 x 4 transpose, chunk
// 2j + h = (word j, j + 4, j + 8, j + 12).

// xp[p] = x[perm[p] / k] with its columns in the stage order above: the layer
// input gathered into the grouped order, so that every GEMM unit's token rows
// are one contiguous tile for the TMA.  One warp per row, 512 bytes (four
// stages) per round: a coalesced 16-byte load per lane, the 4 x 4 word
// transposes through shared memory (4 words of padding per 32, so that the
// transposed reads hit 32 different banks), a coalesced 16-byte store per lane.
__global__ void __launch_bounds__(256) pf_gather_kernel(const uint16_t* __restrict__ x,
                                                        const int32_t* __restrict__ perm, int n, int k, int H,
                                                        uint16_t* __restrict__ xp) {
  __shared__ __align__(16) uint32_t tw[8][4 * 36];
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  uint32_t* t = tw[wp];
  const int per = H / 8;  // 16-byte pieces per row (a multiple of 32: H is a multiple of 256)
  // this lane's output piece: stage lane / 8, piece o = 2j + h of it = words j of pieces 4h .. 4h+3
  const int st = lane >> 3, o = lane & 7, j = o >> 1, h = o & 1;
  auto word_at = [&](int piece, int word) { return t[(st * 8 + piece) * 4 + word + 4 * st]; };
  for (int p = blockIdx.x * (blockDim.x >> 5) + wp; p < n; p += gridDim.x * (blockDim.x >> 5)) {
    const uint4* src = reinterpret_cast<const uint4*>(x) + (int64_t)(perm[p] / k) * per;
    uint4* dst = reinterpret_cast<uint4*>(xp) + (int64_t)p * per;
    for (int c0 = 0; c0 < per; c0 += 32) {
      const uint4 v = src[c0 + lane];
      __syncwarp();
      *reinterpret_cast<uint4*>(&t[lane * 4 + 4 * (lane >> 3)]) = v;  // word w of the round at w + 4 (w / 32)
      __syncwarp();
      dst[c0 + lane] = make_uint4(word_at(4 * h, j), word_at(4 * h + 1, j), word_at(4 * h + 2, j), word_at(4 * h + 3, j));
    }
  }
}

// ------------------------------------------------------------------ tcgen05 GEMM

constexpr int kDqWarps = 16;                  // dequantising warps 0..15, one 16-row weight tile each;
                                              // warps 16..19: epilogue (TMEM lane quarters 0..3)
constexpr int kTokWarp = kDqWarps + 4;        // tensor copies of the token rows
constexpr int kKbWarp = kDqWarps + 5;         // bulk copies of the codes and scales
constexpr int kMmaWarp = kDqWarps + 6;        // TMEM allocation and tcgen05.mma issue
constexpr int kGemmThreads = (kDqWarps + 7) * 32;
constexpr int kTileM = 128;                   // tokens per unit (MMA M = TMEM lanes)
constexpr int kTileN = 256;                   // weight rows per unit (MMA N)
constexpr int kStageK = 64;                   // columns per stage (one 128-byte swizzle span of bf16)
constexpr int kItems = kTileN / 16;           // 16-row weight tiles per unit
constexpr uint32_t kTokBytes = kTileM * 128;  // one stage of token rows
constexpr uint32_t kWBytes = kTileN * 128;    // one stage of dequantised weight rows
constexpr int kMaxRing = 8;

// Position in a ring of mbarrier-tracked buffers: the slot of the next fill
// and the phase parity that fill completes.  A consumer waits for `phase` on
// the full barrier; a producer waits for `phase ^ 1` on the empty barrier,
// which a fresh barrier reports as complete (the first round needs no wait).
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int depth) {
    if (++slot == depth) {
      slot = 0;
      phase ^= 1u;
    }
  }
  // parity of the latest fill of slot q (a slot filled at least once)
  __device__ __forceinline__ uint32_t last_parity(int q) const { return q < slot ? phase : phase ^ 1u; }
};

struct GemmArgs {
  int E, k, sdt, G;
  int K;       // reduction length (H or I): K / 64 stages per unit
  int nkb;     // 256-column code blocks per 16-row tile in the device layout (kpad / 256)
  int ng;      // scale groups per row in the device layout (kpad / G)
  int rtiles;  // weight-row tiles per token tile: I / 128 (gate/up), H / 256 (down)
  int64_t codes[2], scales[2];  // matrix sections in an expert blob: (gate, up) or (down, -)
  const uint8_t* const* blob_hbm;
  const uint8_t* const* blob_host;
  const int32_t* offsets;  // [E+1]
  const int32_t* perm;     // [T*k] slots in (expert, token) order
  const float* topk_w;     // down: routing weight per slot
  uint16_t* out;           // gate/up: h [T*k][I]; down: weighted o [T*k][H], rows in perm order
  int64_t out_ld;
  int nt, nw, nkbs;               // ring depths: token stages, weight stages, code blocks
  uint32_t kb_codes, kb_scales;   // bytes of one 16-row tile's codes / scales per code block
  uint32_t* err;
};

__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  // K-major tile, 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);          // start address
  d |= (uint64_t)1 << 16;                          // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset
  d |= (uint64_t)1 << 46;                          // descriptor version
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}

__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4)                    // D: fp32
         | (1u << 7) | (1u << 10)     // A, B: bf16
         | ((uint32_t)(N >> 3) << 17) // N
         | ((uint32_t)(M >> 4) << 24);  // M
}

__device__ __forceinline__ void umma_bf16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of the warp's 32 TMEM lanes (one per thread), without the wait
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// one 32-byte global store (p 32-byte aligned): a whole sector per thread
__device__ __forceinline__ void st_global_v8(void* p, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, uint32_t w4,
                                             uint32_t w5, uint32_t w6, uint32_t w7) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w0), "r"(w1), "r"(w2), "r"(w3),
               "r"(w4), "r"(w5), "r"(w6), "r"(w7)
               : "memory");
}

// 2-D tiled tensor copy (box of the map) global -> shared, completing on bar
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// The lane's code words of pairs 16q..16q+15 of a (16-row tile, 256-column
// block) chunk in the fragment-ordered layout, renumbered from 0.
template <int B>
__device__ __forceinline__ void chunk_words(const uint8_t* chunk, int lane, int q, uint32_t (&w)[4]) {
  const uint8_t* p = chunk + lane * 16;
  if constexpr (B == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p + q * 512);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (B == 2) {  // words 2q, 2q+1
    const uint2 v = *reinterpret_cast<const uint2*>(p + (q >> 1) * 512 + (q & 1) * 8);
    w[0] = v.x; w[1] = v.y; w[2] = w[3] = 0u;
  } else {  // words 3q .. 3q+2
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int wi = 3 * q + i;
      w[i] = *reinterpret_cast<const uint32_t*>(p + (wi >> 2) * 512 + (wi & 3) * 4);
    }
    w[3] = 0u;
  }
}

// pair i (0..15) of the renumbered words: bf16x2 (128 + u_lo, 128 + u_hi)
template <int B>
__device__ __forceinline__ uint32_t chunk_pair(const uint32_t (&w)[4], int i) {
  constexpr uint32_t kMagic = 0x43004300u;
  if constexpr (B == 4) return and_or(w[i >> 2] >> (4 * (i & 3)), 0x000F000Fu, kMagic);
  else if constexpr (B == 2) return and_or(w[i >> 3] >> (2 * (i & 7)), 0x00030003u, kMagic);
  else {
    if (i < 15) return and_or(w[i / 5] >> (3 * (i % 5)), 0x00070007u, kMagic);
    const uint32_t v = and_or(w[0] >> 15, 0x00010001u, kMagic);
    const uint32_t u = and_or(w[1] >> 14, 0x00020002u, v);
    return and_or(w[2] >> 13, 0x00040004u, u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Shared-memory rings the dequantising warps use.
struct DqRings {
  uint8_t* kbr;  // code-block ring: per slot the 16 tiles' codes, then their scales
  uint32_t kbBytes;
  uint8_t* wr;  // weight ring: per slot 256 dequantised rows x 64 columns, swizzled
  unsigned long long *kbFull, *kbEmpty, *wFull, *wEmpty;
};

// Scale of row r of a 16-row group record (16 scales of SDT).
template <int SDT>
__device__ __forceinline__ float scale_of(const uint8_t* rec, int r) {
  if constexpr (SDT == MOE_SCALE_F32) return reinterpret_cast<const float*>(rec)[r];
  else if constexpr (SDT == MOE_SCALE_BF16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(rec)[r] << 16);
  else return __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(rec)[r]));
}

// Dequantising warp w: its 16-row tile (rows 16w..16w+15 of the unit's 256)
// of every stage, codes and scales from the code-block ring, into bf16 s*q in
// the weight ring, 128-byte-swizzled K-major in the stage K order (see
// pf_gather_kernel).  One code block (256 columns, four stages) per iteration:
// the block's wait and release once, the stages unrolled.
template <int B, int SDT>
__device__ __forceinline__ void dequant_tiles(const GemmArgs& a, const DqRings& r, int nunits, int S, int warp,
                                              int lane) {
  const int g = lane >> 2, tig = lane & 3;
  // the lane's elements of a row in MMA steps 2h and 2h+1 are chunk 2tig + h;
  // swizzled offsets in rows g, g+8
  const uint32_t offh0 = (uint32_t)(((2 * tig) ^ (g & 7)) << 4), offh1 = (uint32_t)(((2 * tig + 1) ^ (g & 7)) << 4);
  constexpr int ssz = SDT == MOE_SCALE_F32 ? 4 : 2;
  const float zb = 128.0f + (float)(1 << (B - 1));
  const uint32_t negzb2 = pack_bf16x2(-zb, -zb);  // exact: 130, 132 or 136
  const int lg_g = 31 - __clz(a.G);                // G = 32, 64 or 128
  RingPos kp, wp;
  for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
    for (int s0 = 0; s0 < S; s0 += 4) {
      const int nq = min(4, S - s0);
      const int kslot = kp.slot;
      mbar_wait<false>(smem_addr(&r.kbFull[kslot]), kp.phase, a.err);
      const uint8_t* kb = r.kbr + (size_t)kslot * r.kbBytes;
      const uint8_t* citem = kb + warp * a.kb_codes;
      const uint8_t* sitem = kb + kItems * a.kb_codes + warp * a.kb_scales;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < nq) {
          const int wslot = wp.slot;
          mbar_wait<false>(smem_addr(&r.wEmpty[wslot]), wp.phase ^ 1u, a.err);
          uint32_t w[4];
          chunk_words<B>(citem, lane, q, w);
          float sc[4];  // rows g, g+8 of the stage's column halves 0 and 1
          {
            const uint8_t* rec = sitem + ((q * 64) >> lg_g) * (16 * ssz);
            sc[0] = scale_of<SDT>(rec, g);
            sc[1] = scale_of<SDT>(rec, g + 8);
            if (a.G >= 64) {  // both halves in one scale group: no second pair of loads
              sc[2] = sc[0];
              sc[3] = sc[1];
            } else {
              const uint8_t* rec1 = sitem + ((q * 64 + 32) >> lg_g) * (16 * ssz);
              sc[2] = scale_of<SDT>(rec1, g);
              sc[3] = scale_of<SDT>(rec1, g + 8);
            }
          }
          uint32_t out[16];  // pair i: MMA step i/4 of the stage, fragment register i%4
          if constexpr (SDT == MOE_SCALE_BF16) {  // (128 + u) - zb is exact in bf16; one rounding for the product
            uint32_t s2[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) s2[h] = pack_bf16x2(sc[h], sc[h]);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t v = chunk_pair<B>(w, i);
              const int kk = i >> 2, rr = i & 3;
              uint32_t t;
              asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(t) : "r"(v), "r"(0x3F803F80u), "r"(negzb2));
              asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out[i]) : "r"(t), "r"(s2[(kk >= 2 ? 2 : 0) + (rr & 1)]));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t v = chunk_pair<B>(w, i);
              const int kk = i >> 2, rr = i & 3;
              const float sv = sc[(kk >= 2 ? 2 : 0) + (rr & 1)];
              out[i] = pack_bf16x2((bf16f(v & 0xffffu) - zb) * sv, (__uint_as_float(v & 0xffff0000u) - zb) * sv);
            }
          }
          uint8_t* r0 = r.wr + (size_t)wslot * kWBytes + (warp * 16 + g) * 128;
          uint8_t* r1 = r0 + 8 * 128;
          *reinterpret_cast<uint4*>(r0 + offh0) = make_uint4(out[0], out[2], out[4], out[6]);
          *reinterpret_cast<uint4*>(r1 + offh0) = make_uint4(out[1], out[3], out[5], out[7]);
          *reinterpret_cast<uint4*>(r0 + offh1) = make_uint4(out[8], out[10], out[12], out[14]);
          *reinterpret_cast<uint4*>(r1 + offh1) = make_uint4(out[9], out[11], out[13], out[15]);
          // every lane's stores visible to the tensor core, then one arrival for the warp
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&r.wFull[wslot]));
          wp.next(a.nw);
        }
      }
      // the warp reads the code block no more
      if (lane == 0) mbar_arrive(smem_addr(&r.kbEmpty[kslot]));
      kp.next(a.nkbs);
    }
  }
}

// Grouped dequant-GEMM over units (expert e, 128 of its tokens, 256 weight rows):
// D[token][row] = sum_k xg[token][k] * s * q[row][k], the token rows (A, M = 128)
// a tile of the grouped activations by tensor copy, the weight rows (B, N = 256)
// dequantised in shared memory.  Gate/up: rows 0-127 of a unit are 128 rows of
// the gate projection, rows 128-255 the same rows of the up projection, and the
// epilogue writes h = silu(g) * u.  Down: 256 rows of H, the epilogue writes the
// slot's routing weight times o.
template <int B, bool GATEUP>
__global__ void __launch_bounds__(kGemmThreads, 1) pf_gemm_kernel(const __grid_constant__ CUtensorMap tok_map,
                                                                   GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  __shared__ __align__(8) unsigned long long tokFull[kMaxRing], tokEmpty[kMaxRing], wFull[kMaxRing],
      wEmpty[kMaxRing], kbFull[4], kbEmpty[4], tfull[2], tempty[2];
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // dynamic window (1024-aligned for the swizzled tiles): token ring | weight
  // ring | code-block ring (codes of the 16 tiles, then their scales) | unit table
  // (offset from the array itself, so that every derived pointer stays a shared-space one)
  uint8_t* smem = dsm + ((1024u - (smem_addr(dsm) & 1023u)) & 1023u);
  uint8_t* tokr = smem;
  uint8_t* wr = tokr + (size_t)a.nt * kTokBytes;
  const uint32_t kbBytes = kItems * (a.kb_codes + a.kb_scales);
  uint8_t* kbr = wr + (size_t)a.nw * kWBytes;
  int* tile_prefix = reinterpret_cast<int*>(kbr + (size_t)a.nkbs * kbBytes);  // [E+1] units before expert e
  const int E = a.E;
  const int S = a.K / kStageK;  // stages per unit

  // unit table: expert e contributes rtiles * ceil(n_e / 128) units
  if (warp == 0) {
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int n = e < E ? a.offsets[e + 1] - a.offsets[e] : 0;
      const int own = a.rtiles * ((n + kTileM - 1) / kTileM);
      int v = own;  // inclusive prefix over the 32 lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (e < E) tile_prefix[e] = carry + v - own;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) tile_prefix[E] = carry;
  }
  if (tid == 0) {
    for (int q = 0; q < a.nt; ++q) {
      mbar_init(smem_addr(&tokFull[q]), 1);
      mbar_init(smem_addr(&tokEmpty[q]), 1);
    }
    for (int q = 0; q < a.nw; ++q) {
      mbar_init(smem_addr(&wFull[q]), kDqWarps);  // one arrival per warp
      mbar_init(smem_addr(&wEmpty[q]), 1);
    }
    for (int q = 0; q < a.nkbs; ++q) {
      mbar_init(smem_addr(&kbFull[q]), 1);
      mbar_init(smem_addr(&kbEmpty[q]), kDqWarps);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(smem_addr(&tfull[q]), 1);
      mbar_init(smem_addr(&tempty[q]), 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {  // TMEM: two accumulators of 256 fp32 columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                 "n"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const int nunits = tile_prefix[E];

  auto decode_unit = [&](int u, int& e, int& rt, int& n0, int& nrows) {
    int lo = 0, hi = E - 1;  // last e with tile_prefix[e] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_prefix[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    const int r = u - tile_prefix[e];
    rt = r % a.rtiles;
    const int tt = r / a.rtiles;
    const int ne = a.offsets[e + 1] - a.offsets[e];
    n0 = a.offsets[e] + tt * kTileM;
    nrows = min(kTileM, ne - tt * kTileM);
  };

  if (warp < kDqWarps) {
    // ------------------------------------------------------------ dequantisers
    const DqRings r{kbr, kbBytes, wr, kbFull, kbEmpty, wFull, wEmpty};
    if (a.sdt == MOE_SCALE_BF16) dequant_tiles<B, MOE_SCALE_BF16>(a, r, nunits, S, warp, lane);
    else if (a.sdt == MOE_SCALE_F16) dequant_tiles<B, MOE_SCALE_F16>(a, r, nunits, S, warp, lane);
    else dequant_tiles<B, MOE_SCALE_F32>(a, r, nunits, S, warp, lane);
  } else if (warp == kKbWarp) {
    // ------------------------------------------------------------ code blocks
    // Per 256-column code block (4 stages) of a unit: the 16 tiles' codes and
    // scales, one bulk copy each from HBM, 16-byte cp.async by all lanes from
    // pinned host memory; as far ahead as the ring allows.
    const int ssz = a.sdt == MOE_SCALE_F32 ? 4 : 2;
    const int gpk = 256 >> (31 - __clz(a.G));  // scale groups per code block
    const int nkbu = (S + 3) >> 2;              // code blocks per unit
    RingPos kp;
    int nkfill = 0;
    uint32_t hostmask = 0;  // slots last written by cp.async
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      int e, rt, n0, nrows;
      decode_unit(u, e, rt, n0, nrows);
      const uint8_t* hb = a.blob_hbm[e];
      const bool host = hb == nullptr;
      const uint8_t* blob = host ? a.blob_host[e] : hb;
      for (int kb = 0; kb < nkbu; ++kb) {
        const int slot = kp.slot;
        mbar_wait<false>(smem_addr(&kbEmpty[slot]), kp.phase ^ 1u, a.err);
        uint8_t* dst = kbr + (size_t)slot * kbBytes;
        const uint32_t bar = smem_addr(&kbFull[slot]);
        if (!host) {
          if (lane == 0) {
            if ((hostmask >> slot) & 1u) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(bar, kbBytes);
          }
          __syncwarp();
          if (lane < kItems) {
            const int mat = GATEUP ? (lane >> 3) : 0;
            const int64_t t16 = GATEUP ? (int64_t)rt * 8 + (lane & 7) : (int64_t)rt * 16 + lane;
            bulk_g2s(smem_addr(dst + lane * a.kb_codes), blob + a.codes[mat] + (t16 * a.nkb + kb) * B * 512,
                     a.kb_codes, bar);
            bulk_g2s(smem_addr(dst + kItems * a.kb_codes + lane * a.kb_scales),
                     blob + a.scales[mat] + (t16 * a.ng + (int64_t)kb * gpk) * 16 * ssz, a.kb_scales, bar);
          }
          hostmask &= ~(1u << slot);
        } else {
          for (int it = 0; it < kItems; ++it) {
            const int mat = GATEUP ? (it >> 3) : 0;
            const int64_t t16 = GATEUP ? (int64_t)rt * 8 + (it & 7) : (int64_t)rt * 16 + it;
            const uint8_t* cs = blob + a.codes[mat] + (t16 * a.nkb + kb) * B * 512;
            const uint8_t* ss = blob + a.scales[mat] + (t16 * a.ng + (int64_t)kb * gpk) * 16 * ssz;
            for (uint32_t c = lane; c < a.kb_codes / 16; c += 32) cp_async16(dst + it * a.kb_codes + c * 16, cs + c * 16);
            for (uint32_t c = lane; c < a.kb_scales / 16; c += 32)
              cp_async16(dst + kItems * a.kb_codes + it * a.kb_scales + c * 16, ss + c * 16);
          }
          cp_async_mbar_arrive(bar);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar);
          hostmask |= 1u << slot;
        }
        kp.next(a.nkbs);
        ++nkfill;
      }
    }
    cp_async_wait<0>();
    // no copy of this CTA is in flight when it exits: the last fill of every slot has landed
    if (lane == 0)
      for (int q = 0; q < a.nkbs && q < nkfill; ++q) mbar_drain(smem_addr(&kbFull[q]), kp.last_parity(q));
    __syncwarp();
  } else if (warp == kTokWarp) {
    // ------------------------------------------------------------ token rows
    // Per stage: the unit's 128 token rows x 64 columns by one tensor copy.
    // Every lane waits on the barriers (a warp-wide wait wakes sooner than
    // one lane's while the other lanes sit at a warp barrier); lane 0 issues.
    RingPos tp;
    int ntfill = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      int e, rt, n0, nrows;
      decode_unit(u, e, rt, n0, nrows);
      for (int s = 0; s < S; ++s) {
        const int slot = tp.slot;
        mbar_wait<false>(smem_addr(&tokEmpty[slot]), tp.phase ^ 1u, a.err);
        if (lane == 0) {
          const uint32_t bar = smem_addr(&tokFull[slot]);
          mbar_arrive_expect_tx(bar, kTokBytes);
          tma_load_2d(smem_addr(tokr + (size_t)slot * kTokBytes), &tok_map, s * kStageK, n0, bar);
        }
        __syncwarp();
        tp.next(a.nt);
        ++ntfill;
      }
    }
    for (int q = 0; q < a.nt && q < ntfill; ++q) mbar_drain(smem_addr(&tokFull[q]), tp.last_parity(q));
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // The whole warp waits; lane 0 issues the MMAs and the commits.
    const uint32_t idesc = idesc_bf16(kTileM, kTileN);
    RingPos tp, wp;
    int ui = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++ui) {
      const int buf = ui & 1;
      mbar_wait<false>(smem_addr(&tempty[buf]), ((uint32_t)(ui >> 1) & 1u) ^ 1u, a.err);  // accumulator free
      tc_fence_after();
      const uint32_t dacc = tmem + (uint32_t)(buf * 256);
      for (int s = 0; s < S; ++s) {
        const int ts = tp.slot, wsl = wp.slot;
        mbar_wait<false>(smem_addr(&tokFull[ts]), tp.phase, a.err);
        mbar_wait<false>(smem_addr(&wFull[wsl]), wp.phase, a.err);
        tc_fence_after();
        if (lane == 0) {
          const uint32_t at = smem_addr(tokr + (size_t)ts * kTokBytes);
          const uint32_t bt = smem_addr(wr + (size_t)wsl * kWBytes);
#pragma unroll
          for (int j = 0; j < kStageK / 16; ++j)
            umma_bf16(dacc, smem_desc_sw128(at + j * 32), smem_desc_sw128(bt + j * 32), idesc, (s | j) ? 1u : 0u);
          umma_commit(smem_addr(&tokEmpty[ts]));  // both stages are free once these MMAs are done
          umma_commit(smem_addr(&wEmpty[wsl]));
        }
        __syncwarp();
        tp.next(a.nt);
        wp.next(a.nw);
      }
      if (lane == 0) umma_commit(smem_addr(&tfull[buf]));
      __syncwarp();
    }
    // the last MMAs have completed before TMEM is released
    for (int j = max(0, ui - 2); j < ui; ++j) mbar_drain(smem_addr(&tfull[j & 1]), (uint32_t)(j >> 1) & 1u);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 16-19)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // token within the unit = TMEM lane
    int ui = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++ui) {
      int e, rt, n0, nrows;
      decode_unit(u, e, rt, n0, nrows);
      const int buf = ui & 1;
      const bool live = row < nrows;
      float wgt = 0.0f;
      if (!GATEUP && live) wgt = a.topk_w[a.perm[n0 + row]];
      mbar_wait<false>(smem_addr(&tfull[buf]), (uint32_t)(ui >> 1) & 1u, a.err);
      tc_fence_after();
      const uint32_t ta = tmem + (uint32_t)(buf * 256) + ((uint32_t)(quad * 32) << 16);
      uint16_t* orow = a.out + (int64_t)(n0 + row) * a.out_ld;
      if constexpr (GATEUP) {
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {  // half (c0 / 32) & 1 of a 64-column stage of h
          uint32_t hp[16];                      // words of the 32 columns, column order
#pragma unroll
          for (int kk1 = 0; kk1 < 2; ++kk1) {
            uint32_t gv[16], uv[16];
            tmem_ld16_nowait(ta + c0 + 16 * kk1, gv);
            tmem_ld16_nowait(ta + 128 + c0 + 16 * kk1, uv);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; c += 2) {
              const float g0 = __uint_as_float(gv[c]), g1 = __uint_as_float(gv[c + 1]);
              const float h0 = g0 / (1.0f + expf(-g0)) * __uint_as_float(uv[c]);
              const float h1 = g1 / (1.0f + expf(-g1)) * __uint_as_float(uv[c + 1]);
              hp[8 * kk1 + (c >> 1)] = pack_bf16x2(h0, h1);
            }
          }
          if (live) {  // h in the stage K order (pf_gather_kernel): the down GEMM's token operand
            uint4* dst = reinterpret_cast<uint4*>(orow + rt * 128 + (c0 & ~63));
            const int h = (c0 >> 5) & 1;
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[2 * j + h] = make_uint4(hp[j], hp[j + 4], hp[j + 8], hp[j + 12]);
          }
        }
      } else {
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 16) {
          uint32_t v[16];
          tmem_ld16_nowait(ta + c0, v);
          tmem_wait_ld();
          uint32_t op[8];
#pragma unroll
          for (int c = 0; c < 16; c += 2)
            op[c >> 1] = pack_bf16x2(wgt * __uint_as_float(v[c]), wgt * __uint_as_float(v[c + 1]));
          if (live) st_global_v8(orow + rt * 256 + c0, op[0], op[1], op[2], op[3], op[4], op[5], op[6], op[7]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tempty[buf]));
    }
  }
  // teardown: the MMA warp frees TMEM once the last accumulator was read
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(512));
  }
}

// y[t][c] = sum over j ascending of o[inv[t*k + j]][c] (bf16 slot outputs, fp32 sum);
// 8 columns per thread, the k slot rows' 16-byte pieces all requested before the sum.
// With res != nullptr also ysum[t][c] = bf16(y[t][c] + res[t][c]) (the residual
// update, res fp32; res and ysum 16-byte aligned).
__global__ void pf_combine_kernel(const uint16_t* __restrict__ o, const int32_t* __restrict__ inv, int T,
                                  int H, int k, uint16_t* __restrict__ y, const float* __restrict__ res,
                                  uint16_t* __restrict__ ysum) {
  const int per = H / 8;
  const int64_t n = (int64_t)T * per;
  const bool y16 = (reinterpret_cast<uintptr_t>(y) & 15u) == 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / per), c = (int)(i % per);
    uint4 v[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) v[j] = reinterpret_cast<const uint4*>(o)[(int64_t)inv[(int64_t)t * k + j] * per + c];
    float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {
        const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          sum[2 * q] += bf16f(w[q] & 0xffffu);
          sum[2 * q + 1] += bf16f(w[q] >> 16);
        }
      }
    }
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      out[q] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(sum[2 * q])) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(sum[2 * q + 1])) << 16);
    if (y16) {
      reinterpret_cast<uint4*>(y)[i] = make_uint4(out[0], out[1], out[2], out[3]);
    } else {  // y need only be 4-byte aligned
#pragma unroll
      for (int q = 0; q < 4; ++q) reinterpret_cast<uint32_t*>(y)[4 * i + q] = out[q];
    }
    if (res) {
      const float4 r0 = reinterpret_cast<const float4*>(res)[2 * i], r1 = reinterpret_cast<const float4*>(res)[2 * i + 1];
      const float rv[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
      uint32_t so[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        so[q] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(bf16f(out[q] & 0xffffu) + rv[2 * q])) |
                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(bf16f(out[q] >> 16) + rv[2 * q + 1])) << 16);
      reinterpret_cast<uint4*>(ysum)[i] = make_uint4(so[0], so[1], so[2], so[3]);
    }
  }
}

// Per-forward accounting (one CTA): every expert with routed tokens is one
// access; a hit iff it is read from HBM; bytes by residence; cache counters
// (count += 1, last = step) and the miss queue as in the decode kernel.
__global__ void pf_stats_kernel(const int32_t* __restrict__ counts, int E, const uint8_t* const* blob_hbm,
                                unsigned long long* stats, int64_t expert_bytes, int64_t router_bytes,
                                int n_pairs, int lfu, int64_t ge0, uint32_t* lfu_count, int32_t* lfu_last,
                                const int* step, int32_t* miss_list, unsigned* miss_count, int miss_cap,
                                uint32_t* overflow, unsigned long long exact_all) {
  __shared__ int sh[2];
  if (threadIdx.x == 0) sh[0] = sh[1] = 0;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    if (counts[e] == 0) continue;
    const bool hit = blob_hbm[e] != nullptr;
    atomicAdd(&sh[0], 1);
    if (hit) atomicAdd(&sh[1], 1);
    if (lfu) {
      lfu_count[ge0 + e] += 1u;
      lfu_last[ge0 + e] = *step;
      if (!hit) {
        const unsigned mi = atomicAdd(miss_count, 1u);
        if ((int)mi < miss_cap) miss_list[mi] = (int32_t)(ge0 + e);
        else *reinterpret_cast<volatile uint32_t*>(overflow) = 1u;  // queue full: latched
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long D = sh[0], hits = sh[1];
    stats[kStatAccesses] += D;
    stats[kStatHits] += hits;
    stats[kStatMisses] += D - hits;
    stats[kStatHbmBytes] += hits * (unsigned long long)expert_bytes + (unsigned long long)router_bytes;
    stats[kStatHostBytes] += (D - hits) * (unsigned long long)expert_bytes;
    stats[kStatPairs] += (unsigned long long)n_pairs;
    stats[kStatForwards] += 1ull;
    stats[kStatRouterExact] += exact_all;
  }
}

template <bool GATEUP>
cudaError_t launch_gemm(int bits, const CUtensorMap& map, const GemmArgs& a, int grid, size_t smem, cudaStream_t s) {
  const void* fn = bits == 2   ? (const void*)pf_gemm_kernel<2, GATEUP>
                   : bits == 3 ? (const void*)pf_gemm_kernel<3, GATEUP>
                               : (const void*)pf_gemm_kernel<4, GATEUP>;
  cudaError_t e = ensure_dynamic_smem(fn, smem);
  if (e != cudaSuccess) return e;
  switch (bits) {
    case 2: pf_gemm_kernel<2, GATEUP><<<grid, kGemmThreads, smem, s>>>(map, a); break;
    case 3: pf_gemm_kernel<3, GATEUP><<<grid, kGemmThreads, smem, s>>>(map, a); break;
    default: pf_gemm_kernel<4, GATEUP><<<grid, kGemmThreads, smem, s>>>(map, a); break;
  }
  return cudaGetLastError();
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// Tensor map of a row-major bf16 matrix [rows][cols] read as boxes of 128
// rows x 64 columns, 128-byte swizzled (rows past the end read as zero).
cudaError_t rows_map(CUtensorMap* map, const uint16_t* base, int64_t rows, int cols) {
  const EncodeTiledFn f = encode_tiled();
  if (!f) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kStageK, (cuuint32_t)kTileM};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = f(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Ring depths within the opt-in shared memory: two code blocks, three weight
// stages (two if three leave fewer than three token stages), and as many
// token stages as fit (at most kMaxRing).
bool ring_depths(GemmArgs& a, int optin, int E) {
  const size_t kb = (size_t)kItems * (a.kb_codes + a.kb_scales);
  const size_t fixed = 2048 /* static */ + 1024 /* alignment */ + ((size_t)(E + 1) * 4 + 15) / 16 * 16;
  if ((size_t)optin < fixed + 2 * kb) return false;
  const size_t room = (size_t)optin - fixed - 2 * kb;
  a.nkbs = 2;
  for (int nw = 3; nw >= 2; --nw) {
    if (room < (size_t)nw * kWBytes) continue;
    const int nt = (int)std::min<size_t>(kMaxRing, (room - (size_t)nw * kWBytes) / kTokBytes);
    if (nt >= 3 || (nw == 2 && nt >= 2)) {
      a.nw = nw;
      a.nt = nt;
      return true;
    }
  }
  return false;
}

size_t gemm_smem(const GemmArgs& a, int E) {
  return 1024 + (size_t)a.nt * kTokBytes + (size_t)a.nw * kWBytes +
         (size_t)a.nkbs * kItems * (a.kb_codes + a.kb_scales) + (size_t)(E + 1) * 4;
}

}  // namespace

cudaError_t moe::router_norms(const uint16_t* wr, int E, int H, float* out, cudaStream_t s) {
  router_norm_kernel<<<(E + 7) / 8, 256, 0, s>>>(wr, E, H, out);
  return cudaGetLastError();
}

cudaError_t moe::prefill_forward(Plan& p, int layer, const uint16_t* x, int T, uint16_t* y,
                                 cudaStream_t s, const moe_routing_out* dbg, bool lfu,
                                 const uint8_t* const* blob_hbm, const float* res, uint16_t* ysum) {
  const moe_plan_desc& d = p.d;
  const int E = d.num_experts, H = d.hidden, I = d.inter, k = d.top_k;
  const int n = T * k;
  cudaError_t e;
  unsigned long long* st = p.stats + (int64_t)layer * kNumStats;
  const bool all_logits = dbg && dbg->logits;
  if (all_logits) {  // every logit in the fixed order (the caller reads them)
    const dim3 grid((T + kRtTok - 1) / kRtTok, (E + kRtExp - 1) / kRtExp);
    if ((e = ensure_dynamic_smem((const void*)pf_router_kernel, kRtSmem)) != cudaSuccess) return e;
    pf_router_kernel<<<grid, 256, kRtSmem, s>>>(x, T, H, p.wr[layer], p.bias[layer], E, p.logits);
    pf_topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(p.logits, T, E, k, p.topk_idx, p.topk_w);
  } else {  // bounded tensor-core logits, then the fixed order for the candidates only
    const float one = 1.0f, zero = 0.0f;
    cublasStatus_t bs = cublasSetStream(p.blas, s);
    if (bs == CUBLAS_STATUS_SUCCESS)
      bs = cublasGemmEx(p.blas, CUBLAS_OP_T, CUBLAS_OP_N, E, T, H, &one, p.wr[layer], CUDA_R_16BF, H, x,
                        CUDA_R_16BF, H, &zero, p.logits, CUDA_R_32F, E, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
    if (bs != CUBLAS_STATUS_SUCCESS) {  // the caller reports the cuBLAS status
      p.blas_status = (int)bs;
      return cudaErrorUnknown;
    }
    if (E <= 16 * 32)
      pf_select_kernel<16><<<(T + 7) / 8, 256, 0, s>>>(x, T, H, p.wr[layer], p.bias[layer],
                                                       p.wnorm_all + (int64_t)layer * E, E, k, p.logits,
                                                       p.topk_idx, p.topk_w, st + kStatRouterExact);
    else
      pf_select_kernel<0><<<(T + 7) / 8, 256, 0, s>>>(x, T, H, p.wr[layer], p.bias[layer],
                                                      p.wnorm_all + (int64_t)layer * E, E, k, p.logits,
                                                      p.topk_idx, p.topk_w, st + kStatRouterExact);
  }
  {
    const int nb = (n + kGroupChunk - 1) / kGroupChunk;
    const size_t hsm = (size_t)E * 4, wsm = (size_t)8 * E * 4;
    if (wsm > 48 * 1024 &&
        (e = ensure_dynamic_smem((const void*)pf_bucket_place, wsm)) != cudaSuccess)
      return e;
    pf_bucket_count<<<nb, 256, hsm, s>>>(p.topk_idx, n, E, p.pf_bucket);
    pf_bucket_scan<<<1, 1024, 0, s>>>(p.pf_bucket, E, nb, p.counts, p.offsets);
    pf_bucket_place<<<nb, 256, wsm, s>>>(p.topk_idx, n, E, p.pf_bucket, p.perm, p.inv);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // token rows in grouped order, into the o buffer (free until the down projection)
  pf_gather_kernel<<<std::min((n + 7) / 8, 16 * p.sms), 256, 0, s>>>(x, p.perm, n, k, H, p.pf_o);

  const int64_t ge0 = (int64_t)layer * E;
  const int G = d.group_size;
  const int ssz = d.scale_dtype == MOE_SCALE_F32 ? 4 : 2;
  GemmArgs g{};
  g.E = E;
  g.k = k;
  g.sdt = d.scale_dtype;
  g.G = G;
  const uint8_t* const* bhbm = blob_hbm ? blob_hbm : p.blob_hbm + ge0;
  g.blob_hbm = bhbm;
  g.blob_host = p.blob_host + ge0;
  g.offsets = p.offsets;
  g.perm = p.perm;
  g.topk_w = p.topk_w;
  g.err = p.err_dev;
  g.kb_codes = (uint32_t)d.weight_bits * 512u;
  g.kb_scales = (uint32_t)((256 / G) * 16 * ssz);
  int optin = 0;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d.device)) != cudaSuccess)
    return e;
  if (!ring_depths(g, optin, E)) return cudaErrorInvalidConfiguration;
  const size_t smem = gemm_smem(g, E);
  CUtensorMap map;
  // gate / up -> h
  {
    GemmArgs a = g;
    a.K = H;
    a.nkb = p.lay.m[0].kpad / 256;
    a.ng = p.lay.m[0].kpad / G;
    a.rtiles = I / 128;
    a.codes[0] = p.lay.m[0].codes_off;
    a.scales[0] = p.lay.m[0].scales_off;
    a.codes[1] = p.lay.m[1].codes_off;
    a.scales[1] = p.lay.m[1].scales_off;
    a.out = p.pf_h;
    a.out_ld = I;
    if ((e = rows_map(&map, p.pf_o, n, H)) != cudaSuccess) return e;
    if ((e = launch_gemm<true>(d.weight_bits, map, a, p.sms, smem, s)) != cudaSuccess) return e;
  }
  // down -> weighted o per slot
  {
    GemmArgs a = g;
    a.K = I;
    a.nkb = p.lay.m[2].kpad / 256;
    a.ng = p.lay.m[2].kpad / G;
    a.rtiles = H / 256;
    a.codes[0] = p.lay.m[2].codes_off;
    a.scales[0] = p.lay.m[2].scales_off;
    a.out = p.pf_o;
    a.out_ld = H;
    if ((e = rows_map(&map, p.pf_h, n, I)) != cudaSuccess) return e;
    if ((e = launch_gemm<false>(d.weight_bits, map, a, p.sms, smem, s)) != cudaSuccess) return e;
  }
  pf_combine_kernel<<<4 * p.sms, 256, 0, s>>>(p.pf_o, p.inv, T, H, k, y, res, ysum);
  pf_stats_kernel<<<1, 512, 0, s>>>(p.counts, E, bhbm, st,
                                    p.lay.algo_bytes, (int64_t)E * H * 2, n,
                                    lfu && d.cache_policy == MOE_POLICY_LFU, ge0, p.lfu_count, p.lfu_last,
                                    &p.ctl->step, p.miss_list, p.miss_count, d.num_layers * p.max_distinct,
                                    p.err_dev + 1, all_logits ? (unsigned long long)T * E : 0ull);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (dbg) {  // optional routing outputs
    if (dbg->logits) cudaMemcpyAsync(dbg->logits, p.logits, (size_t)T * E * 4, cudaMemcpyDeviceToDevice, s);
    if (dbg->topk_idx) cudaMemcpyAsync(dbg->topk_idx, p.topk_idx, (size_t)n * 4, cudaMemcpyDeviceToDevice, s);
    if (dbg->topk_w) cudaMemcpyAsync(dbg->topk_w, p.topk_w, (size_t)n * 4, cudaMemcpyDeviceToDevice, s);
    if (dbg->counts) cudaMemcpyAsync(dbg->counts, p.counts, (size_t)E * 4, cudaMemcpyDeviceToDevice, s);
    if (dbg->offsets) cudaMemcpyAsync(dbg->offsets, p.offsets, (size_t)(E + 1) * 4, cudaMemcpyDeviceToDevice, s);
    if (dbg->perm) cudaMemcpyAsync(dbg->perm, p.perm, (size_t)n * 4, cudaMemcpyDeviceToDevice, s);
    if (dbg->inv) cudaMemcpyAsync(dbg->inv, p.inv, (size_t)n * 4, cudaMemcpyDeviceToDevice, s);
    e = cudaGetLastError();
  }
  return e;
}
