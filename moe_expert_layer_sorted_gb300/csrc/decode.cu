// Decode-batch forward (T <= 8 tokens): two kernels.
//
// 1. router_logits_kernel: fp32 router logits x.Wr^T (+ bias) in the fixed
//    summation order below, one warp per expert, plus the scale-group sums of
//    x used by the expert kernel.  All of a warp's router-weight loads are in
//    flight at once.
//
// 2. expert_decode_kernel (programmatic dependent launch): a persistent grid
//    sized to be co-resident.  Every CTA
//      - stages the T input rows before it waits for the router;
//      - takes the top-k of every token itself (logit descending, ties to the
//        lower expert index), the renormalised softmax weights, the grouping
//        of (token, expert) pairs by expert and the residence of each distinct
//        expert (an HBM slot, or pinned host memory read in place over UVA),
//        so no CTA waits on a serial last-block phase; CTA 0 alone writes the
//        routing outputs and the cache accounting;
//      - then runs its share of the work units, assigned round robin:
//          A unit (expert d, 16 rows of I, gate or up): that projection for
//            the expert's tokens -> gu buffer;
//          B unit (expert d, 64 rows of H): h = silu(g) * u, o = Wd h for those
//            rows times the routing weight -> obuf[slot]; the last B unit of a
//            row block sums each token's k slots (j ascending) into y (bf16).
//        A units come first (host-resident experts first, so the slow link
//        reads start earliest and overlap the HBM ones); a B unit waits
//        (bounded) for its expert's A units.  Each unit's weights and scales
//        (24 KB at the decode shape) stream through a ring of cp.async slots,
//        so the next units' bytes are in flight while one is computed.
//
// The MoE layer is that of "763B MoE in two 96 GB cards" (section "Where the
// VRAM gap comes from": per layer, a token is routed to k of E experts; the
// idle ones can live in host memory and be read by the GPU over UVA); the
// per-expert residence is the per-expert plan of its "Same idea, native vLLM
// fails" side-box.
//
// Dot products run on mma.sync.m16n8k16 (bf16 x bf16 -> fp32): a 16-row
// weight tile is the A operand, decoded in registers; the expert's (up to 8)
// tokens are the 8 columns of the B operand.  A code u is decoded as the bf16
// value 128 + u (one mask-and-or yields two of them), so a tile product is
// sum (128 + u) x = sum q x + (128 + 2^(b-1)) sum x with q = u - 2^(b-1); the
// second term is subtracted per scale group from the fp32 accumulator.  All
// products are exact in fp32; accumulation is fp32.  The down projection
// feeds h as two bf16 parts (hi + lo) so that it sees ~16 significant bits.
#include <stdio.h>

#include <algorithm>

#include "internal.h"

using namespace moe;

namespace {

constexpr int kRouterWarps = 4;
constexpr int kSlots = 3;                               // cp.async ring depth, in units
constexpr int kHostCtas = 16;  // CTAs given the host-resident experts' units (enough to fill the link)
constexpr int kMaxSlots = kDecodeMaxTokens * kMaxTopK;  // (token, expert) pairs per forward

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// ------------------------------------------------------------------ router

struct RouterArgs {
  const uint16_t* x;
  int T, H, E;
  const uint16_t* wr;
  const float* bias;
  float* logits;  // [T][E]
  float* xsum;    // [T][H/G]: zcorr * sum of x over each scale group
  int group;
  float zcorr;
  unsigned* done_a;
  int nda;
  unsigned* done_b;
  int ndb;
};

// Logits in the fixed order: lane j accumulates, from +0, fmaf(x[i], w[i], acc)
// over i = 256m + 8j + r (m ascending, r ascending); the 32 lane sums are then
// combined by xor-butterfly adds with offsets 16, 8, 4, 2, 1 (every lane ends
// with the same value); the bias is added last.
__global__ void __launch_bounds__(kRouterWarps * 32)
router_logits_kernel(RouterArgs a) {
  extern __shared__ uint4 r_smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(r_smem);  // [T][H] bf16
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, H = a.H, E = a.E;
  // the dependent expert kernel may be scheduled now: it waits for this
  // grid's completion itself (griddepcontrol.wait) and this grid never waits on it
  asm volatile("griddepcontrol.launch_dependents;");

  const int e = blockIdx.x * kRouterWarps + warp;
  const bool ev = e < E;
  const int nm = H / 256;
  const uint4* w = reinterpret_cast<const uint4*>(a.wr + (int64_t)(ev ? e : 0) * H);
  uint4 wv[16];
#pragma unroll
  for (int q = 0; q < 16; ++q)
    if (ev && q < nm) wv[q] = __ldg(w + q * 32 + lane);
  {  // x -> shared memory, eight 16-byte loads in flight per thread
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    const int n = T * H / 8;
    for (int i0 = 0; i0 < n; i0 += 8 * kRouterWarps * 32) {
      uint4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * kRouterWarps * 32 + tid;
        if (i < n) v[q] = __ldg(src + i);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * kRouterWarps * 32 + tid;
        if (i < n) dst[i] = v[q];
      }
    }
  }
  if (blockIdx.x == 0) {  // the expert kernel's counters start at zero
    for (int i = tid; i < a.nda; i += blockDim.x) a.done_a[i] = 0u;
    for (int i = tid; i < a.ndb; i += blockDim.x) a.done_b[i] = 0u;
  }
  __syncthreads();

  if (ev) {
    float acc[kDecodeMaxTokens];
#pragma unroll
    for (int t = 0; t < kDecodeMaxTokens; ++t) acc[t] = 0.0f;
    for (int m0 = 0; m0 < nm; m0 += 16) {
      if (m0 > 0) {
#pragma unroll
        for (int q = 0; q < 16; ++q)
          if (m0 + q < nm) wv[q] = __ldg(w + (m0 + q) * 32 + lane);
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        if (m0 + q >= nm) break;
        const uint32_t wq[4] = {wv[q].x, wv[q].y, wv[q].z, wv[q].w};
#pragma unroll
        for (int t = 0; t < kDecodeMaxTokens; ++t) {
          if (t >= T) break;
          const uint4 xv = reinterpret_cast<const uint4*>(xs + t * H)[(m0 + q) * 32 + lane];
          const uint32_t xq[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const uint32_t xb = (r & 1) ? (xq[r >> 1] >> 16) : (xq[r >> 1] & 0xffffu);
            const uint32_t wb = (r & 1) ? (wq[r >> 1] >> 16) : (wq[r >> 1] & 0xffffu);
            acc[t] = fmaf(bf16f(xb), bf16f(wb), acc[t]);
          }
        }
      }
    }
    const float b = a.bias[e];
#pragma unroll
    for (int t = 0; t < kDecodeMaxTokens; ++t) {
      if (t >= T) break;
      float v = acc[t];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) a.logits[t * E + e] = v + b;
    }
  }
  // scale-group sums of x: pair q = (t, group), one warp each
  const int ng = H / a.group;
  for (int q = blockIdx.x * kRouterWarps + warp; q < T * ng; q += gridDim.x * kRouterWarps) {
    const int t = q / ng, grp = q % ng;
    float v = 0.f;
    for (int i = lane; i < a.group; i += 32) v += bf16f(xs[t * H + grp * a.group + i]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) a.xsum[q] = a.zcorr * v;
  }
}

// ------------------------------------------------------------ expert kernel

struct MatOff {
  int64_t codes, scales;
};

struct ExpertArgs {
  const uint16_t* x;
  int T, H, I, E, k;
  int kpadI;  // I rounded up to a multiple of 256 (down-projection K)
  const float* logits;
  const float* xsum;
  const uint8_t* const* blob_hbm;   // [E] of this layer
  const uint8_t* const* blob_host;  // [E] of this layer
  int64_t ge0;                      // global id of expert 0 of this layer
  int32_t* topk_idx;
  float* topk_w;
  int32_t* perm;
  int32_t* inv;
  moe_routing_out dbg;
  unsigned long long* stats;  // this layer's counters
  int64_t expert_bytes, router_bytes;
  int lfu;
  uint32_t* lfu_count;
  int32_t* lfu_last;
  int step;
  int32_t* miss_list;
  unsigned* miss_count;
  int miss_cap;
  unsigned* done_a;  // [maxD]
  unsigned* done_b;  // [H / kBRows]
  float* gu;         // [maxD][2][tstride][I]
  int tstride;
  float* obuf;  // [T*k][H]
  uint16_t* y;
  MatOff m[3];
  int group, sdt;
  float zcorr;  // 128 + 2^(b-1)
  uint32_t* err;
  int slot_bytes;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float scale_at(const uint8_t* base, int idx, int sdt) {
  if (sdt == MOE_SCALE_F32) return reinterpret_cast<const float*>(base)[idx];
  const unsigned short h = reinterpret_cast<const unsigned short*>(base)[idx];
  if (sdt == MOE_SCALE_BF16) return __uint_as_float((uint32_t)h << 16);
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ bool wait_count(const unsigned* ctr, unsigned target, uint32_t* err) {
  // bounded spin: gives up after ~2^22 polls (well over a second) and latches an error
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    __nanosleep(it < 64 ? 32 : 256);
  }
  *reinterpret_cast<volatile uint32_t*>(err) = kErrTimeout;
  __threadfence_system();
  return false;
}


// (a & m) | c in one instruction.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
  return d;
}

// bf16x2 register (128 + u_lo, 128 + u_hi) of pair P (0..63) of a lane's
// 256-column block held in w (its 4*B words); P is a compile-time constant
// after unrolling.  Field placement: see repack_codes_kernel in plan.cu.
template <int B>
__device__ __forceinline__ uint32_t pair_of(const uint32_t (&w)[4 * B], int P) {
  constexpr uint32_t kMagic = 0x43004300u;  // bf16 128.0 in both halves
  if constexpr (B == 4) {
    return and_or(w[P >> 2] >> (4 * (P & 3)), 0x000F000Fu, kMagic);
  } else if constexpr (B == 2) {
    return and_or(w[P >> 3] >> (2 * (P & 7)), 0x00030003u, kMagic);
  } else {
    const int t = P >> 4, m = P & 15;
    if (m < 15) return and_or(w[3 * t + m / 5] >> (3 * (m % 5)), 0x00070007u, kMagic);
    const uint32_t v = and_or(w[3 * t] >> 15, 0x00010001u, kMagic);
    const uint32_t u = and_or(w[3 * t + 1] >> 14, 0x00020002u, v);
    return and_or(w[3 * t + 2] >> 13, 0x00040004u, u);
  }
}

// One 256-column block of a 16-row weight tile (codes at `tile`, the lane's
// words at tile + q*512 + lane*16) against the lane's B-operand row `bh`
// (and, with HILO, the low part `bl`): for every scale group of the block,
// acc += s * (C_group - z), where s = sc[gi*16] (row g) / sc[gi*16 + 8]
// (row g + 8) and z = z0[gi*9] / z1[gi*9] for the lane's two C columns.
// Two accumulator chains per part (even / odd steps) keep MMAs in flight.
template <int B, int G, bool HILO>
__device__ __forceinline__ void tile_block(const uint8_t* tile, int lane, const uint16_t* bh,
                                           const uint16_t* bl, const float* sc, const float* z0,
                                           const float* z1, float (&acc)[4]) {
  uint32_t w[4 * B];
#pragma unroll
  for (int q = 0; q < B; ++q) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + q * 512 + lane * 16);
    w[4 * q + 0] = v.x;
    w[4 * q + 1] = v.y;
    w[4 * q + 2] = v.z;
    w[4 * q + 3] = v.w;
  }
  float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
  float f0[4] = {0.f, 0.f, 0.f, 0.f}, f1[4] = {0.f, 0.f, 0.f, 0.f};
  constexpr int kSteps = G / 16;
#pragma unroll
  for (int kt = 0; kt < 16; ++kt) {
    const uint32_t a0 = pair_of<B>(w, 4 * kt), a1 = pair_of<B>(w, 4 * kt + 1);
    const uint32_t a2 = pair_of<B>(w, 4 * kt + 2), a3 = pair_of<B>(w, 4 * kt + 3);
    const uint32_t h0 = *reinterpret_cast<const uint32_t*>(bh + kt * 16);
    const uint32_t h1 = *reinterpret_cast<const uint32_t*>(bh + kt * 16 + 8);
    mma_bf16((kt & 1) ? e1 : e0, a0, a1, a2, a3, h0, h1);
    if constexpr (HILO) {
      const uint32_t l0 = *reinterpret_cast<const uint32_t*>(bl + kt * 16);
      const uint32_t l1 = *reinterpret_cast<const uint32_t*>(bl + kt * 16 + 8);
      mma_bf16((kt & 1) ? f1 : f0, a0, a1, a2, a3, l0, l1);
    }
    if ((kt + 1) % kSteps == 0) {  // end of scale group gi (folded at compile time)
      const int gi = (kt + 1) / kSteps - 1;
      const float s0 = sc[gi * 16], s1 = sc[gi * 16 + 8];
      const float y0 = z0[gi * 9], y1 = z1[gi * 9];
      float c[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) c[q] = HILO ? (e0[q] + e1[q]) + (f0[q] + f1[q]) : e0[q] + e1[q];
      acc[0] = fmaf(s0, c[0] - y0, acc[0]);
      acc[1] = fmaf(s0, c[1] - y1, acc[1]);
      acc[2] = fmaf(s1, c[2] - y0, acc[2]);
      acc[3] = fmaf(s1, c[3] - y1, acc[3]);
#pragma unroll
      for (int q = 0; q < 4; ++q) e0[q] = e1[q] = f0[q] = f1[q] = 0.f;
    }
  }
}

template <int B, bool HILO>
__device__ __forceinline__ void tile_block_g(int G, const uint8_t* tile, int lane,
                                             const uint16_t* bh, const uint16_t* bl,
                                             const float* sc, const float* z0, const float* z1,
                                             float (&acc)[4]) {
  if (G == 128) tile_block<B, 128, HILO>(tile, lane, bh, bl, sc, z0, z1, acc);
  else if (G == 64) tile_block<B, 64, HILO>(tile, lane, bh, bl, sc, z0, z1, acc);
  else tile_block<B, 32, HILO>(tile, lane, bh, bl, sc, z0, z1, acc);
}

struct Routing {  // per-CTA copy of this forward's routing (shared memory)
  int e[kMaxSlots];                   // expert of slot s = t*k + j
  float w[kMaxSlots];                 // renormalised weight of slot s
  int perm[kMaxSlots];                // slots ordered by (expert, token)
  int rank[kMaxSlots];                // position of slot s in perm
  int first[kMaxSlots];               // perm position p starts a distinct expert: 1 = HBM, 2 = host
  const uint8_t* pblob[kMaxSlots];
  int wl_off[kMaxSlots];              // distinct expert d (host-resident first): perm offset,
  int wl_cnt[kMaxSlots];              //   token count,
  int wl_e[kMaxSlots];                //   expert id,
  const uint8_t* wl_blob[kMaxSlots];  //   and where its weights are read from
  int D, nh;
  int flag;
};

template <int B>
__global__ void __launch_bounds__(kWarps * 32)
expert_decode_kernel(ExpertArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ Routing R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k, KP = a.kpadI, G = a.group;
  const int ngH = H / G, ngI = KP / G, nkbH = H / kBlockK, nkbI = KP / kBlockK;
  const int xstride = H + 8, hstride = KP + 8;  // bf16 elements; pads spread rows over banks
  const int ssz = a.sdt == MOE_SCALE_F32 ? 4 : 2;
  const int gpb = kBlockK / G;  // scale groups per 256-column block

  // shared memory carve-up (all offsets multiples of 16 bytes).  Row T of xs
  // and of hh / hl is all zeros: B-operand columns of absent tokens read it.
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm);  // [T+1][H+8]
  size_t off = ((size_t)(T + 1) * xstride * 2 + 15) / 16 * 16;
  float* csa = reinterpret_cast<float*>(sm + off);  // [ngH][9], column 8 = 0
  off += ((size_t)ngH * 9 * 4 + 15) / 16 * 16;
  uint8_t* ring = sm + off;  // kSlots units
  off += (size_t)kSlots * a.slot_bytes;
  uint16_t* hh = reinterpret_cast<uint16_t*>(sm + off);  // [T+1][KP+8]
  uint16_t* hl = hh + (size_t)(T + 1) * hstride;         // [T+1][KP+8]
  off += ((size_t)2 * (T + 1) * hstride * 2 + 15) / 16 * 16;
  float* csb = reinterpret_cast<float*>(sm + off);  // [ngI][9], column 8 = 0
  off += ((size_t)ngI * 9 * 4 + 15) / 16 * 16;
  float* red = reinterpret_cast<float*>(sm + off);  // [8][16][8]
  off += (size_t)kWarps * 128 * 4;
  float* sf = reinterpret_cast<float*>(sm + off);  // unit scales as fp32

  for (int i = tid; i < xstride; i += blockDim.x) xs[(size_t)T * xstride + i] = 0;
  for (int i = tid; i < hstride; i += blockDim.x) {
    hh[(size_t)T * hstride + i] = 0;
    hl[(size_t)T * hstride + i] = 0;
  }
  for (int i = tid; i < ngH; i += blockDim.x) csa[i * 9 + 8] = 0.f;
  for (int i = tid; i < ngI; i += blockDim.x) csb[i * 9 + 8] = 0.f;

  // ---- the layer input is not produced by the router: stage it first
  for (int t = 0; t < T; ++t)
    for (int c0 = 0; c0 < H / 8; c0 += 4 * kWarps * 32) {  // four 16-byte loads in flight
      uint4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = c0 + q * kWarps * 32 + tid;
        if (c < H / 8) v[q] = *reinterpret_cast<const uint4*>(a.x + (int64_t)t * H + c * 8);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = c0 + q * kWarps * 32 + tid;
        if (c < H / 8) *reinterpret_cast<uint4*>(xs + t * xstride + c * 8) = v[q];
      }
    }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- top-k, one warp per token.  E <= 512: every lane holds the logits of
  // experts lane, lane+32, ...; each of the k rounds takes the lane's best
  // untaken logit (lowest index among equals), then a warp max over an
  // order-preserving integer key and a warp min over the index among the
  // lanes that hold the max (ties -> lower expert index).
  if (warp < T && E <= 32 * 16) {
    const int t = warp;
    float vb[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int ee = q * 32 + lane;
      vb[q] = ee < E ? __ldcg(a.logits + t * E + ee) : 0.f;
    }
    uint32_t taken = 0u;
    for (int j = 0; j < k; ++j) {
      float bv = 0.f;
      int bq = -1;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int ee = q * 32 + lane;
        if (ee < E && !((taken >> q) & 1u) && (bq < 0 || vb[q] > bv)) {
          bv = vb[q];
          bq = q;
        }
      }
      uint32_t key = 0u;  // below every real key
      if (bq >= 0) {
        uint32_t ub = __float_as_uint(bv == 0.0f ? 0.0f : bv);  // -0 ties +0
        key = (ub & 0x80000000u) ? ~ub : (ub | 0x80000000u);
      }
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
      const uint32_t mine = (bq >= 0 && key == kmax) ? (uint32_t)(bq * 32 + lane) : 0xffffffffu;
      const uint32_t win = __reduce_min_sync(0xffffffffu, mine);
      const float wv = __shfl_sync(0xffffffffu, bv, (int)(win & 31u));
      if (bq >= 0 && (uint32_t)(bq * 32 + lane) == win) taken |= 1u << bq;
      if (lane == 0) {
        R.e[t * k + j] = (int)win;
        R.w[t * k + j] = wv;  // logit for now
      }
    }
    __syncwarp();
    if (lane == 0) {
      const float l0 = R.w[t * k];
      float ex[kMaxTopK];
      float z = 0.0f;
      for (int j = 0; j < k; ++j) {
        ex[j] = expf(R.w[t * k + j] - l0);
        z += ex[j];
      }
      for (int j = 0; j < k; ++j) R.w[t * k + j] = ex[j] / z;
    }
  }
  // ---- larger E: each lane keeps its own best 8 (logit desc, index asc)
  // over experts lane, lane+32, ...; then k rounds of warp argmax
  if (warp < T && E > 32 * 16) {
    const int t = warp;
    float lv[kMaxTopK];
    int li[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      lv[j] = -INFINITY;
      li[j] = 0x7fffffff;
    }
    for (int base = 0; base < E; base += 32 * 16) {
      float vb[16];  // one round trip for 16 logits per lane
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int ee = base + q * 32 + lane;
        vb[q] = ee < E ? __ldcg(a.logits + t * E + ee) : 0.f;
      }
#pragma unroll 1
      for (int q = 0; q < 16; ++q) {
        const int ee = base + q * 32 + lane;
        float cv = vb[q];
        // indices arrive ascending, so strict '>' keeps the lower index first on ties
        if (ee < E && (cv > lv[kMaxTopK - 1] || li[kMaxTopK - 1] == 0x7fffffff)) {
          int ci = ee;
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j) {
            if (li[j] == 0x7fffffff || cv > lv[j]) {
              const float tv = lv[j];
              const int ti = li[j];
              lv[j] = cv;
              li[j] = ci;
              cv = tv;
              ci = ti;
            }
          }
        }
      }
    }
    for (int j = 0; j < k; ++j) {
      float bv = lv[0];  // this lane's head (the list shifts on pop)
      int bi = li[0];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
          bv = ov;
          bi = oi;
        }
      }
      if (li[0] == bi) {  // this lane owned the winner: pop its head
#pragma unroll
        for (int q = 0; q < kMaxTopK - 1; ++q) {
          lv[q] = lv[q + 1];
          li[q] = li[q + 1];
        }
        lv[kMaxTopK - 1] = -INFINITY;
        li[kMaxTopK - 1] = 0x7fffffff;
      }
      if (lane == 0) {
        R.e[t * k + j] = bi;
        R.w[t * k + j] = bv;  // logit for now
      }
    }
    __syncwarp();
    if (lane == 0) {
      const float l0 = R.w[t * k];
      float ex[kMaxTopK];
      float z = 0.0f;
      for (int j = 0; j < k; ++j) {
        ex[j] = expf(R.w[t * k + j] - l0);
        z += ex[j];
      }
      for (int j = 0; j < k; ++j) R.w[t * k + j] = ex[j] / z;
    }
  }
  for (int i = tid; i < T * ngH; i += blockDim.x) {
    const int t = i / ngH, grp = i % ngH;
    csa[grp * 9 + t] = __ldcg(a.xsum + i);
  }
  __syncthreads();

  // ---- grouping by (expert, token) and the distinct-expert work list
  const int n = T * k;
  for (int s = tid; s < n; s += blockDim.x) {
    const int key = R.e[s] * T + s / k;
    int r = 0;
    for (int q = 0; q < n; ++q) r += (R.e[q] * T + q / k) < key;
    R.rank[s] = r;
    R.perm[r] = s;
  }
  __syncthreads();
  for (int p = tid; p < n; p += blockDim.x) {
    const int ee = R.e[R.perm[p]];
    int f = 0;
    if (p == 0 || R.e[R.perm[p - 1]] != ee) {
      const uint8_t* hb = a.blob_hbm[ee];
      f = hb ? 1 : 2;
      R.pblob[p] = hb ? hb : a.blob_host[ee];
    }
    R.first[p] = f;
  }
  __syncthreads();
  for (int p = tid; p < n; p += blockDim.x) {
    const int f = R.first[p];
    if (!f) continue;
    int nh_all = 0, before = 0;
    for (int q = 0; q < n; ++q) {
      nh_all += R.first[q] == 2;
      before += q < p && R.first[q] == f;
    }
    const int d = f == 2 ? before : nh_all + before;
    int cnt = 1;
    while (p + cnt < n && R.first[p + cnt] == 0) ++cnt;
    R.wl_off[d] = p;
    R.wl_cnt[d] = cnt;
    R.wl_e[d] = R.e[R.perm[p]];
    R.wl_blob[d] = R.pblob[p];
  }
  if (tid == 0) {
    int nd = 0, nh = 0;
    for (int q = 0; q < n; ++q) {
      nd += R.first[q] != 0;
      nh += R.first[q] == 2;
    }
    R.D = nd;
    R.nh = nh;
  }
  __syncthreads();
  const int D = R.D;

  // ---- CTA 0: routing outputs and accounting (off the critical path of the others)
  if (blockIdx.x == 0) {
    for (int s = tid; s < n; s += blockDim.x) {
      a.topk_idx[s] = R.e[s];
      a.topk_w[s] = R.w[s];
      a.perm[s] = R.perm[s];
      a.inv[s] = R.rank[s];
      if (a.dbg.topk_idx) a.dbg.topk_idx[s] = R.e[s];
      if (a.dbg.topk_w) a.dbg.topk_w[s] = R.w[s];
      if (a.dbg.perm) a.dbg.perm[s] = R.perm[s];
      if (a.dbg.inv) a.dbg.inv[s] = R.rank[s];
    }
    if (a.dbg.counts || a.dbg.offsets) {
      for (int ee = tid; ee <= E; ee += blockDim.x) {
        int below = 0, eq = 0;
        for (int q = 0; q < n; ++q) {
          below += R.e[q] < ee;
          eq += R.e[q] == ee;
        }
        if (a.dbg.offsets) a.dbg.offsets[ee] = below;
        if (a.dbg.counts && ee < E) a.dbg.counts[ee] = eq;
      }
    }
    if (a.dbg.logits)
      for (int i = tid; i < T * E; i += blockDim.x) a.dbg.logits[i] = __ldcg(a.logits + i);
    if (a.lfu) {
      for (int d = tid; d < D; d += blockDim.x) {  // distinct experts: no two threads share g
        const int64_t gid = a.ge0 + R.wl_e[d];
        a.lfu_count[gid] += 1u;
        a.lfu_last[gid] = a.step;
        if (d < R.nh) {
          const unsigned mi = atomicAdd(a.miss_count, 1u);
          if ((int)mi < a.miss_cap) a.miss_list[mi] = (int32_t)gid;
        }
      }
    }
    if (tid == 0) {
      unsigned long long* st = a.stats;
      const int nh = R.nh;
      const unsigned long long v0 = st[kStatAccesses], v1 = st[kStatHits], v2 = st[kStatMisses],
                               v3 = st[kStatHbmBytes], v4 = st[kStatHostBytes],
                               v5 = st[kStatPairs], v6 = st[kStatForwards];
      st[kStatAccesses] = v0 + D;
      st[kStatHits] = v1 + (D - nh);
      st[kStatMisses] = v2 + nh;
      st[kStatHbmBytes] = v3 + (unsigned long long)(D - nh) * a.expert_bytes + a.router_bytes;
      st[kStatHostBytes] = v4 + (unsigned long long)nh * a.expert_bytes;
      st[kStatPairs] = v5 + n;
      st[kStatForwards] = v6 + 1;
    }
  }

  // ---- work units
  const int tilesI = I / kTileRows;
  const int nA = 2 * tilesI;  // (row tile, gate|up) per expert
  const int nB = H / kBRows;  // 64-row blocks of the down projection per expert
  const int64_t a_codes = (int64_t)kTileRows * H * B / 8;
  const int a_scales = ngH * kTileRows * ssz;
  const int64_t b_codes = (int64_t)kBRows * KP * B / 8;
  const int b_scales = (kBRows / kTileRows) * ngI * kTileRows * ssz;

  // Unit lists.  When some but not all routed experts are host-resident,
  // the first Ch CTAs take the host experts' units and the others the HBM
  // experts' units, so the slow link reads run alongside the HBM stream
  // instead of holding every CTA's first slots.  Within each list all A
  // units come before all B units (a B unit waits only on A units, which
  // never wait), and every CTA of the grid is resident, so no wait can block
  // the units it waits for.
  const int nh = R.nh;
  int Ch = 0;
  if (nh > 0 && nh < D && gridDim.x >= 2)
    Ch = min(kHostCtas, min(nh * (nA + nB), (int)gridDim.x / 2));
  const bool hostcta = (int)blockIdx.x < Ch;
  const int dlo = (Ch == 0 || hostcta) ? 0 : nh;
  const int dn = Ch == 0 ? D : (hostcta ? nh : D - nh);
  const int cidx = (Ch == 0 || hostcta) ? (int)blockIdx.x : (int)blockIdx.x - Ch;
  const int cstride = Ch == 0 ? (int)gridDim.x : (hostcta ? Ch : (int)gridDim.x - Ch);
  const int Ul = dn * (nA + nB);
  // i-th unit of this CTA: expert d, A (row tile r>>1, matrix r&1) or B (row block r)
  auto unit_of = [&](int i, int& d, int& r, bool& isA) -> bool {
    const int v = cidx + i * cstride;
    if (v >= Ul) return false;
    if (v < dn * nA) {
      isA = true;
      d = dlo + v / nA;
      r = v % nA;
    } else {
      isA = false;
      const int w = v - dn * nA;
      d = dlo + w / nB;
      r = w % nB;
    }
    return true;
  };

  // warps 1..7 issue the copies; warp 0 never has copies in flight, so its
  // fences (the signals below) do not wait for the prefetch of later units
  auto issue = [&](int i, int slot) {
    int d, r;
    bool isA;
    if (!unit_of(i, d, r, isA) || tid < 32) return;
    const uint8_t* src_c;
    const uint8_t* src_s;
    int nc, ns;
    const uint8_t* blob = R.wl_blob[d];
    if (isA) {
      const int mm = r & 1, mt = r >> 1;
      src_c = blob + a.m[mm].codes + (int64_t)mt * a_codes;
      src_s = blob + a.m[mm].scales + (int64_t)mt * a_scales;
      nc = (int)(a_codes / 16);
      ns = a_scales / 16;
    } else {
      src_c = blob + a.m[2].codes + (int64_t)r * b_codes;
      src_s = blob + a.m[2].scales + (int64_t)r * b_scales;
      nc = (int)(b_codes / 16);
      ns = b_scales / 16;
    }
    uint8_t* dst = ring + (size_t)slot * a.slot_bytes;
    const int nthr = blockDim.x - 32;
    for (int c = tid - 32; c < nc; c += nthr) cp_async16(dst + c * 16, src_c + c * 16);
    uint8_t* dsts = dst + (size_t)nc * 16;
    for (int c = tid - 32; c < ns; c += nthr) cp_async16(dsts + c * 16, src_s + c * 16);
  };

#pragma unroll
  for (int i = 0; i < kSlots - 1; ++i) {
    issue(i, i);
    cp_async_commit();
  }
  for (int i = 0;; ++i) {
    int d, r;
    bool isA;
    if (!unit_of(i, d, r, isA)) break;
    issue(i + kSlots - 1, (i + kSlots - 1) % kSlots);
    cp_async_commit();
    cp_async_wait<kSlots - 1>();
    __syncthreads();
    const uint8_t* slot = ring + (size_t)(i % kSlots) * a.slot_bytes;

    if (isA) {
      // ------------------------------------------------ A unit
      const int mm = r & 1, mt = r >> 1;
      const int Te = R.wl_cnt[d], poff = R.wl_off[d];
      const int c0 = 2 * tig, c1 = 2 * tig + 1;  // C columns (token slots) of this lane
      const int tg = g < Te ? R.perm[poff + g] / k : T;  // B column g: its token, or the zero row
      const int z0i = c0 < Te ? R.perm[poff + c0] / k : 8;
      const int z1i = c1 < Te ? R.perm[poff + c1] / k : 8;
      for (int i = tid; i < ngH * kTileRows; i += blockDim.x) sf[i] = scale_at(slot + a_codes, i, a.sdt);
      __syncthreads();
      const uint16_t* xb = xs + (size_t)tg * xstride + 2 * tig;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int kb = warp; kb < nkbH; kb += kWarps)
        tile_block_g<B, false>(G, slot + (size_t)kb * B * 512, lane, xb + kb * kBlockK, nullptr,
                               sf + kb * gpb * kTileRows + g, csa + kb * gpb * 9 + z0i,
                               csa + kb * gpb * 9 + z1i, acc);
      float* rw = red + warp * 128;  // [row 16][col 8]
      rw[g * 8 + c0] = acc[0];
      rw[g * 8 + c1] = acc[1];
      rw[(g + 8) * 8 + c0] = acc[2];
      rw[(g + 8) * 8 + c1] = acc[3];
      __syncthreads();
      if (tid < 128) {
        const int row = tid >> 3, col = tid & 7;
        if (col < Te) {
          float v = 0.f;
#pragma unroll
          for (int ww = 0; ww < kWarps; ++ww) v += red[ww * 128 + tid];
          a.gu[(((int64_t)d * 2 + mm) * a.tstride + col) * I + mt * kTileRows + row] = v;
        }
      }
      __syncthreads();
      if (tid == 0) {  // release: the barrier above orders the CTA's stores before this fence
        __threadfence();
        atomicAdd(&a.done_a[d], 1u);
      }
    } else {
      // ------------------------------------------------ B unit
      const int rb = r;
      const int Te = R.wl_cnt[d], poff = R.wl_off[d];
      if (tid == 0) R.flag = wait_count(&a.done_a[d], (unsigned)nA, a.err) ? 1 : 0;
      __syncthreads();
      if (R.flag) {
        // h = silu(g) * u for the expert's tokens, split into bf16 hi + lo
        for (int j = 0; j < Te; ++j) {
          const float* gj = a.gu + (((int64_t)d * 2 + 0) * a.tstride + j) * I;
          const float* uj = a.gu + (((int64_t)d * 2 + 1) * a.tstride + j) * I;
          for (int k0 = 0; k0 < KP; k0 += 4 * kWarps * 32) {
            float gv[4], uv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // all loads of the batch in flight at once
              const int kk = k0 + q * kWarps * 32 + tid;
              gv[q] = kk < I ? __ldcg(gj + kk) : 0.f;
              uv[q] = kk < I ? __ldcg(uj + kk) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int kk = k0 + q * kWarps * 32 + tid;
              if (kk < KP) {
                const float h = gv[q] / (1.0f + expf(-gv[q])) * uv[q];
                const __nv_bfloat16 vh = __float2bfloat16_rn(h);
                const __nv_bfloat16 vl = __float2bfloat16_rn(h - __bfloat162float(vh));
                hh[j * hstride + kk] = __bfloat16_as_ushort(vh);
                hl[j * hstride + kk] = __bfloat16_as_ushort(vl);
              }
            }
          }
        }
        __syncthreads();
        // scale-group sums of hi + lo, one warp per (group, token)
        for (int q = warp; q < ngI * Te; q += kWarps) {
          const int grp = q % ngI, j = q / ngI;
          float sv = 0.f;
          for (int i = lane; i < G; i += 32) {
            const int kk = grp * G + i;
            sv += bf16f(hh[j * hstride + kk]) + bf16f(hl[j * hstride + kk]);
          }
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
          if (lane == 0) csb[grp * 9 + j] = a.zcorr * sv;
        }
        for (int i = tid; i < (kBRows / kTileRows) * ngI * kTileRows; i += blockDim.x)
          sf[i] = scale_at(slot + b_codes, i, a.sdt);
        __syncthreads();
        const int tl = warp & 3, kpar = warp >> 2;  // row tile within the block, column-block parity
        const int c0 = 2 * tig, c1 = 2 * tig + 1;
        const int hr = g < Te ? g : T;  // B column g: the expert's token slot g, or the zero row
        const uint16_t* hb = hh + (size_t)hr * hstride + 2 * tig;
        const uint16_t* lb = hl + (size_t)hr * hstride + 2 * tig;
        const int z0i = c0 < Te ? c0 : 8, z1i = c1 < Te ? c1 : 8;
        const uint8_t* tile = slot + (size_t)tl * nkbI * B * 512;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int kb = kpar; kb < nkbI; kb += 2)
          tile_block_g<B, true>(G, tile + (size_t)kb * B * 512, lane, hb + kb * kBlockK,
                                lb + kb * kBlockK, sf + (tl * ngI + kb * gpb) * kTileRows + g,
                                csb + kb * gpb * 9 + z0i, csb + kb * gpb * 9 + z1i, acc);
        float* rw = red + warp * 128;
        rw[g * 8 + c0] = acc[0];
        rw[g * 8 + c1] = acc[1];
        rw[(g + 8) * 8 + c0] = acc[2];
        rw[(g + 8) * 8 + c1] = acc[3];
        __syncthreads();
        for (int i = tid; i < kBRows * 8; i += blockDim.x) {
          const int row = i >> 3, col = i & 7;
          if (col < Te) {
            const int t4 = row >> 4, r16 = row & 15;
            const float o = red[t4 * 128 + r16 * 8 + col] + red[(t4 + 4) * 128 + r16 * 8 + col];
            const int s = R.perm[poff + col];
            a.obuf[(int64_t)s * H + rb * kBRows + row] = R.w[s] * o;
          }
        }
        __syncthreads();
        if (tid == 0) {  // release our rows, acquire everyone else's if we are last
          __threadfence();
          R.flag = (atomicAdd(&a.done_b[rb], 1u) == (unsigned)D - 1) ? 2 : 0;
          __threadfence();
        }
        __syncthreads();
        if (R.flag == 2) {  // every expert's contribution to these rows is in: combine
          for (int i = tid; i < T * kBRows; i += blockDim.x) {
            const int t = i / kBRows, row = rb * kBRows + i % kBRows;
            float ov[kMaxTopK];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)  // all k loads in flight, then summed in j order
              if (j < k) ov[j] = __ldcg(a.obuf + (int64_t)(t * k + j) * H + row);
            float o = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)
              if (j < k) o += ov[j];
            a.y[(int64_t)t * H + row] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
          }
        }
      }
    }
    __syncthreads();  // the slot is refilled by the next iteration's issue
  }
  cp_async_wait<0>();
}

template <int B>
cudaError_t launch_expert(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, expert_decode_kernel<B>, a);
}

}  // namespace

cudaError_t moe::decode_forward(Plan& p, int layer, const uint16_t* x, int T, uint16_t* y,
                                cudaStream_t s, const moe_routing_out* dbg) {
  const moe_plan_desc& d = p.d;
  const int E = d.num_experts, H = d.hidden, I = d.inter, k = d.top_k, G = d.group_size;
  const int64_t ge0 = (int64_t)layer * E;
  const float zcorr = 128.0f + (float)(1 << (d.weight_bits - 1));

  RouterArgs r{};
  r.x = x;
  r.T = T;
  r.H = H;
  r.E = E;
  r.wr = p.wr[layer];
  r.bias = p.bias[layer];
  r.logits = p.logits;
  r.xsum = p.xsum;
  r.group = G;
  r.zcorr = zcorr;
  r.done_a = p.done_a;
  r.nda = p.max_distinct;
  r.done_b = p.done_b;
  r.ndb = H / kBRows;
  const int rgrid = (E + kRouterWarps - 1) / kRouterWarps;
  Plan::DecodeCfg& cf = p.dcfg[T];
  cudaError_t e = cudaSuccess;
  if (!cf.ready) {  // launch configuration for this batch size, once per plan
    const int KP = p.lay.m[2].kpad, ssz = scale_size(d.scale_dtype), b = d.weight_bits;
    const size_t a_unit = (size_t)kTileRows * H * b / 8 + (size_t)(H / G) * kTileRows * ssz;
    const size_t b_unit =
        (size_t)kBRows * KP * b / 8 + (size_t)(kBRows / kTileRows) * (KP / G) * kTileRows * ssz;
    cf.slot_bytes = (int)((std::max(a_unit, b_unit) + 127) / 128 * 128);
    const size_t ngH = H / G, ngI = KP / G;
    cf.smem = ((size_t)(T + 1) * (H + 8) * 2 + 15) / 16 * 16 + (ngH * 9 * 4 + 15) / 16 * 16 +
              (size_t)kSlots * cf.slot_bytes + ((size_t)2 * (T + 1) * (KP + 8) * 2 + 15) / 16 * 16 +
              (ngI * 9 * 4 + 15) / 16 * 16 + (size_t)kWarps * 128 * 4 +
              std::max(ngH, (size_t)(kBRows / kTileRows) * ngI) * kTileRows * 4;
    cf.rsmem = (size_t)T * H * 2;
    const void* kfn = b == 2   ? (const void*)expert_decode_kernel<2>
                      : b == 3 ? (const void*)expert_decode_kernel<3>
                               : (const void*)expert_decode_kernel<4>;
    if (cf.smem > p.dsmem_set) {  // only ever raised: a larger batch may already rely on it
      e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cf.smem);
      if (e != cudaSuccess) return e;
      p.dsmem_set = cf.smem;
    }
    if (cf.rsmem > p.rsmem_set) {
      e = cudaFuncSetAttribute(router_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)cf.rsmem);
      if (e != cudaSuccess) return e;
      p.rsmem_set = cf.rsmem;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, kWarps * 32, cf.smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    // every CTA must be resident at once (B units wait on A units of other CTAs)
    const int maxD = std::min(E, T * k);
    const int units = maxD * (2 * (I / kTileRows) + H / kBRows);
    cf.grid = std::max(1, std::min(units, p.sms * per_sm));
    cf.ready = true;
  }
  const size_t rsmem = cf.rsmem;
  router_logits_kernel<<<rgrid, kRouterWarps * 32, rsmem, s>>>(r);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  ExpertArgs a{};
  a.x = x;
  a.T = T;
  a.H = H;
  a.I = I;
  a.E = E;
  a.k = k;
  a.kpadI = p.lay.m[2].kpad;
  a.logits = p.logits;
  a.xsum = p.xsum;
  a.blob_hbm = p.blob_hbm + ge0;
  a.blob_host = p.blob_host + ge0;
  a.ge0 = ge0;
  a.topk_idx = p.topk_idx;
  a.topk_w = p.topk_w;
  a.perm = p.perm;
  a.inv = p.inv;
  if (dbg) a.dbg = *dbg;
  a.stats = p.stats + (int64_t)layer * kNumStats;
  a.expert_bytes = p.lay.algo_bytes;
  a.router_bytes = (int64_t)E * H * 2;
  a.lfu = d.cache_policy == MOE_POLICY_LFU;
  a.lfu_count = p.lfu_count;
  a.lfu_last = p.lfu_last;
  a.step = p.step;
  a.miss_list = p.miss_list;
  a.miss_count = p.miss_count;
  a.miss_cap = d.num_layers * p.max_distinct;
  a.done_a = p.done_a;
  a.done_b = p.done_b;
  a.gu = p.hbuf;
  a.tstride = std::min(d.max_tokens, kDecodeMaxTokens);
  a.obuf = p.obuf;
  a.y = y;
  for (int m = 0; m < 3; ++m) {
    a.m[m].codes = p.lay.m[m].codes_off;
    a.m[m].scales = p.lay.m[m].scales_off;
  }
  a.group = G;
  a.sdt = d.scale_dtype;
  a.zcorr = zcorr;
  a.err = p.err_dev;
  a.slot_bytes = cf.slot_bytes;
  const int b = d.weight_bits, grid = cf.grid;
  const size_t smem = cf.smem;
  switch (b) {
    case 2: return launch_expert<2>(a, grid, smem, s);
    case 3: return launch_expert<3>(a, grid, smem, s);
    default: return launch_expert<4>(a, grid, smem, s);
  }
}
