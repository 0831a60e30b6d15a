// Decode-batch forward (T <= 8 tokens): two kernels.
//
// 1. router_logits_kernel: fp32 router logits x.Wr^T (+ bias) in the fixed
//    summation order below, one warp per expert, plus the scale-group sums of
//    x used by the expert kernel; it also advances the forward's epoch.
//
// 2. expert_decode_kernel (programmatic dependent launch): a persistent grid,
//    one CTA of 16 warps per SM, all co-resident.  Every CTA
//      - stages the T input rows before it waits for the router;
//      - takes the top-k of every token itself (logit descending, ties to the
//        lower expert index), the renormalised softmax weights, the grouping
//        of (token, expert) pairs by expert and the residence of each distinct
//        expert (an HBM slot, or pinned host memory read in place over UVA);
//        CTA 0's producer warp alone writes the routing outputs and the
//        cache accounting, once it has issued its units;
//      - then runs its share of the work:
//          A task (expert d, 16 rows of I): gate and up projections of those
//            rows for the expert's tokens, streamed as NP units (column
//            ranges of both matrices, up to 4096 columns per unit); at the
//            end h = silu(g) * u in bf16,
//            published to the other CTAs;
//          B unit (expert d, 128 rows of H): o = Wd h for those rows times the
//            routing weight -> obuf[slot]; the B unit of the last distinct
//            expert of a row block then sums each token's k slots (j
//            ascending) into y (bf16).
//        A tasks are dealt round robin and come first; B units follow in
//        contiguous runs (so a CTA stages an expert's h once for several
//        units), balanced against the A work.  Each unit's weights and
//        scales (25.6 KB at the decode shape) stream through a ring of
//        cp.async slots, so the next units' bytes are in flight while one is
//        computed.  When some routed experts are host-resident, a few CTAs
//        take all of their work, so the slow link reads overlap the HBM ones.
//
// Hand-offs between CTAs carry no fences or counters: every published word is
// 64 bits, payload in the low half and the forward's epoch in the high half,
// written and read with single-copy-atomic relaxed accesses; a reader waits
// (bounded) until the word carries the current epoch.  Work is ordered so
// that a unit only waits on units that come before it in every CTA's list,
// and all CTAs are resident, so every wait ends.
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
// takes h rounded to bf16 (the layer output is bf16 as well).
#include <stdio.h>

#include <algorithm>

#include "internal.h"

using namespace moe;

namespace {

#include "device_common.cuh"

constexpr int kRouterWarps = 4;
constexpr int kMaxRing = 8;                             // cp.async ring depth bound, in units
constexpr int kHostCtasMin = 4, kHostCtasMax = 16;  // CTAs given the host-resident experts' work
// Work-time weight of a host-resident expert's units against an HBM one's when
// the grid is split: a CTA reads pinned host memory over the link several
// times slower than it streams and computes a unit from HBM.
constexpr int kHostCost = 1;
constexpr int kMaxSlots = kDecodeMaxTokens * kMaxTopK;  // (token, expert) pairs per forward

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
  unsigned* epoch;  // advanced once per forward
};

// Logits in the fixed order: lane j accumulates, from +0, fmaf(x[i], w[i], acc)
// over i = 256m + 8j + r (m ascending, r ascending); the 32 lane sums are then
// combined by xor-butterfly adds with offsets 16, 8, 4, 2, 1 (every lane ends
// with the same value); the bias is added last.  Grid: (experts / 4) x
// (token pairs); one warp per (expert, pair of tokens), the pair's inputs
// converted to fp32 in shared memory once per CTA.
constexpr int kRouterTok = 2;

__global__ void __launch_bounds__(kRouterWarps * 32)
router_logits_kernel(RouterArgs a) {
  extern __shared__ uint4 r_smem[];
  float* xf = reinterpret_cast<float*>(r_smem);  // [kRouterTok][H] fp32
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, E = a.E;
  const int t0 = blockIdx.y * kRouterTok, nt = min(kRouterTok, a.T - t0);
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
  {  // this pair's inputs -> fp32 shared memory, four 16-byte loads in flight per thread
    const uint4* src = reinterpret_cast<const uint4*>(a.x + (int64_t)t0 * H);
    const int n = nt * H / 8;
    for (int i0 = 0; i0 < n; i0 += 4 * kRouterWarps * 32) {
      uint4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + q * kRouterWarps * 32 + tid;
        if (i < n) v[q] = __ldg(src + i);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + q * kRouterWarps * 32 + tid;
        if (i < n) {
          float4* d = reinterpret_cast<float4*>(xf + (size_t)i * 8);
          d[0] = make_float4(bf16f(v[q].x & 0xffffu), bf16f(v[q].x >> 16), bf16f(v[q].y & 0xffffu),
                             bf16f(v[q].y >> 16));
          d[1] = make_float4(bf16f(v[q].z & 0xffffu), bf16f(v[q].z >> 16), bf16f(v[q].w & 0xffffu),
                             bf16f(v[q].w >> 16));
        }
      }
    }
  }
  if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) {  // a new epoch for this forward (never 0)
    const unsigned ep = *a.epoch + 1u;
    *a.epoch = ep ? ep : 1u;
  }
  __syncthreads();

  if (ev) {
    float acc[kRouterTok];
#pragma unroll
    for (int t = 0; t < kRouterTok; ++t) acc[t] = 0.0f;
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
        float wf[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) wf[r] = (r & 1) ? __uint_as_float(wq[r >> 1] & 0xffff0000u)
                                                    : bf16f(wq[r >> 1] & 0xffffu);
#pragma unroll
        for (int t = 0; t < kRouterTok; ++t) {
          if (t >= nt) break;
          const float4* xv = reinterpret_cast<const float4*>(xf + (size_t)t * H + ((m0 + q) * 32 + lane) * 8);
          const float4 xa = xv[0], xb = xv[1];
          const float xr[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
          for (int r = 0; r < 8; ++r) acc[t] = fmaf(xr[r], wf[r], acc[t]);
        }
      }
    }
    const float b = a.bias[e];
#pragma unroll
    for (int t = 0; t < kRouterTok; ++t) {
      if (t >= nt) break;
      float v = acc[t];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) a.logits[(t0 + t) * E + e] = v + b;
    }
  }
  // scale-group sums of x: pair q = (t, group) of this CTA's tokens, one warp each
  const int ng = H / a.group;
  for (int q = blockIdx.x * kRouterWarps + warp; q < nt * ng; q += gridDim.x * kRouterWarps) {
    const int t = q / ng, grp = q % ng;
    float v = 0.f;
    for (int i = lane; i < a.group; i += 32) v += xf[(size_t)t * H + grp * a.group + i];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) a.xsum[(t0 + t) * ng + grp] = a.zcorr * v;
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
  const int* step;  // cache step counter (device)
  int32_t* miss_list;
  unsigned* miss_count;
  int miss_cap;
  const unsigned* epoch;
  unsigned long long* hbuf;  // [maxD][tstride][kpadI/2] tagged bf16 pairs of h
  unsigned long long* obuf;  // [T*k][H] tagged fp32 weighted expert outputs
  int tstride;
  uint16_t* y;
  const float* res;  // with ysum: ysum = bf16(y + res), the residual update (nullptr: none)
  uint16_t* ysum;
  MatOff m[3];
  int group, sdt;
  float zcorr;  // 128 + 2^(b-1)
  uint32_t* err;
  int slot_bytes, nslots;
  int skip_h;  // test hook: publish no h (the down units' waits run out)
};

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long tagged(uint32_t payload, uint32_t epoch) {
  return (unsigned long long)payload | ((unsigned long long)epoch << 32);
}

// Waits (bounded) until each word q of p(q) = base + q*stride with bit q of
// `valid` set carries `epoch`; v holds their first reads.  All stale words are
// read again together, so a wait costs one round trip per poll.  After ~2^22
// polls (well over a second) it latches a timeout in the plan's error word and
// the stale payloads read as 0, so the kernel always ends.
template <int N>
__device__ __forceinline__ void wait_words(const unsigned long long* base, int64_t stride, unsigned valid,
                                           uint32_t epoch, uint32_t* err, unsigned long long (&v)[N]) {
  for (uint32_t it = 0;; ++it) {
    unsigned stale = 0u;
#pragma unroll
    for (int q = 0; q < N; ++q)
      if (((valid >> q) & 1u) && (uint32_t)(v[q] >> 32) != epoch) stale |= 1u << q;
    if (!stale) return;
    // give up at once if another wait of this forward already timed out
    if (it >= (1u << 22) || ((it & 4095u) == 4095u && *reinterpret_cast<volatile uint32_t*>(err))) {
      if (it >= (1u << 22)) {
        *reinterpret_cast<volatile uint32_t*>(err) = kErrTimeout;
        __threadfence_system();
      }
#pragma unroll
      for (int q = 0; q < N; ++q)
        if ((stale >> q) & 1u) v[q] = 0ull;
      return;
    }
    if (it >= 64) __nanosleep(128);
#pragma unroll
    for (int q = 0; q < N; ++q)
      if ((stale >> q) & 1u) v[q] = ld_relaxed_u64(base + q * stride);
  }
}

// B-operand rows in shared memory are kept in fragment order: for column
// block kb (256 columns), quad tig (lane % 4) and 16-column step kt, the two
// bf16 pairs a lane feeds one mma.m16n8k16 (columns kt*16 + 2tig, +1 and
// kt*16 + 8 + 2tig, +9) sit at byte kb*576 + tig*144 + kt*8 (+4), so one
// 16-byte load serves two steps.  The 144-byte quad stride and a row stride
// of 64 (mod 128) bytes keep a quarter-warp's loads on distinct banks.
__host__ __device__ inline int frag_row_bytes(int nkb) { return nkb * 576 + ((nkb & 1) ? 0 : 64); }
__device__ __forceinline__ int frag_offset(int col) {  // byte offset of the pair holding column col (even)
  const int kb = col >> 8, kk = col & 255;
  return kb * 576 + ((kk & 7) >> 1) * 144 + (kk >> 4) * 8 + ((kk >> 3) & 1) * 4;
}

__device__ __forceinline__ void mma_bf16_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// One 256-column block of a 16-row weight tile (codes at `tile`, the lane's
// words at tile + q*512 + lane*16) against the lane's B-operand fragments
// `bf` (its quad's 144 bytes of the block): for every scale group gi of the
// block, acc += s * (C_gi - z), where s is the scale of the lane's row g
// (element si + gi*16 of `scb`) or row g + 8 (si + gi*16 + 8), and
// z = z0[gi*9] / z1[gi*9] for the lane's two C columns.  Two accumulator
// chains (even / odd steps) keep MMAs in flight; each group's first MMA of a
// chain starts from zero.
template <int B, int G>
__device__ __forceinline__ void tile_block(const uint8_t* tile, int lane, const uint8_t* bf,
                                           const uint8_t* scb, int si, int sdt, const float* z0,
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
  float e0[4], e1[4];
  constexpr int kSteps = G / 16;
#pragma unroll
  for (int k2 = 0; k2 < 8; ++k2) {
    const uint4 hv = *reinterpret_cast<const uint4*>(bf + k2 * 16);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int kt = 2 * k2 + h;
      const uint32_t a0 = pair_of<B>(w, 4 * kt), a1 = pair_of<B>(w, 4 * kt + 1);
      const uint32_t a2 = pair_of<B>(w, 4 * kt + 2), a3 = pair_of<B>(w, 4 * kt + 3);
      const uint32_t h0 = h ? hv.z : hv.x, h1 = h ? hv.w : hv.y;
      if (kt % kSteps < 2) {
        if (h) mma_bf16_zc(e1, a0, a1, a2, a3, h0, h1);
        else mma_bf16_zc(e0, a0, a1, a2, a3, h0, h1);
      } else {
        mma_bf16(h ? e1 : e0, a0, a1, a2, a3, h0, h1);
      }
      if ((kt + 1) % kSteps == 0) {  // end of scale group gi (folded at compile time)
        const int gi = (kt + 1) / kSteps - 1;
        const float s0 = scale_at(scb, si + gi * 16, sdt), s1 = scale_at(scb, si + gi * 16 + 8, sdt);
        const float y0 = z0[gi * 9], y1 = z1[gi * 9];
        acc[0] = fmaf(s0, (e0[0] + e1[0]) - y0, acc[0]);
        acc[1] = fmaf(s0, (e0[1] + e1[1]) - y1, acc[1]);
        acc[2] = fmaf(s1, (e0[2] + e1[2]) - y0, acc[2]);
        acc[3] = fmaf(s1, (e0[3] + e1[3]) - y1, acc[3]);
      }
    }
  }
}

template <int B>
__device__ __forceinline__ void tile_block_g(int G, const uint8_t* tile, int lane,
                                             const uint8_t* bf, const uint8_t* scb, int si,
                                             int sdt, const float* z0, const float* z1,
                                             float (&acc)[4]) {
  if (G == 128) tile_block<B, 128>(tile, lane, bf, scb, si, sdt, z0, z1, acc);
  else if (G == 64) tile_block<B, 64>(tile, lane, bf, scb, si, sdt, z0, z1, acc);
  else tile_block<B, 32>(tile, lane, bf, scb, si, sdt, z0, z1, acc);
}

struct Routing {  // per-CTA copy of this forward's routing (shared memory)
  int e[kMaxSlots];                   // expert of slot s = t*k + j
  float w[kMaxSlots];                 // renormalised weight of slot s
  int perm[kMaxSlots];                // slots ordered by (expert, token)
  int ptok[kMaxSlots];                // token of perm[p]
  int rank[kMaxSlots];                // position of slot s in perm
  int wl_off[kMaxSlots];              // distinct expert d (host-resident first): perm offset,
  int wl_cnt[kMaxSlots];              //   token count,
  int wl_e[kMaxSlots];                //   expert id,
  const uint8_t* wl_blob[kMaxSlots];  //   and where its weights are read from
  int D, nh;
};

template <int B>
__global__ void __launch_bounds__((kWarps + 1) * 32, 1)
expert_decode_kernel(ExpertArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ Routing R;
  __shared__ __align__(8) unsigned long long fullb[kMaxRing], emptyb[kMaxRing];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k, KP = a.kpadI, G = a.group;
  const int ngH = H / G, ngI = KP / G, nkbH = H / kBlockK, nkbI = KP / kBlockK;
  const int xrow = frag_row_bytes(nkbH), hrow = frag_row_bytes(nkbI);  // fragment-ordered row bytes
  const int ssz = a.sdt == MOE_SCALE_F32 ? 4 : 2;
  const int gpb = kBlockK / G;  // scale groups per 256-column block
  const int sdt = a.sdt;

  // shared memory carve-up (all offsets multiples of 16 bytes).  A CTA runs
  // all of its A tasks before its first B unit, and the last A task ends with
  // a barrier of every consumer warp, so the B units' operands (h and its
  // group sums) reuse the A tasks' (x and its group sums): a deeper ring.
  uint8_t* xs = sm;  // [T] fragment-ordered rows of the layer input (A tasks) ...
  uint8_t* hs = sm;  // ... then [T] fragment-ordered rows of one expert's h (B units)
  size_t off = (size_t)T * max(xrow, hrow);
  float* csa = reinterpret_cast<float*>(sm + off);  // [ngH][9] (A) / [ngI][9] (B), column 8 = 0
  float* csb = csa;
  off += ((size_t)max(ngH, ngI) * 9 * 4 + 15) / 16 * 16;
  float* red = reinterpret_cast<float*>(sm + off);  // [2][kWarps][16][8] per-warp partials
  off += (size_t)2 * kWarps * 128 * 4;

  uint8_t* ring = sm + off;  // a.nslots units

  for (int i = tid; i < max(ngH, ngI); i += blockDim.x) csa[i * 9 + 8] = 0.f;

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
        if (c < H / 8) {  // 8 columns = the same step and half for the four quads
          uint32_t* dq = reinterpret_cast<uint32_t*>(xs + (size_t)t * xrow + frag_offset(c * 8));
          dq[0] = v[q].x;
          dq[36] = v[q].y;  // +144 bytes per quad
          dq[72] = v[q].z;
          dq[108] = v[q].w;
        }
      }
    }
  // the residence tables are not written by the router (only by an earlier
  // step end, complete before it started): pull them into L1 while waiting,
  // so that the grouping's lookups after routing do not go to L2
  if (warp == kWarps - 1)
    for (int e0 = lane * 16; e0 < E; e0 += 32 * 16) {  // 16 pointers per 128-byte line
      asm volatile("prefetch.global.L1 [%0];" ::"l"(a.blob_hbm + e0));
      asm volatile("prefetch.global.L1 [%0];" ::"l"(a.blob_host + e0));
    }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // scale-group sums of x (written by the router) into shared memory, by the
  // highest-numbered threads, so that the top-k warps start at once
  for (int i = (int)blockDim.x - 1 - tid; i < T * ngH; i += blockDim.x) {
    const int t = i / ngH, grp = i % ngH;
    csa[grp * 9 + t] = __ldcg(a.xsum + i);
  }

  // Softmax over a token's k logits (R.w[t*k + j], j < k, descending), one
  // lane per slot: w_j = exp(l_j - l_0) / sum_j exp(l_j - l_0), the sum in j order.
  auto renormalise = [&](int t) {
    __syncwarp();
    const float l0 = R.w[t * k];
    const float ex = lane < k ? expf(R.w[t * k + lane] - l0) : 0.f;
    float z = 0.f;
    for (int j = 0; j < k; ++j) z += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) R.w[t * k + lane] = ex / z;
  };
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
    renormalise(t);
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
    renormalise(t);
  }
  __syncthreads();

  // ---- grouping by (expert, token) and the distinct-expert work list, by
  // warp 0 alone (n = T*k <= 64: two slots / perm positions per lane)
  const int n = T * k;
  if (warp == 0) {
    constexpr unsigned kAll = 0xffffffffu;
    const int s0 = lane, s1 = lane + 32;
    const int key0 = s0 < n ? R.e[s0] * T + s0 / k : 0x7fffffff;  // unique per slot
    const int key1 = s1 < n ? R.e[s1] * T + s1 / k : 0x7fffffff;
    int r0 = 0, r1 = 0;
    if (n <= 32) {  // rank = number of smaller keys
#pragma unroll 8
      for (int j = 0; j < n; ++j) r0 += __shfl_sync(kAll, key0, j) < key0;
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int o0 = __shfl_sync(kAll, key0, j), o1 = __shfl_sync(kAll, key1, j);
        r0 += (o0 < key0) + (o1 < key0);
        r1 += (o0 < key1) + (o1 < key1);
      }
    }
    if (s0 < n) {
      R.rank[s0] = r0;
      R.perm[r0] = s0;
      R.ptok[r0] = s0 / k;
    }
    if (s1 < n) {
      R.rank[s1] = r1;
      R.perm[r1] = s1;
      R.ptok[r1] = s1 / k;
    }
    __syncwarp();
    // perm positions p0 = lane, p1 = lane + 32: expert, first-of-run flag, residence
    const int pe0 = s0 < n ? R.e[R.perm[s0]] : -1, pe1 = s1 < n ? R.e[R.perm[s1]] : -1;
    const int up0 = __shfl_up_sync(kAll, pe0, 1), up1 = __shfl_up_sync(kAll, pe1, 1);
    const int last0 = __shfl_sync(kAll, pe0, 31);
    const bool f0 = s0 < n && (lane == 0 || up0 != pe0);
    const bool f1 = s1 < n && ((lane == 0 ? last0 : up1) != pe1);
    const uint8_t* hb0 = f0 ? a.blob_hbm[pe0] : nullptr;  // both tables read at once
    const uint8_t* hh0 = f0 ? a.blob_host[pe0] : nullptr;
    const uint8_t* hb1 = f1 ? a.blob_hbm[pe1] : nullptr;
    const uint8_t* hh1 = f1 ? a.blob_host[pe1] : nullptr;
    const unsigned F0 = __ballot_sync(kAll, f0), F1 = __ballot_sync(kAll, f1);
    const unsigned X0 = __ballot_sync(kAll, f0 && !hb0), X1 = __ballot_sync(kAll, f1 && !hb1);  // host
    const int nh = __popc(X0) + __popc(X1), nd = __popc(F0) + __popc(F1);
    const unsigned lt = (1u << lane) - 1u;
    if (f0) {  // host-resident experts first, each group in perm order
      const int d = !hb0 ? __popc(X0 & lt) : nh + __popc((F0 & ~X0) & lt);
      const unsigned above = F0 & ~lt & ~(1u << lane);
      const int nxt = above ? __ffs(above) - 1 : (F1 ? 32 + __ffs(F1) - 1 : n);
      R.wl_off[d] = s0;
      R.wl_cnt[d] = min(nxt, n) - s0;
      R.wl_e[d] = pe0;
      R.wl_blob[d] = hb0 ? hb0 : hh0;
    }
    if (f1) {
      const int d = !hb1 ? __popc(X0) + __popc(X1 & lt)
                         : nh + __popc(F0 & ~X0) + __popc((F1 & ~X1) & lt);
      const unsigned above = F1 & ~lt & ~(1u << lane);
      const int nxt = above ? 32 + __ffs(above) - 1 : n;
      R.wl_off[d] = s1;
      R.wl_cnt[d] = nxt - s1;
      R.wl_e[d] = pe1;
      R.wl_blob[d] = hb1 ? hb1 : hh1;
    }
    if (lane == 0) {
      R.D = nd;
      R.nh = nh;
    }
  }
  __syncthreads();
  const int D = R.D;

  // ---- routing outputs and cache accounting: CTA 0's producer warp, once
  // it has issued its units (no other work depends on them in this forward)
  auto account = [&]() {
    for (int s = lane; s < n; s += 32) {
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
      for (int ee = lane; ee <= E; ee += 32) {
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
      for (int i = lane; i < T * E; i += 32) a.dbg.logits[i] = __ldcg(a.logits + i);
    if (a.lfu) {
      for (int d = lane; d < D; d += 32) {  // distinct experts: no two threads share g
        const int64_t gid = a.ge0 + R.wl_e[d];
        a.lfu_count[gid] += 1u;
        a.lfu_last[gid] = *a.step;
        if (d < R.nh) {
          const unsigned mi = atomicAdd(a.miss_count, 1u);
          if ((int)mi < a.miss_cap) a.miss_list[mi] = (int32_t)gid;
          else *reinterpret_cast<volatile uint32_t*>(a.err + 1) = 1u;  // queue full: latched
        }
      }
    }
    if (lane == 0) {
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
  };

  // ---- work
  const uint32_t epoch = *reinterpret_cast<const volatile unsigned*>(a.epoch);
  const int tilesI = I / kTileRows;
  const int nB = H / kBRows;                      // 128-row blocks of the down projection
  const int NP = (nkbH + 15) / 16;                // units per A task (up to 16 column blocks of both
                                                  // matrices per unit: two per warp)
  const int kbpp = (nkbH + NP - 1) / NP;          // column blocks per A unit (the last may have fewer)
  const int64_t b_codes = (int64_t)kBRows * KP * B / 8;
  const int b_scales = (kBRows / kTileRows) * ngI * kTileRows * ssz;

  // Work lists.  When some but not all routed experts are host-resident, the
  // first Ch CTAs take the host experts' work and the others the HBM
  // experts'.  In a list, A tasks are dealt round robin and every CTA runs
  // its A tasks before its B units; B units, ordered by (expert, row block),
  // are split into contiguous runs, CTAs with fewer A tasks first.  The
  // combines of row blocks come last.  A B unit waits only on A tasks and a
  // combine only on B units, so every wait is on work that some resident CTA
  // runs before anything it could be blocked by.
  const int nh = R.nh;
  int Ch = 0;
  if (nh > 0 && nh < D && gridDim.x >= 2) {  // the host share of the grid: the host units' share
                                             // of the work time, within [kHostCtasMin, kHostCtasMax]
    const int wh = kHostCost * nh, wt = wh + (D - nh);
    Ch = min(min(kHostCtasMax, max(kHostCtasMin, ((int)gridDim.x * wh + wt / 2) / wt)),
             min(nh * (tilesI + nB), (int)gridDim.x / 2));
  }
  const bool hostcta = (int)blockIdx.x < Ch;
  const int dlo = (Ch == 0 || hostcta) ? 0 : nh;
  const int dn = Ch == 0 ? D : (hostcta ? nh : D - nh);
  const int cidx = (Ch == 0 || hostcta) ? (int)blockIdx.x : (int)blockIdx.x - Ch;
  const int cs = Ch == 0 ? (int)gridDim.x : (hostcta ? Ch : (int)gridDim.x - Ch);
  const int nAt = dn * tilesI, nBu = dn * nB;
  const int nAc = cidx < nAt ? (nAt - 1 - cidx) / cs + 1 : 0;  // A tasks of this CTA
  const int ord = (cidx - nAt % cs + cs) % cs;
  const int bq = nBu / cs, br = nBu % cs;
  const int nBc = bq + (ord < br ? 1 : 0);
  const int blo = ord * bq + min(ord, br);
  const int nU = nAc * NP + nBc;
  // i-th unit of this CTA: expert d; A: row tile r, part pa; B: row block r
  auto unit_of = [&](int i, int& d, int& r, int& pa) -> bool {
    if (i < nAc * NP) {
      const int task = cidx + (i / NP) * cs;
      pa = i % NP;
      d = dlo + task / tilesI;
      r = task % tilesI;
    } else {
      const int v = blo + (i - nAc * NP);
      pa = -1;
      d = dlo + v / nB;
      r = v % nB;
    }
    return true;
  };

  // Producer warp: unit i into ring slot `slot`.  hostmask bit s: the slot's
  // previous unit was written by cp.async (then the bulk copy that reuses it
  // is ordered after those writes by a proxy fence).
  auto issue = [&](int i, int slot, uint32_t& hostmask) {
    int d, r, pa;
    unit_of(i, d, r, pa);
    const uint8_t* blob = R.wl_blob[d];
    uint8_t* dst = ring + (size_t)slot * a.slot_bytes;
    const uint32_t bar = smem_addr(&fullb[slot]);
    // segments: A = gate codes | up codes | gate scales | up scales of the
    // column range; B = codes | scales of 4 row tiles of the down projection
    const uint8_t* src[4];
    uint32_t len[4];
    int nseg;
    if (pa >= 0) {
      const int kb0 = pa * kbpp, nkp = min(nkbH, kb0 + kbpp) - kb0;
      const int64_t co = ((int64_t)r * nkbH + kb0) * B * 512;
      const int64_t so = ((int64_t)r * ngH + (int64_t)kb0 * gpb) * kTileRows * ssz;
      src[0] = blob + a.m[0].codes + co;
      src[1] = blob + a.m[1].codes + co;
      src[2] = blob + a.m[0].scales + so;
      src[3] = blob + a.m[1].scales + so;
      len[0] = len[1] = (uint32_t)nkp * B * 512;
      len[2] = len[3] = (uint32_t)(nkp * gpb * kTileRows * ssz);
      nseg = 4;
    } else {
      src[0] = blob + a.m[2].codes + (int64_t)r * b_codes;
      src[1] = blob + a.m[2].scales + (int64_t)r * b_scales;
      len[0] = (uint32_t)b_codes;
      len[1] = (uint32_t)b_scales;
      len[2] = len[3] = 0;
      nseg = 2;
    }
    if (d >= R.nh) {  // HBM-resident: lane 0's bulk copies
      if (lane == 0) {
        uint32_t tot = 0;
        for (int q = 0; q < nseg; ++q) tot += len[q];
        if ((hostmask >> slot) & 1u) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(bar, tot);
        uint32_t o = 0;
        for (int q = 0; q < nseg; ++q) {
          bulk_g2s(smem_addr(dst + o), src[q], len[q], bar);
          o += len[q];
        }
      }
      hostmask &= ~(1u << slot);
    } else {  // pinned host memory: 16-byte cp.async by the producer's lanes
      uint32_t o = 0;
      for (int q = 0; q < nseg; ++q) {
        for (uint32_t c = lane; c < len[q] / 16; c += 32) cp_async16(dst + o + c * 16, src[q] + c * 16);
        o += len[q];
      }
      cp_async_mbar_arrive(bar);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
      hostmask |= 1u << slot;
    }
  };

  const int nring = a.nslots;
  if (tid == 0) {
    for (int q = 0; q < nring; ++q) {
      mbar_init(smem_addr(&fullb[q]), 1);
      mbar_init(smem_addr(&emptyb[q]), kWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == kWarps) {  // ---------------- producer warp: keeps the ring full
    uint32_t hostmask = 0;
    for (int i = 0; i < nU; ++i) {
      const int sl = i % nring, use = i / nring;
      if (use > 0) mbar_wait(smem_addr(&emptyb[sl]), (uint32_t)(use - 1) & 1u, a.err);
      issue(i, sl, hostmask);
    }
    if (blockIdx.x == 0) account();
    cp_async_wait<0>();
    return;
  }
  // ---------------- consumer warps
  const int c0 = 2 * tig, c1 = 2 * tig + 1;  // C columns (token slots) of this lane
  float acc[4] = {0.f, 0.f, 0.f, 0.f};       // A task partials (kept across its units) / B unit sums
  int hd = -1;                               // expert whose h is staged in hs
  int rp = 0;                                // which half of red the next reduction uses
  for (int i = 0; i < nU; ++i) {
    int d, r, pa;
    unit_of(i, d, r, pa);
    const int sl = i % nring;
    const int Te = R.wl_cnt[d], poff = R.wl_off[d];
    if (pa < 0 && d != hd) {  // B unit of a new expert: stage its h (waiting, bounded, for its
                              // A tasks) and the zero-point group sums
      const int np2 = KP / 2, ip2 = I / 2;
      const unsigned long long* hsrc = a.hbuf + (int64_t)d * a.tstride * np2;
      for (int i0 = tid; i0 < Te * np2; i0 += 4 * kWarps * 32) {
        unsigned long long v[4];
        unsigned valid = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // four reads in flight, waited on together
          const int ii = i0 + q * kWarps * 32;
          const bool ok = ii < Te * np2 && ii % np2 < ip2;
          v[q] = ok ? ld_relaxed_u64(hsrc + ii) : 0ull;
          valid |= (unsigned)ok << q;
        }
        wait_words<4>(hsrc + i0, kWarps * 32, valid, epoch, a.err, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ii = i0 + q * kWarps * 32;
          if (ii < Te * np2) {
            const int n = ii / np2, c = ii % np2;
            const uint32_t pr = c < ip2 ? (uint32_t)v[q] : 0u;
            *reinterpret_cast<uint32_t*>(hs + (size_t)n * hrow + frag_offset(2 * c)) = pr;
          }
        }
      }
      consumer_sync();
      // zero-point group sums of h: fp32 sums of 16 rows (ascending), then of a
      // group's 16-row sums; scratch in the half of red the next reduction uses
      // (the previous unit's readers use the other half)
      float* ssum = red + (rp & 1) * kWarps * 128;  // [Te][tilesI]
      for (int q = tid; q < Te * tilesI; q += kWarps * 32) {
        const int n = q / tilesI, mt = q % tilesI;
        const uint8_t* hrow_n = hs + (size_t)n * hrow;
        float s16 = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t pr = *reinterpret_cast<const uint32_t*>(hrow_n + frag_offset(2 * (8 * mt + c)));
          s16 += bf16f(pr & 0xffffu);
          s16 += bf16f(pr >> 16);
        }
        ssum[q] = s16;
      }
      consumer_sync();
      const int tpg = G / kTileRows;  // 16-row sums per scale group
      for (int q = tid; q < ngI * Te; q += kWarps * 32) {
        const int grp = q % ngI, n = q / ngI;
        float sv = 0.f;
        for (int j = 0; j < tpg; ++j) {
          const int mt = grp * tpg + j;
          if (mt < tilesI) sv += ssum[n * tilesI + mt];
        }
        csb[grp * 9 + n] = a.zcorr * sv;
      }
      hd = d;
      consumer_sync();
    }

    // ---- the unit's dot products: one code path for both kinds
    // A (task d, tile r, part pa): warp w takes matrix w&1 (gate / up) and
    //   the part's column blocks w>>1, w>>1 + 8, ...; B column g = token of
    //   the expert's slot g, against the layer input.
    // B (expert d, row block r): warp w takes row tile w&7 and column blocks
    //   w>>3, w>>3 + 2, ...; B column g = the expert's slot g, against h.
    // Columns g >= Te read a real row; their C columns are never used.
    const uint8_t* slot = ring + (size_t)sl * a.slot_bytes;
    const uint8_t* tbase;  // codes of the warp's tile, column block 0 of the unit
    const uint8_t* scb;    // scales of the unit
    const uint8_t* bbase;   // the lane's quad of its B-operand row, column block 0
    const float* zb;        // zero-point sums at column block 0
    int si, j0, jstep, jn, kbase;
    if (pa >= 0) {
      const int mm = warp & 1;
      const int kb0 = pa * kbpp, nkp = min(nkbH, kb0 + kbpp) - kb0;
      tbase = slot + (size_t)mm * nkp * B * 512;
      scb = slot + (size_t)2 * nkp * B * 512 + (size_t)mm * nkp * gpb * kTileRows * ssz;
      si = g;
      j0 = warp >> 1, jstep = kWarps / 2, jn = nkp, kbase = kb0;
      bbase = xs + (size_t)R.ptok[poff + (g < Te ? g : 0)] * xrow + tig * 144;
      zb = csa;
      if (pa == 0) acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    } else {
      const int tl = warp & 7;  // row tile w % 8 of the unit's eight
      tbase = slot + (size_t)tl * nkbI * B * 512;
      scb = slot + b_codes;
      si = tl * ngI * kTileRows + g;
      j0 = warp >> 3, jstep = kWarps / 8, jn = nkbI, kbase = 0;
      bbase = hs + (size_t)(g < Te ? g : 0) * hrow + tig * 144;
      zb = csb;
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    }
    const int z0i = c0 < Te ? (pa >= 0 ? R.ptok[poff + c0] : c0) : 8;
    const int z1i = c1 < Te ? (pa >= 0 ? R.ptok[poff + c1] : c1) : 8;
    mbar_wait(smem_addr(&fullb[sl]), (uint32_t)(i / nring) & 1u, a.err);  // the unit's bytes are in
#pragma unroll 1
    for (int j = j0; j < jn; j += jstep)
      tile_block_g<B>(G, tbase + (size_t)j * B * 512, lane, bbase + (kbase + j) * 576, scb,
                      si + j * gpb * kTileRows, sdt, zb + (kbase + j) * gpb * 9 + z0i,
                      zb + (kbase + j) * gpb * 9 + z1i, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&emptyb[sl]));  // this warp reads the slot no more

    if (pa >= 0) {
      if (pa == NP - 1) {  // A task complete: h for these 16 rows, published
        const int mt = r;
        float* rb2 = red + (rp & 1) * kWarps * 128;
        ++rp;
        float* rw = rb2 + warp * 128;  // [row 16][col 8]
        rw[g * 8 + c0] = acc[0];
        rw[g * 8 + c1] = acc[1];
        rw[(g + 8) * 8 + c0] = acc[2];
        rw[(g + 8) * 8 + c1] = acc[3];
        consumer_sync();
        if (tid < 128) {  // (row, token slot) = (tid / 8, tid % 8): gate and up over the warps, h
          const int row = tid >> 3, col = tid & 7;
          float gv = 0.f, uv = 0.f;
#pragma unroll
          for (int ww = 0; ww < kWarps / 2; ++ww) {
            gv += rb2[(2 * ww) * 128 + tid];
            uv += rb2[(2 * ww + 1) * 128 + tid];
          }
          const float h = gv / (1.0f + expf(-gv)) * uv;
          const uint32_t hb = __bfloat16_as_ushort(__float2bfloat16_rn(h));
          const uint32_t next = __shfl_down_sync(0xffffffffu, hb, 8);  // row + 1, same token slot
          if (!(row & 1) && col < Te && !a.skip_h)  // bf16 pair (rows row, row + 1) of token slot col
            st_relaxed_u64(a.hbuf + ((int64_t)d * a.tstride + col) * (KP / 2) + mt * 8 + (row >> 1),
                           tagged(hb | (next << 16), epoch));
        }
      }
    } else {
      const int rb = r;
      float* rb2 = red + (rp & 1) * kWarps * 128;
      ++rp;
      float* rw = rb2 + warp * 128;
      rw[g * 8 + c0] = acc[0];
      rw[g * 8 + c1] = acc[1];
      rw[(g + 8) * 8 + c0] = acc[2];
      rw[(g + 8) * 8 + c1] = acc[3];
      consumer_sync();
      for (int i2 = tid; i2 < kBRows * 8; i2 += kWarps * 32) {
        const int row = i2 >> 3, col = i2 & 7;
        if (col < Te) {
          const int t4 = row >> 4, r16 = row & 15;  // row tile t4 of the unit's eight
          float o = 0.f;
#pragma unroll
          for (int ww = 0; ww < kWarps / 8; ++ww) o += rb2[(8 * ww + t4) * 128 + r16 * 8 + col];
          const int sl2 = R.perm[poff + col];
          st_relaxed_u64(a.obuf + (int64_t)sl2 * H + rb * kBRows + row,
                         tagged(__float_as_uint(R.w[sl2] * o), epoch));
        }
      }
    }
  }
  // ---- combine: after all of its B units, a CTA of the last list sums every
  // token's k slots (j ascending) of row blocks cidx, cidx + cs, ... into y.
  // It waits (bounded) only on B units, which never wait on a combine.
  if (Ch == 0 || !hostcta) {
    for (int rb = cidx; rb < nB; rb += cs) {
      for (int i2 = tid; i2 < T * kBRows; i2 += kWarps * 32) {
        const int t = i2 / kBRows, row = rb * kBRows + i2 % kBRows;
        unsigned long long v[kMaxTopK];
        const float rv = a.res ? __ldg(a.res + (int64_t)t * H + row) : 0.f;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)  // all k reads in flight, waited on together, summed in j order
          if (j < k) v[j] = ld_relaxed_u64(a.obuf + (int64_t)(t * k + j) * H + row);
        wait_words<kMaxTopK>(a.obuf + (int64_t)(t * k) * H + row, H, (1u << k) - 1u, epoch, a.err, v);
        float o = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
          if (j < k) o += __uint_as_float((uint32_t)v[j]);
        const uint16_t yb = __bfloat16_as_ushort(__float2bfloat16_rn(o));
        a.y[(int64_t)t * H + row] = yb;
        if (a.res) a.ysum[(int64_t)t * H + row] = __bfloat16_as_ushort(__float2bfloat16_rn(bf16f(yb) + rv));
      }
    }
  }
}

template <int B>
cudaError_t launch_expert(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3((kWarps + 1) * 32);  // consumer warps + the producer warp
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
                                cudaStream_t s, const moe_routing_out* dbg, const float* res, uint16_t* ysum) {
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
  r.epoch = &p.ctl->epoch;
  const dim3 rgrid((E + kRouterWarps - 1) / kRouterWarps, (T + kRouterTok - 1) / kRouterTok);
  Plan::DecodeCfg& cf = p.dcfg[T];
  cudaError_t e = cudaSuccess;
  if (!cf.ready) {  // launch configuration for this batch size, once per plan
    const int KP = p.lay.m[2].kpad, ssz = scale_size(d.scale_dtype), b = d.weight_bits;
    const int nkbH = H / kBlockK, NP = (nkbH + 15) / 16, kbpp = (nkbH + NP - 1) / NP;
    const size_t a_unit = (size_t)2 * kbpp * b * 512 + (size_t)2 * kbpp * (kBlockK / G) * kTileRows * ssz;
    const size_t b_unit =
        (size_t)kBRows * KP * b / 8 + (size_t)(kBRows / kTileRows) * (KP / G) * kTileRows * ssz;
    cf.slot_bytes = (int)((std::max(a_unit, b_unit) + 127) / 128 * 128);
    const size_t ngH = H / G, ngI = KP / G;
    const size_t fixed = (size_t)T * std::max(frag_row_bytes(H / kBlockK), frag_row_bytes(KP / kBlockK)) +
                         (std::max(ngH, ngI) * 9 * 4 + 15) / 16 * 16 + (size_t)2 * kWarps * 128 * 4;
    const void* kfn = b == 2   ? (const void*)expert_decode_kernel<2>
                      : b == 3 ? (const void*)expert_decode_kernel<3>
                               : (const void*)expert_decode_kernel<4>;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d.device);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa{};
    if ((e = cudaFuncGetAttributes(&fa, kfn)) != cudaSuccess) return e;
    // ring depth: as many units as fit beside the static routing state
    const long avail = (long)optin - (long)fa.sharedSizeBytes - (long)fixed;
    cf.nslots = (int)std::min<long>(kMaxRing, avail / cf.slot_bytes);
    if (cf.nslots < 2) return cudaErrorInvalidConfiguration;
    cf.smem = fixed + (size_t)cf.nslots * cf.slot_bytes;
    cf.rsmem = (size_t)kRouterTok * H * 4;
    if ((e = ensure_dynamic_smem(kfn, cf.smem)) != cudaSuccess) return e;
    if ((e = ensure_dynamic_smem((const void*)router_logits_kernel, cf.rsmem)) != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, (kWarps + 1) * 32, cf.smem);
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
  a.step = &p.ctl->step;
  a.miss_list = p.miss_list;
  a.miss_count = p.miss_count;
  a.miss_cap = d.num_layers * p.max_distinct;
  a.epoch = &p.ctl->epoch;
  a.hbuf = p.hbuf;
  a.tstride = std::min(d.max_tokens, kDecodeMaxTokens);
  a.obuf = p.obuf;
  a.y = y;
  a.res = ysum ? res : nullptr;
  a.ysum = ysum;
  for (int m = 0; m < 3; ++m) {
    a.m[m].codes = p.lay.m[m].codes_off;
    a.m[m].scales = p.lay.m[m].scales_off;
  }
  a.group = G;
  a.sdt = d.scale_dtype;
  a.zcorr = zcorr;
  a.err = p.err_dev;
  a.skip_h = p.fail_next ? 1 : 0;
  p.fail_next = false;
  a.slot_bytes = cf.slot_bytes;
  a.nslots = cf.nslots;
  const int b = d.weight_bits, grid = cf.grid;
  const size_t smem = cf.smem;
  switch (b) {
    case 2: return launch_expert<2>(a, grid, smem, s);
    case 3: return launch_expert<3>(a, grid, smem, s);
    default: return launch_expert<4>(a, grid, smem, s);
  }
}
