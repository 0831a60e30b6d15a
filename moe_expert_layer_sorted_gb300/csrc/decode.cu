// Decode-batch forward (T <= 8 tokens): two kernels.
//
// 1. router_decode_kernel: fp32 router logits x.Wr^T (+ bias) in the fixed
//    summation order below, one warp per expert; the last CTA to finish takes
//    the top-k per token (logit descending, ties to the lower expert index),
//    the renormalised softmax weights, the grouping of (token, expert) pairs by
//    expert, the residence lookup of each distinct expert (HBM slot or host
//    memory read in place through UVA) with its cache accounting, and writes the
//    work list of the expert kernel.
//
// 2. expert_decode_kernel (launched with programmatic dependent launch):
//    a persistent grid pulling work units from an atomic queue.
//      A unit (expert d, 16 rows of I): g = Wg x, u = Wu x for the expert's
//        tokens, h = silu(g) * u -> hbuf.
//      B unit (expert d, 128 rows of H): o = Wd h for those rows, times the
//        routing weight -> obuf[slot]; the last B unit of a row block sums the
//        k slots of every token (j ascending) into y (bf16).
//    Weights stream straight from HBM or, for host-resident experts, from
//    pinned host memory over the C2C/PCIe link; host experts' units are
//    queued first so the slow link reads start earliest and overlap the HBM
//    work.  A B unit issues its weight loads before it waits for its expert's
//    A units (bounded wait).
//
// The MoE layer is that of "763B MoE in two 96 GB cards" (section "Where the
// VRAM gap comes from": per layer, a token is routed to k of E experts; the
// idle ones can live in host memory and be read by the GPU over UVA); the
// per-expert residence is the per-expert plan of its "Same idea, native vLLM
// fails" side-box.
#include <stdio.h>

#include <algorithm>

#include "internal.h"

using namespace moe;

namespace {

struct RouterArgs {
  const uint16_t* x;
  int T, H, E, k;
  const uint16_t* wr;
  const float* bias;
  float* logits;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* wl_expert;
  int32_t* wl_off;
  int32_t* wl_cnt;
  const uint8_t** wl_blob;
  unsigned* done_a;
  unsigned* done_b;
  int nb;
  Ctl* ctl;
  const uint8_t* const* blob_hbm;   // [E] of this layer
  const uint8_t* const* blob_host;  // [E] of this layer
  int64_t ge0;                      // global id of expert 0 of this layer
  int lfu;
  uint32_t* lfu_count;
  int32_t* lfu_last;
  int step;
  int32_t* miss_list;
  unsigned* miss_count;
  int miss_cap;
  unsigned long long* stats;  // this layer's counters
  int64_t expert_bytes, router_bytes;
  float* xsum;  // [T][H/G]: zcorr * (sum of x over each scale group), for the expert kernel
  int group;
  float zcorr;
  moe_routing_out dbg;
};

constexpr int kRouterWarps = 4;

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Logits in the fixed order: lane j accumulates, from +0, fmaf(x[i], w[i], acc)
// over i = 256m + 8j + r (m ascending, r ascending); the 32 lane sums are then
// combined by xor-butterfly adds with offsets 16, 8, 4, 2, 1 (every lane ends
// with the same value); the bias is added last.
__global__ void __launch_bounds__(kRouterWarps * 32)
router_decode_kernel(RouterArgs a) {
  extern __shared__ uint4 r_smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(r_smem);  // [T][H] bf16
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, H = a.H, E = a.E, k = a.k;

  // let the dependent expert kernel be scheduled now: its CTAs wait for this
  // grid's completion themselves (griddepcontrol.wait) and this grid never
  // waits on them
  asm volatile("griddepcontrol.launch_dependents;");

  {
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    const int n = T * H / 8;
    for (int i = tid; i < n; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();

  const int e = blockIdx.x * kRouterWarps + warp;
  if (e < E) {
    const uint4* w = reinterpret_cast<const uint4*>(a.wr + (int64_t)e * H);
    float acc[kDecodeMaxTokens];
#pragma unroll
    for (int t = 0; t < kDecodeMaxTokens; ++t) acc[t] = 0.0f;
    const int nm = H / 256;
    for (int m0 = 0; m0 < nm; m0 += 8) {
      uint4 wv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (m0 + q < nm) wv[q] = __ldg(w + (m0 + q) * 32 + lane);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
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

  // scale-group sums of x for the expert kernel: pair q = (t, group), one warp each
  {
    const int ng = H / a.group, npairs = T * ng;
    for (int q = blockIdx.x * kRouterWarps + warp; q < npairs; q += gridDim.x * kRouterWarps) {
      const int t = q / ng, grp = q % ng;
      float v = 0.f;
      for (int i = lane; i < a.group; i += 32) v += bf16f(xs[t * H + grp * a.group + i]);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) a.xsum[q] = a.zcorr * v;
    }
  }

  // ---- grid-wide completion: the last CTA does the rest
  __shared__ unsigned s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&a.ctl->ticket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  __shared__ int s_e[kDecodeMaxTokens * kMaxTopK];     // chosen expert per slot
  __shared__ float s_w[kDecodeMaxTokens * kMaxTopK];   // weight per slot
  __shared__ int s_rank[kDecodeMaxTokens * kMaxTopK];  // position of slot in perm
  __shared__ int s_perm[kDecodeMaxTokens * kMaxTopK];
  __shared__ int s_nd;

  // top-k, one warp per token: each lane keeps its own best 8 (logit desc,
  // index asc) over experts lane, lane+32, ...; then k rounds of warp argmax.
  for (int t = warp; t < T; t += kRouterWarps) {
    float lv[kMaxTopK];
    int li[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) { lv[j] = -INFINITY; li[j] = 0x7fffffff; }
    for (int base = 0; base < E; base += 32 * 16) {
      float vb[16];  // one round trip for 16 logits per lane
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int ee = base + q * 32 + lane;
        vb[q] = ee < E ? __ldcg(a.logits + t * E + ee) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int ee = base + q * 32 + lane;
        const float v = vb[q];
        // indices arrive ascending, so strict '>' keeps the lower index first on ties
        if (ee < E && (v > lv[kMaxTopK - 1] || li[kMaxTopK - 1] == 0x7fffffff)) {
          float cv = v;
          int ci = ee;
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j) {
            const bool better = (li[j] == 0x7fffffff) || (cv > lv[j]);
            if (better) {
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
        s_e[t * k + j] = bi;
        s_w[t * k + j] = bv;  // logit for now
      }
    }
    __syncwarp();
    if (lane == 0) {
      const float l0 = s_w[t * k];
      float ex[kMaxTopK];
      float z = 0.0f;
      for (int j = 0; j < k; ++j) {
        ex[j] = expf(s_w[t * k + j] - l0);
        z += ex[j];
      }
      for (int j = 0; j < k; ++j) s_w[t * k + j] = ex[j] / z;
    }
  }
  __syncthreads();

  const int n = T * k;
  // stable grouping: rank of slot s by key (expert, token)
  for (int s = tid; s < n; s += blockDim.x) {
    const int key = s_e[s] * T + s / k;
    int r = 0;
    for (int q = 0; q < n; ++q) r += (s_e[q] * T + q / k) < key;
    s_rank[s] = r;
    s_perm[r] = s;
  }
  __syncthreads();
  for (int s = tid; s < n; s += blockDim.x) {
    a.topk_idx[s] = s_e[s];
    a.topk_w[s] = s_w[s];
    a.perm[s] = s_perm[s];
    a.inv[s] = s_rank[s];
    if (a.dbg.topk_idx) a.dbg.topk_idx[s] = s_e[s];
    if (a.dbg.topk_w) a.dbg.topk_w[s] = s_w[s];
    if (a.dbg.perm) a.dbg.perm[s] = s_perm[s];
    if (a.dbg.inv) a.dbg.inv[s] = s_rank[s];
  }
  if (a.dbg.counts || a.dbg.offsets) {
    for (int ee = tid; ee <= E; ee += blockDim.x) {
      int below = 0, eq = 0;
      for (int q = 0; q < n; ++q) {
        below += s_e[q] < ee;
        eq += s_e[q] == ee;
      }
      if (a.dbg.offsets) a.dbg.offsets[ee] = below;
      if (a.dbg.counts && ee < E) a.dbg.counts[ee] = eq;
    }
  }
  if (a.dbg.logits)
    for (int i = tid; i < T * E; i += blockDim.x) a.dbg.logits[i] = __ldcg(a.logits + i);

  // distinct experts in ascending order, host-resident ones first: position p
  // of perm starts a distinct expert when its expert differs from p-1's
  __shared__ int s_first[kDecodeMaxTokens * kMaxTopK];  // 1 = HBM-first, 2 = host-first, 0 = not first
  __shared__ const uint8_t* s_blob[kDecodeMaxTokens * kMaxTopK];
  for (int p = tid; p < n; p += blockDim.x) {
    const int ee = s_e[s_perm[p]];
    int f = 0;
    if (p == 0 || s_e[s_perm[p - 1]] != ee) {
      const uint8_t* hb = a.blob_hbm[ee];
      f = hb ? 1 : 2;
      s_blob[p] = hb ? hb : a.blob_host[ee];
    }
    s_first[p] = f;
  }
  __syncthreads();
  for (int p = tid; p < n; p += blockDim.x) {
    const int f = s_first[p];
    if (!f) continue;
    int nh_all = 0, before = 0;
    for (int q = 0; q < n; ++q) {
      nh_all += s_first[q] == 2;
      before += q < p && s_first[q] == f;
    }
    const int slot = f == 2 ? before : nh_all + before;
    const int ee = s_e[s_perm[p]];
    int cnt = 1;
    while (p + cnt < n && s_first[p + cnt] == 0) ++cnt;
    a.wl_expert[slot] = ee;
    a.wl_off[slot] = p;
    a.wl_cnt[slot] = cnt;
    a.wl_blob[slot] = s_blob[p];
    if (a.lfu) {  // distinct experts: no two threads touch the same g
      const int64_t g = a.ge0 + ee;
      a.lfu_count[g] += 1u;
      a.lfu_last[g] = a.step;
      if (f == 2) {
        const unsigned mi = atomicAdd(a.miss_count, 1u);
        if ((int)mi < a.miss_cap) a.miss_list[mi] = (int32_t)g;
      }
    }
  }
  if (tid == 0) {
    int nd = 0, nh = 0;
    for (int q = 0; q < n; ++q) {
      nd += s_first[q] != 0;
      nh += s_first[q] == 2;
    }
    s_nd = nd;
    a.ctl->ndistinct = nd;
    a.ctl->nhost = nh;
    a.ctl->queue = 0;
    unsigned long long* st = a.stats;
    const unsigned long long v0 = st[kStatAccesses], v1 = st[kStatHits], v2 = st[kStatMisses],
                             v3 = st[kStatHbmBytes], v4 = st[kStatHostBytes], v5 = st[kStatPairs],
                             v6 = st[kStatForwards];
    st[kStatAccesses] = v0 + nd;
    st[kStatHits] = v1 + (nd - nh);
    st[kStatMisses] = v2 + nh;
    st[kStatHbmBytes] = v3 + (unsigned long long)(nd - nh) * a.expert_bytes + a.router_bytes;
    st[kStatHostBytes] = v4 + (unsigned long long)nh * a.expert_bytes;
    st[kStatPairs] = v5 + n;
    st[kStatForwards] = v6 + 1;
  }
  __syncthreads();
  for (int i = tid; i < s_nd; i += blockDim.x) a.done_a[i] = 0;
  for (int i = tid; i < a.nb; i += blockDim.x) a.done_b[i] = 0;
  if (tid == 0) a.ctl->ticket = 0;
  __threadfence();
}

// ------------------------------------------------------------ expert kernel
//
// Dot products run on mma.sync.m16n8k16 (bf16 x bf16 -> fp32): the weight
// tile is the A operand, decoded in registers; the (up to 8) tokens of the
// expert are the 8 columns of the B operand.  A code u is decoded as the
// bf16 value 128 + u (one mask-and-or yields two of them), so the tile
// product is  sum (128 + u) x = sum q x + (128 + 2^(b-1)) sum x  with
// q = u - 2^(b-1); the second term is subtracted per scale group from the
// fp32 accumulator.  All products are exact in fp32 (8-bit by 8-bit
// significands); accumulation is fp32.

struct MatOff {
  int64_t codes, scales;
};

struct ExpertArgs {
  const uint16_t* x;
  int T, H, I, k;
  int kpadI;  // I rounded up to a multiple of 256 (down-projection K)
  const int32_t* perm;
  const float* topk_w;
  const int32_t* wl_off;
  const int32_t* wl_cnt;
  const uint8_t* const* wl_blob;
  Ctl* ctl;
  unsigned* done_a;
  unsigned* done_b;
  float* hbuf;  // [maxD][tstride][I]
  int tstride;
  float* obuf;  // [T*k][H]
  uint16_t* y;
  MatOff m[3];
  int group, sdt;
  float zcorr;         // 128 + 2^(b-1)
  const float* xsum;   // [T][H/G] from the router: zcorr * group sums of x
  uint32_t* err;
  int nA, nB;
};

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float ld_scale(const uint8_t* base, int64_t idx, int sdt) {
  if (sdt == MOE_SCALE_F32) return __ldg(reinterpret_cast<const float*>(base) + idx);
  const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(base) + idx);
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

// bf16x2 register (128 + u_lo, 128 + u_hi) of pair P (0..63) of a lane's
// column block; w holds the lane's 4*B words; P is a compile-time constant
// after unrolling.  Field placement: see repack_codes_kernel in plan.cu.
template <int B>
__device__ __forceinline__ uint32_t pair_bits(const uint32_t (&w)[4 * B], int P) {
  constexpr uint32_t kMagic = 0x43004300u;  // bf16 128.0 in both halves
  if constexpr (B == 4) {
    return ((w[P >> 2] >> (4 * (P & 3))) & 0x000F000Fu) | kMagic;
  } else if constexpr (B == 2) {
    return ((w[P >> 3] >> (2 * (P & 7))) & 0x00030003u) | kMagic;
  } else {
    const int t = P >> 4, m = P & 15;
    if (m < 15) return ((w[3 * t + m / 5] >> (3 * (m % 5))) & 0x00070007u) | kMagic;
    return ((w[3 * t] >> 15) & 0x00010001u) | ((w[3 * t + 1] >> 14) & 0x00020002u) |
           ((w[3 * t + 2] >> 13) & 0x00040004u) | kMagic;
  }
}

template <int B>
__device__ __forceinline__ void words_of(const uint4 (&p)[B], uint32_t (&w)[4 * B]) {
#pragma unroll
  for (int q = 0; q < B; ++q) {
    w[4 * q + 0] = p[q].x;
    w[4 * q + 1] = p[q].y;
    w[4 * q + 2] = p[q].z;
    w[4 * q + 3] = p[q].w;
  }
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

// Group sums of the B operand rows: csum[g * 8 + t] = zcorr * sum_{k in group g} v_t[k]
// for t < Te (entries for t >= Te are left unset and never used for an
// output); one warp per (group, token), fixed order.
__device__ void group_sums(const uint16_t* hi, const uint16_t* lo, int stride, int K, int G,
                           int Te, float zcorr, float* csum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = K / G;
  for (int q = warp; q < ng * Te; q += kWarps) {  // only real tokens; others are never read
    const int g = q % ng, t = q / ng;
    float v = 0.f;
    for (int i = lane; i < G; i += 32) {
      const int k = g * G + i;
      v += bf16f(hi[t * stride + k]);
      if (lo) v += bf16f(lo[t * stride + k]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) csum[g * 8 + t] = zcorr * v;
  }
}

// A unit: rows [mt*16, mt*16+16) of Wg and Wu, all H columns, for the
// expert's Te tokens; warp w takes column blocks w, w+8, ...; warps are
// summed in order through shared memory; h = silu(g) * u -> hbuf.
template <int B>
__device__ void a_unit(const ExpertArgs& a, int d, int mt, uint8_t* smem, const int* toks, int Te) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int H = a.H, nkb = H / kBlockK, G = a.group, ng = H / G;
  const int xstride = H + 8;  // bf16 elements; the pad spreads rows over banks
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  float* csum = reinterpret_cast<float*>(smem + (size_t)a.T * xstride * 2);
  float* red = csum + ng * 8;
  float* ssc = red + kWarps * 256;  // [2][ng][16] gate / up scales of this row tile
  const uint8_t* blob = a.wl_blob[d];
  const uint8_t* gb = blob + a.m[0].codes + (int64_t)mt * nkb * B * 512 + lane * 16;
  const uint8_t* ub = blob + a.m[1].codes + (int64_t)mt * nkb * B * 512 + lane * 16;
  const int gpb = kBlockK / G;  // scale groups per block
  // two column blocks of this warp are in flight before x and the scales are
  // staged; the loop keeps two in flight (one body copy, rotating buffers)
  uint4 cg_[B], cu_[B], ng_[B], nu_[B];
  auto load = [&](uint4(&pg)[B], uint4(&pu)[B], int kb) {
    if (kb < nkb) {
#pragma unroll
      for (int q = 0; q < B; ++q) {
        pg[q] = ld_stream(gb + ((int64_t)kb * B + q) * 512);
        pu[q] = ld_stream(ub + ((int64_t)kb * B + q) * 512);
      }
    }
  };
  load(cg_, cu_, warp);
  load(ng_, nu_, warp + kWarps);
  for (int i = tid; i < 2 * ng * kTileRows; i += blockDim.x) {
    const int m = i / (ng * kTileRows), j = i % (ng * kTileRows);
    ssc[i] = ld_scale(blob + a.m[m].scales, (int64_t)mt * ng * kTileRows + j, a.sdt);
  }
  for (int i = tid; i < Te * (H / 8); i += blockDim.x) {
    const int t = i / (H / 8), c = i % (H / 8);
    *reinterpret_cast<uint4*>(xs + t * xstride + c * 8) =
        *reinterpret_cast<const uint4*>(a.x + (int64_t)toks[t] * H + c * 8);
  }
  for (int i = tid; i < ng * Te; i += blockDim.x) {
    const int grp = i % ng, t = i / ng;
    csum[grp * 8 + t] = __ldcg(a.xsum + (int64_t)toks[t] * ng + grp);
  }
  __syncthreads();

  const bool tv = g < Te;  // this lane's B-operand column is a real token
  const uint16_t* xrow = xs + g * xstride + 2 * tig;
  float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int kb = warp; kb < nkb; kb += kWarps) {
    uint32_t wg[4 * B], wu[4 * B];
    words_of<B>(cg_, wg);
    words_of<B>(cu_, wu);
#pragma unroll
    for (int q = 0; q < B; ++q) {
      cg_[q] = ng_[q];
      cu_[q] = nu_[q];
    }
    load(ng_, nu_, kb + 2 * kWarps);
    float cg[4] = {0.f, 0.f, 0.f, 0.f}, cu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kt = 0; kt < 16; ++kt) {
      const int k0 = kb * kBlockK + kt * 16;
      const uint32_t b0 = tv ? *reinterpret_cast<const uint32_t*>(xrow + k0) : 0u;
      const uint32_t b1 = tv ? *reinterpret_cast<const uint32_t*>(xrow + k0 + 8) : 0u;
      mma_bf16(cg, pair_bits<B>(wg, 4 * kt), pair_bits<B>(wg, 4 * kt + 1),
               pair_bits<B>(wg, 4 * kt + 2), pair_bits<B>(wg, 4 * kt + 3), b0, b1);
      mma_bf16(cu, pair_bits<B>(wu, 4 * kt), pair_bits<B>(wu, 4 * kt + 1),
               pair_bits<B>(wu, 4 * kt + 2), pair_bits<B>(wu, 4 * kt + 3), b0, b1);
      if (((kt + 1) * 16) % G == 0) {  // end of a scale group
        const int grp = kb * gpb + ((kt + 1) * 16) / G - 1;
        const float* sg = ssc + grp * kTileRows + g;
        const float* su = sg + ng * kTileRows;
        const float z0 = csum[grp * 8 + 2 * tig], z1 = csum[grp * 8 + 2 * tig + 1];
        accg[0] = fmaf(sg[0], cg[0] - z0, accg[0]);
        accg[1] = fmaf(sg[0], cg[1] - z1, accg[1]);
        accg[2] = fmaf(sg[8], cg[2] - z0, accg[2]);
        accg[3] = fmaf(sg[8], cg[3] - z1, accg[3]);
        accu[0] = fmaf(su[0], cu[0] - z0, accu[0]);
        accu[1] = fmaf(su[0], cu[1] - z1, accu[1]);
        accu[2] = fmaf(su[8], cu[2] - z0, accu[2]);
        accu[3] = fmaf(su[8], cu[3] - z1, accu[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) cg[i] = cu[i] = 0.f;
      }
    }
  }
  // red[w][m][row][token], m = 0 gate / 1 up
  float* rw = red + warp * 2 * 128;
  rw[g * 8 + 2 * tig] = accg[0];
  rw[g * 8 + 2 * tig + 1] = accg[1];
  rw[(g + 8) * 8 + 2 * tig] = accg[2];
  rw[(g + 8) * 8 + 2 * tig + 1] = accg[3];
  rw[128 + g * 8 + 2 * tig] = accu[0];
  rw[128 + g * 8 + 2 * tig + 1] = accu[1];
  rw[128 + (g + 8) * 8 + 2 * tig] = accu[2];
  rw[128 + (g + 8) * 8 + 2 * tig + 1] = accu[3];
  __syncthreads();
  if (tid < 128) {
    const int row = tid >> 3, t = tid & 7;
    if (t < Te) {
      float gv = 0.f, uv = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        gv += red[w * 256 + tid];
        uv += red[w * 256 + 128 + tid];
      }
      a.hbuf[((int64_t)d * a.tstride + t) * a.I + mt * kTileRows + row] =
          gv / (1.0f + expf(-gv)) * uv;
    }
  }
  __syncthreads();
}

// B unit: rows [ub*128, ub*128+128) of Wd (warp w: row tile ub*8 + w), all
// columns, for the expert's tokens.  h is split into bf16 hi + lo parts (two
// MMAs per step), so the down projection sees h to ~16 significant bits.
// The weight loads are issued before the wait on the expert's A units.
template <int B>
__device__ bool b_unit(const ExpertArgs& a, int d, int ub, uint8_t* smem, const int* slots,
                       int Te, int* s_flag) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int I = a.I, KP = a.kpadI, nkb = KP / kBlockK, G = a.group, ng = KP / G;
  const int hstride = KP + 8;
  uint16_t* hh = reinterpret_cast<uint16_t*>(smem);
  uint16_t* hl = hh + (size_t)a.T * hstride;
  float* csum = reinterpret_cast<float*>(hl + (size_t)a.T * hstride);
  float* ssc = csum + ng * 8;  // [8 row tiles][ng][16] scales of this unit
  const int mtg = ub * (kBRows / kTileRows) + warp;
  const uint8_t* blob = a.wl_blob[d];
  const uint8_t* db = blob + a.m[2].codes + (int64_t)mtg * nkb * B * 512 + lane * 16;
  const uint8_t* ds = blob + a.m[2].scales;
  constexpr int kPre = 4;  // column blocks loaded before the wait, then kept in flight
  const int gpb = kBlockK / G;
  uint4 q0[B], q1[B], q2[B], q3[B];
  auto load = [&](uint4(&p)[B], int kb) {
    if (kb < nkb) {
#pragma unroll
      for (int q = 0; q < B; ++q) p[q] = ld_stream(db + ((int64_t)kb * B + q) * 512);
    }
  };
  load(q0, 0);
  load(q1, 1);
  load(q2, 2);
  load(q3, 3);
  {
    const int64_t s0 = (int64_t)ub * (kBRows / kTileRows) * ng * kTileRows;
    for (int i = tid; i < (kBRows / kTileRows) * ng * kTileRows; i += blockDim.x)
      ssc[i] = ld_scale(ds, s0 + i, a.sdt);
  }
  if (tid == 0) *s_flag = wait_count(&a.done_a[d], (unsigned)a.nA, a.err) ? 1 : 0;
  __syncthreads();
  if (!*s_flag) return false;
  for (int i = tid; i < Te * KP; i += blockDim.x) {
    const int t = i / KP, k = i % KP;
    const float v = k < I ? __ldcg(a.hbuf + ((int64_t)d * a.tstride + t) * I + k) : 0.f;
    const __nv_bfloat16 vh = __float2bfloat16_rn(v);
    const __nv_bfloat16 vl = __float2bfloat16_rn(v - __bfloat162float(vh));
    hh[t * hstride + k] = __bfloat16_as_ushort(vh);
    hl[t * hstride + k] = __bfloat16_as_ushort(vl);
  }
  __syncthreads();
  group_sums(hh, hl, hstride, KP, G, Te, a.zcorr, csum);
  __syncthreads();
  const bool tv = g < Te;
  const uint16_t* hrow = hh + g * hstride + 2 * tig;
  const uint16_t* lrow = hl + g * hstride + 2 * tig;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const float* wsc = ssc + warp * ng * kTileRows + g;  // this warp's row tile, row g
#pragma unroll 1
  for (int kb = 0; kb < nkb; ++kb) {
    uint32_t w[4 * B];
    words_of<B>(q0, w);
#pragma unroll
    for (int q = 0; q < B; ++q) {
      q0[q] = q1[q];
      q1[q] = q2[q];
      q2[q] = q3[q];
    }
    load(q3, kb + kPre);
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kt = 0; kt < 16; ++kt) {
      const int k0 = kb * kBlockK + kt * 16;
      const uint32_t a0 = pair_bits<B>(w, 4 * kt), a1 = pair_bits<B>(w, 4 * kt + 1);
      const uint32_t a2 = pair_bits<B>(w, 4 * kt + 2), a3 = pair_bits<B>(w, 4 * kt + 3);
      const uint32_t h0 = tv ? *reinterpret_cast<const uint32_t*>(hrow + k0) : 0u;
      const uint32_t h1 = tv ? *reinterpret_cast<const uint32_t*>(hrow + k0 + 8) : 0u;
      const uint32_t l0 = tv ? *reinterpret_cast<const uint32_t*>(lrow + k0) : 0u;
      const uint32_t l1 = tv ? *reinterpret_cast<const uint32_t*>(lrow + k0 + 8) : 0u;
      mma_bf16(c, a0, a1, a2, a3, h0, h1);
      mma_bf16(c, a0, a1, a2, a3, l0, l1);
      if (((kt + 1) * 16) % G == 0) {  // end of a scale group
        const int grp = kb * gpb + ((kt + 1) * 16) / G - 1;
        const float s0 = wsc[grp * kTileRows], s1 = wsc[grp * kTileRows + 8];
        const float z0 = csum[grp * 8 + 2 * tig], z1 = csum[grp * 8 + 2 * tig + 1];
        acc[0] = fmaf(s0, c[0] - z0, acc[0]);
        acc[1] = fmaf(s0, c[1] - z1, acc[1]);
        acc[2] = fmaf(s1, c[2] - z0, acc[2]);
        acc[3] = fmaf(s1, c[3] - z1, acc[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = 0.f;
      }
    }
  }
  const int H = a.H;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = 2 * tig + (i & 1);
    const int row = mtg * kTileRows + g + 8 * (i >> 1);
    if (t < Te) {
      const int s = slots[t];
      a.obuf[(int64_t)s * H + row] = a.topk_w[s] * acc[i];
    }
  }
  __syncthreads();
  return true;
}

// The last B unit of row block ub (over all D experts) sums each token's k
// weighted slot outputs, j ascending, into y.
__device__ void combine_rows(const ExpertArgs& a, int ub, unsigned D, int* s_flag) {
  const int tid = threadIdx.x;
  __threadfence();
  __syncthreads();
  if (tid == 0) *s_flag = (atomicAdd(&a.done_b[ub], 1u) == D - 1) ? 2 : 0;
  __syncthreads();
  if (*s_flag != 2) return;
  __threadfence();
  const int k = a.k, H = a.H;
  for (int i = tid; i < a.T * kBRows; i += blockDim.x) {
    const int t = i / kBRows, row = ub * kBRows + i % kBRows;
    float v = 0.f;
    for (int j = 0; j < k; ++j) v += __ldcg(a.obuf + (int64_t)(t * k + j) * H + row);
    a.y[(int64_t)t * H + row] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

template <int B>
__global__ void __launch_bounds__(kWarps * 32, 2)
expert_decode_kernel(ExpertArgs a) {
  extern __shared__ __align__(16) uint8_t e_smem[];
  __shared__ unsigned s_unit;
  __shared__ int s_toks[kDecodeMaxTokens], s_slots[kDecodeMaxTokens];
  __shared__ int s_flag;
  const int tid = threadIdx.x;
  // wait for the router (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const unsigned D = *reinterpret_cast<volatile unsigned*>(&a.ctl->ndistinct);
  const unsigned total = D * (unsigned)(a.nA + a.nB);
  for (;;) {
    if (tid == 0) s_unit = atomicAdd(&a.ctl->queue, 1u);
    __syncthreads();
    const unsigned u = s_unit;
    if (u >= total) break;
    const bool isA = u < D * (unsigned)a.nA;
    const unsigned v = isA ? u : u - D * (unsigned)a.nA;
    const int d = (int)(v / (unsigned)(isA ? a.nA : a.nB));
    const int r = (int)(v % (unsigned)(isA ? a.nA : a.nB));
    const int Te = a.wl_cnt[d];
    if (tid < Te) {
      const int s = a.perm[a.wl_off[d] + tid];
      s_slots[tid] = s;
      s_toks[tid] = s / a.k;
    }
    __syncthreads();
    if (isA) {
      a_unit<B>(a, d, r, e_smem, s_toks, Te);
      __threadfence();
      __syncthreads();
      if (tid == 0) atomicAdd(&a.done_a[d], 1u);
    } else if (b_unit<B>(a, d, r, e_smem, s_slots, Te, &s_flag)) {
      combine_rows(a, r, D, &s_flag);
    }
    __syncthreads();
  }
}

template <int B>
cudaError_t launch_expert(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s) {
  auto kern = expert_decode_kernel<B>;
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
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

cudaError_t moe::decode_forward(Plan& p, int layer, const uint16_t* x, int T, uint16_t* y,
                                cudaStream_t s, const moe_routing_out* dbg) {
  const moe_plan_desc& d = p.d;
  const int E = d.num_experts, H = d.hidden, I = d.inter, k = d.top_k;
  const int64_t ge0 = (int64_t)layer * E;
  RouterArgs r{};
  r.x = x;
  r.T = T;
  r.H = H;
  r.E = E;
  r.k = k;
  r.wr = p.wr[layer];
  r.bias = p.bias[layer];
  r.logits = p.logits;
  r.topk_idx = p.topk_idx;
  r.topk_w = p.topk_w;
  r.counts = p.counts;
  r.offsets = p.offsets;
  r.perm = p.perm;
  r.inv = p.inv;
  r.wl_expert = p.wl_expert;
  r.wl_off = p.wl_off;
  r.wl_cnt = p.wl_cnt;
  r.wl_blob = p.wl_blob;
  r.done_a = p.done_a;
  r.done_b = p.done_b;
  r.nb = H / kBRows;
  r.ctl = p.ctl;
  r.blob_hbm = p.blob_hbm + ge0;
  r.blob_host = p.blob_host + ge0;
  r.ge0 = ge0;
  r.lfu = d.cache_policy == MOE_POLICY_LFU;
  r.lfu_count = p.lfu_count;
  r.lfu_last = p.lfu_last;
  r.step = p.step;
  r.miss_list = p.miss_list;
  r.miss_count = p.miss_count;
  r.miss_cap = d.num_layers * p.max_distinct;
  r.stats = p.stats + (int64_t)layer * kNumStats;
  r.expert_bytes = p.lay.algo_bytes;
  r.router_bytes = (int64_t)E * H * 2;
  r.xsum = p.xsum;
  r.group = d.group_size;
  r.zcorr = 128.0f + (float)(1 << (d.weight_bits - 1));
  if (dbg) r.dbg = *dbg;
  const int rgrid = (E + kRouterWarps - 1) / kRouterWarps;
  const size_t rsmem = (size_t)T * H * 2;
  cudaError_t e = cudaFuncSetAttribute(router_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsmem);
  if (e != cudaSuccess) return e;
  router_decode_kernel<<<rgrid, kRouterWarps * 32, rsmem, s>>>(r);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  ExpertArgs a{};
  a.x = x;
  a.T = T;
  a.H = H;
  a.I = I;
  a.k = k;
  a.perm = p.perm;
  a.topk_w = p.topk_w;
  a.wl_off = p.wl_off;
  a.wl_cnt = p.wl_cnt;
  a.wl_blob = p.wl_blob;
  a.ctl = p.ctl;
  a.done_a = p.done_a;
  a.done_b = p.done_b;
  a.hbuf = p.hbuf;
  a.tstride = std::min(d.max_tokens, kDecodeMaxTokens);
  a.obuf = p.obuf;
  a.y = y;
  for (int m = 0; m < 3; ++m) {
    a.m[m].codes = p.lay.m[m].codes_off;
    a.m[m].scales = p.lay.m[m].scales_off;
  }
  a.group = d.group_size;
  a.sdt = d.scale_dtype;
  a.zcorr = 128.0f + (float)(1 << (d.weight_bits - 1));
  a.xsum = p.xsum;
  a.err = p.err_dev;
  a.kpadI = p.lay.m[2].kpad;
  a.nA = I / kTileRows;
  a.nB = H / kBRows;
  const size_t smem_a = (size_t)T * (H + 8) * 2 + (size_t)(H / d.group_size) * 8 * 4 +
                        (size_t)kWarps * 256 * 4 + (size_t)2 * (H / d.group_size) * kTileRows * 4;
  const size_t smem_b = (size_t)2 * T * (a.kpadI + 8) * 2 + (size_t)(a.kpadI / d.group_size) * 8 * 4 +
                        (size_t)(kBRows / kTileRows) * (a.kpadI / d.group_size) * kTileRows * 4;
  const size_t smem = (std::max(smem_a, smem_b) + 15) / 16 * 16;
  const int maxD = std::min(E, T * k);
  const int units = maxD * (a.nA + a.nB);
  int per_sm = 0;
  const void* kfn = d.weight_bits == 2   ? (const void*)expert_decode_kernel<2>
                    : d.weight_bits == 3 ? (const void*)expert_decode_kernel<3>
                                         : (const void*)expert_decode_kernel<4>;
  e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, kWarps * 32, smem);
  if (e != cudaSuccess) return e;
  per_sm = std::max(1, std::min(per_sm, 4));
  const int grid = std::max(1, std::min(units, p.sms * per_sm));
  switch (d.weight_bits) {
    case 2: return launch_expert<2>(a, grid, smem, s);
    case 3: return launch_expert<3>(a, grid, smem, s);
    default: return launch_expert<4>(a, grid, smem, s);
  }
}
