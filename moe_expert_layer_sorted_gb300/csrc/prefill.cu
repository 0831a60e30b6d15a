// Prefill-batch forward (T > 8 tokens), the shape of "763B MoE in two 96 GB
// cards" (section "Where the VRAM gap comes from": each token routed to k of
// E experts, the layer output the routing-weighted sum of the experts'
// SwiGLU FFNs), as six launches on the caller's stream:
//
//   1. pf_router_kernel   fp32 router logits in the library's fixed summation
//                         order (lane j of a warp owns elements 256m + 8j + r;
//                         xor-butterfly; bias last), tiled 16 tokens x 16
//                         experts per CTA, operands staged as fp32.
//   2. pf_topk_kernel     per token: k largest logits (ties -> lower expert
//                         index), softmax renormalised over the k.
//   3. pf_count_kernel / pf_scan_kernel / pf_place_kernel
//                         grouping by expert: per-expert counts, exclusive
//                         offsets, and the stable (expert, token) order perm /
//                         inv, one CTA per expert compacting the slots in
//                         ascending order.
//   4. pf_gemm_kernel<gate/up>  for every routed (expert, 128 rows of I,
//                         <= 256 of its tokens): gate and up projections on
//                         tcgen05 tensor cores with fp32 accumulators in TMEM;
//                         the epilogue writes h = silu(g) * u (bf16) per
//                         (token, expert) slot.
//   5. pf_gemm_kernel<down>  o = Wd h per (expert, 128 rows of H, tokens),
//                         times the slot's routing weight, bf16 per slot.
//   6. pf_combine_kernel  y[t] = sum over j ascending of the slot outputs, bf16.
//
// GEMM kernel layout (one CTA of 9 warps per SM, persistent over work units):
//   warps 0-3  producers: dequantise the unit's 128 weight rows x 64 columns
//              per stage (int-b codes in the library's fragment-ordered device
//              layout -> bf16 s*q) and gather its token rows, both into
//              128-byte-swizzled K-major shared memory tiles;
//   warp 8     allocates TMEM and (lane 0) issues tcgen05.mma (M = 128 weight
//              rows, N = tokens, K = 16 per instruction) per stage, releasing
//              the stage by tcgen05.commit;
//   warps 4-7  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//              lanes 32(w%4)..+31, i.e. weight rows), activation / scaling,
//              global stores.
// Stages and the accumulator hand-off are tracked by mbarriers; every wait is
// bounded and latches the plan's error word.
#include <stdio.h>

#include <algorithm>

#include "internal.h"

using namespace moe;

namespace {

#include "device_common.cuh"

// ------------------------------------------------------------------ router

constexpr int kRtTile = 16;  // tokens and experts per router CTA

// xs/ws element (j, r) of a 256-wide block is stored at float4 index (r/4)*32 + j
// so that the lanes' 16-byte reads are conflict-free.
__global__ void __launch_bounds__(256) pf_router_kernel(const uint16_t* __restrict__ x, int T, int H,
                                                        const uint16_t* __restrict__ wr,
                                                        const float* __restrict__ bias, int E,
                                                        float* __restrict__ logits) {
  __shared__ float4 xs[kRtTile][64];
  __shared__ float4 ws[kRtTile][64];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kRtTile, e0 = blockIdx.y * kRtTile;
  const int tw = (warp & 3) * 4, ew = (warp >> 2) * 8;  // warp tile: 4 tokens x 8 experts
  float acc[4][8];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
  for (int m = 0; m < H / 256; ++m) {
    // stage: 16 rows x 32 uint4 of each operand; item i -> (operand, row, chunk j)
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int op = h >> 1, i = tid + (h & 1) * 256;  // i in 0..511
      const int row = i >> 5, j = i & 31;
      uint4 v = make_uint4(0, 0, 0, 0);
      const uint16_t* src = op == 0 ? x : wr;
      const int lim = op == 0 ? T : E;
      const int r0 = (op == 0 ? t0 : e0) + row;
      if (r0 < lim) v = *reinterpret_cast<const uint4*>(src + (int64_t)r0 * H + m * 256 + j * 8);
      float4* dst = op == 0 ? xs[row] : ws[row];
      dst[j] = make_float4(bf16f(v.x & 0xffffu), bf16f(v.x >> 16), bf16f(v.y & 0xffffu), bf16f(v.y >> 16));
      dst[32 + j] = make_float4(bf16f(v.z & 0xffffu), bf16f(v.z >> 16), bf16f(v.w & 0xffffu), bf16f(v.w >> 16));
    }
    __syncthreads();
    float xv[4][8], wv[8][8];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float4 p = xs[tw + a][lane], q = xs[tw + a][32 + lane];
      xv[a][0] = p.x; xv[a][1] = p.y; xv[a][2] = p.z; xv[a][3] = p.w;
      xv[a][4] = q.x; xv[a][5] = q.y; xv[a][6] = q.z; xv[a][7] = q.w;
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const float4 p = ws[ew + b][lane], q = ws[ew + b][32 + lane];
      wv[b][0] = p.x; wv[b][1] = p.y; wv[b][2] = p.z; wv[b][3] = p.w;
      wv[b][4] = q.x; wv[b][5] = q.y; wv[b][6] = q.z; wv[b][7] = q.w;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(xv[a][r], wv[b][r], acc[a][b]);
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      float v = acc[a][b];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
      const int t = t0 + tw + a, e = e0 + ew + b;
      if (lane == ((a * 8 + b) & 31) && t < T && e < E) logits[(int64_t)t * E + e] = v + bias[e];
    }
}

// One warp per token: k rounds of (lane's best untaken logit, warp max by an
// order-preserving key, warp min of the index among the lanes holding it);
// lanes scan experts lane, lane+32, ... so ties resolve to the lower index.
__global__ void pf_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                               int32_t* __restrict__ idx, float* __restrict__ wout) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* l = logits + (int64_t)t * E;
  int chosen[kMaxTopK];
  float cv[kMaxTopK];
  for (int j = 0; j < k; ++j) {
    uint32_t best = 0u;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      bool taken = false;
      for (int q = 0; q < j; ++q) taken |= chosen[q] == e;
      if (taken) continue;
      const float v = l[e];
      const uint32_t ub = __float_as_uint(v == 0.0f ? 0.0f : v);
      const uint32_t key = (ub & 0x80000000u) ? ~ub : (ub | 0x80000000u);
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
  if (lane == 0) {
    float ex[kMaxTopK];
    float z = 0.0f;
    for (int j = 0; j < k; ++j) {
      ex[j] = expf(cv[j] - cv[0]);
      z += ex[j];
    }
    for (int j = 0; j < k; ++j) {
      idx[(int64_t)t * k + j] = chosen[j];
      wout[(int64_t)t * k + j] = ex[j] / z;
    }
  }
}

// ------------------------------------------------------------------ grouping

// Block-wide exclusive prefix of a 0/1 flag over blockDim.x (multiple of 32)
// threads; returns the prefix and the block total in *tot.
__device__ int block_prefix(int flag, int* wsum, int* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned b = __ballot_sync(0xffffffffu, flag);
  const int inwarp = __popc(b & ((1u << lane) - 1u));
  if (lane == 0) wsum[warp] = __popc(b);
  __syncthreads();
  int before = 0, all = 0;
  for (int w = 0; w < nw; ++w) {
    const int c = wsum[w];
    before += w < warp ? c : 0;
    all += c;
  }
  __syncthreads();
  *tot = all;
  return before + inwarp;
}

__global__ void pf_count_kernel(const int32_t* __restrict__ idx, int n, int32_t* __restrict__ counts) {
  __shared__ int wsum[32];
  const int e = blockIdx.x;
  int total = 0;
  for (int s0 = 0; s0 < n; s0 += blockDim.x) {
    const int s = s0 + threadIdx.x;
    int tot;
    block_prefix(s < n && idx[s] == e, wsum, &tot);
    total += tot;
  }
  if (threadIdx.x == 0) counts[e] = total;
}

__global__ void pf_scan_kernel(const int32_t* __restrict__ counts, int E, int32_t* __restrict__ offsets) {
  if (threadIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      offsets[e] = run;
      run += counts[e];
    }
    offsets[E] = run;
  }
}

// perm[offsets[e] + r] = the r-th slot (ascending) routed to e; inv is its inverse
__global__ void pf_place_kernel(const int32_t* __restrict__ idx, int n, const int32_t* __restrict__ offsets,
                                int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  __shared__ int wsum[32];
  const int e = blockIdx.x;
  int base = offsets[e];
  for (int s0 = 0; s0 < n; s0 += blockDim.x) {
    const int s = s0 + threadIdx.x;
    const bool f = s < n && idx[s] == e;
    int tot;
    const int r = block_prefix(f, wsum, &tot);
    if (f) {
      perm[base + r] = s;
      inv[s] = base + r;
    }
    base += tot;
  }
}

// ------------------------------------------------------------------ tcgen05 GEMM

constexpr int kProdWarps = 8;                       // producer warps (0..7)
constexpr int kEpiWarp0 = kProdWarps;               // epilogue warps kEpiWarp0..+3
constexpr int kMmaWarp = kProdWarps + 4;            // TMEM allocation and MMA issue
constexpr int kGemmThreads = (kProdWarps + 5) * 32;
constexpr int kTileM = 128;        // weight rows per unit
constexpr int kTileN = 192;        // max tokens per unit
constexpr int kStageK = 64;        // columns per stage (one 128-byte swizzle span of bf16)

struct GemmArgs {
  int E, k, bits, group, sdt;
  int K, kpad;       // reduction length (H or I) and its padded length in the device layout
  int rows;          // weight rows of the matrix (I for gate/up, H for down)
  int64_t codes[2], scales[2];  // matrix sections in an expert blob (gate, up) or (down, -)
  const uint8_t* const* blob_hbm;
  const uint8_t* const* blob_host;
  const int32_t* offsets;  // [E+1]
  const int32_t* perm;     // [T*k] slots in (expert, token) order
  const uint16_t* x;       // gate/up: layer input [T][H]
  const uint16_t* hin;     // down: h [T*k][I] per perm position
  const float* topk_w;     // down: routing weight per slot
  uint16_t* hout;          // gate/up: h [T*k][I]
  uint16_t* oout;          // down: weighted o [T*k][H]
  int64_t out_ld;          // row pitch of the output (I or H)
  int nstages;             // shared-memory ring depth
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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// byte offset of (row, 16-byte chunk) in a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return (uint32_t)row * 128u + (uint32_t)((chunk ^ (row & 7)) << 4);
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

template <int B, bool GATEUP>
__global__ void __launch_bounds__(kGemmThreads, 1) pf_gemm_kernel(GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  __shared__ __align__(8) unsigned long long fullb[4], emptyb[4], tfull[2], tempty[2];
  __shared__ uint32_t tmem_base;
  __shared__ int rowsrc[kTileN];     // source row of each token of the current unit (producers)
  __shared__ float wslot[2][kTileN]; // down: routing weight of each token of a unit (epilogue)
  constexpr int NMAT = GATEUP ? 2 : 1;
  constexpr int NBUF = GATEUP ? 1 : 2;  // accumulator buffers in TMEM (512 columns either way)
  constexpr uint32_t kATile = kTileM * 128;  // bytes of one 128 x 64 bf16 weight tile
  constexpr uint32_t kBTile = kTileN * 128;
  // per stage, after the tiles: the stage's code words (each lane's 16-byte
  // share of each (row tile, matrix)) and scale rows, fetched two stages ahead
  constexpr uint32_t kCodes = NMAT * 8 * 32 * 16;
  constexpr uint32_t kScales = NMAT * 8 * 2 * 64;
  constexpr uint32_t kStage = NMAT * kATile + kBTile + kCodes + kScales;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the dynamic window is 1024-aligned for the swizzled tiles
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  const int E = a.E, NS = a.nstages;
  int* tile_prefix = reinterpret_cast<int*>(smem + (size_t)NS * kStage);  // [E+1] units before expert e
  const int mtiles = a.rows / kTileM;
  const int S = a.kpad / kStageK;  // stages per unit
  const int nkb = a.kpad / 256;
  const int G = a.group;

  // unit table: expert e contributes mtiles * ceil(n_e / 256) units
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      tile_prefix[e] = run;
      const int n = a.offsets[e + 1] - a.offsets[e];
      run += mtiles * ((n + kTileN - 1) / kTileN);
    }
    tile_prefix[E] = run;
    for (int q = 0; q < NS; ++q) {
      mbar_init(smem_addr(&fullb[q]), kProdWarps * 32);
      mbar_init(smem_addr(&emptyb[q]), 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(smem_addr(&tfull[q]), 1);
      mbar_init(smem_addr(&tempty[q]), 128);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {  // TMEM: 512 fp32 accumulator columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                 "n"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const int nunits = tile_prefix[E];

  auto decode_unit = [&](int u, int& e, int& mt, int& n0, int& nrows) {
    int lo = 0, hi = E - 1;  // last e with tile_prefix[e] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_prefix[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    const int r = u - tile_prefix[e];
    mt = r % mtiles;
    const int nt = r / mtiles;
    const int ne = a.offsets[e + 1] - a.offsets[e];
    n0 = a.offsets[e] + nt * kTileN;
    nrows = min(kTileN, ne - nt * kTileN);
  };

  if (warp < kProdWarps) {
    // ------------------------------------------------------------ producers
    // Per stage: the token rows of stage s+1 are requested (cp.async) and the
    // codes and scales of stage s+1 loaded into registers while stage s's
    // weights are dequantised into shared memory, so global latency overlaps
    // a stage of work.
    constexpr int NIT = NMAT * 8 / kProdWarps;  // (row tile, matrix) items per warp per stage
    const int g = lane >> 2, tig = lane & 3;
    uint32_t offc[8];  // swizzled byte offset of the lane's 4 bytes in 16-byte chunk c of rows g, g+8
#pragma unroll
    for (int c = 0; c < 8; ++c) offc[c] = (uint32_t)(((c ^ (g & 7)) << 4) + 4 * tig);
    const bool bfs = a.sdt == MOE_SCALE_BF16;
    const int ssz = a.sdt == MOE_SCALE_F32 ? 4 : 2;
    const float zb = 128.0f + (float)(1 << (a.bits - 1));
    const uint32_t negzb2 = pack_bf16x2(-zb, -zb);  // exact: 130, 132 or 136
    const int64_t ng = a.kpad / G;
    const uint16_t* bsrc = GATEUP ? a.x : a.hin;
    int gs = 0;  // stages produced so far (all units)
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      int e, mt, n0, nrows;
      decode_unit(u, e, mt, n0, nrows);
      const int N = (nrows + 15) & ~15;
      const uint8_t* hb = a.blob_hbm[e];
      const uint8_t* blob = hb ? hb : a.blob_host[e];
      asm volatile("bar.sync 2, %0;" ::"n"(kProdWarps * 32) : "memory");  // previous unit's rows unused now
      for (int n = tid; n < kTileN; n += kProdWarps * 32) {
        int src = -1;
        if (n < nrows) src = GATEUP ? a.perm[n0 + n] / a.k : n0 + n;
        rowsrc[n] = src;
      }
      asm volatile("bar.sync 2, %0;" ::"n"(kProdWarps * 32) : "memory");
      // every global read of stage s2 into its slot: token rows, code words, scale rows
      auto fetch = [&](int s2) {
        const int gsl = gs + s2, slot = gsl % NS, use = gsl / NS;
        if (use > 0) mbar_wait(smem_addr(&emptyb[slot]), (uint32_t)(use - 1) & 1u, a.err);
        uint8_t* st = smem + (size_t)slot * kStage;
        uint8_t* bt = st + NMAT * kATile;
        const int k0 = s2 * kStageK;
        for (int c = tid; c < N * 8; c += kProdWarps * 32) {
          const int n = c >> 3, cc = c & 7;
          const int src = rowsrc[n], col = k0 + cc * 8;
          uint8_t* dst = bt + sw128(n, cc);
          if (src >= 0 && col < a.K) cp_async16(dst, bsrc + (int64_t)src * a.K + col);
          else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
        const int kb = s2 >> 2, q = s2 & 3;
        uint8_t* cw = st + NMAT * kATile + kBTile;
        uint8_t* sw = cw + kCodes;
#pragma unroll
        for (int j = 0; j < NIT; ++j) {
          const int it = warp + kProdWarps * j, mat = it / 8, rt = it % 8;
          const int64_t tile = (int64_t)mt * 8 + rt;
          const uint8_t* chunk = blob + a.codes[mat] + (tile * nkb + kb) * B * 512 + lane * 16;
          uint8_t* dw = cw + (it * 32 + lane) * 16;
          if constexpr (B == 4) {
            cp_async16(dw, chunk + q * 512);
          } else if constexpr (B == 2) {
            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dw)),
                         "l"(chunk + (q >> 1) * 512 + (q & 1) * 8) : "memory");
          } else {
#pragma unroll
            for (int i = 0; i < 3; ++i) {
              const int wi = 3 * q + i;
              asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dw + 4 * i)),
                           "l"(chunk + (wi >> 2) * 512 + (wi & 3) * 4) : "memory");
            }
          }
          // scale rows of the stage's two 32-column halves (16 rows each); lanes
          // 0..7 copy the 16-byte pieces
          if (lane < 8) {
            const int h = lane >> 2, piece = lane & 3;
            const int gi = (kb * 256 + q * 64 + 32 * h) / G;
            if (piece * 16 < 16 * ssz)
              cp_async16(sw + (it * 2 + h) * 64 + piece * 16,
                         blob + a.scales[mat] + (tile * ng + gi) * 16 * ssz + piece * 16);
          }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      };
      fetch(0);
      if (S > 1) fetch(1);
      for (int s = 0; s < S; ++s) {
        const int slot = (gs + s) % NS;
        // stage s+1's reads may still be in flight; stage s's have landed
        if (s + 1 < S) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncwarp();  // scale rows were fetched by other lanes of this warp
        uint8_t* st = smem + (size_t)slot * kStage;
        const uint8_t* cw = st + NMAT * kATile + kBTile;
        const uint8_t* sw = cw + kCodes;
#pragma unroll
        for (int j = 0; j < NIT; ++j) {
          const int it = warp + kProdWarps * j, mat = it / 8, rt = it % 8;
          const uint4 wv = *reinterpret_cast<const uint4*>(cw + (it * 32 + lane) * 16);
          const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
          float sc[4];  // rows g, g+8 of halves 0 and 1
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            sc[2 * h] = scale_at(sw + (it * 2 + h) * 64, g, a.sdt);
            sc[2 * h + 1] = scale_at(sw + (it * 2 + h) * 64, g + 8, a.sdt);
          }
          uint8_t* r0 = st + mat * kATile + (rt * 16 + g) * 128;
          uint8_t* r1 = r0 + 8 * 128;
          uint32_t s2[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) s2[h] = pack_bf16x2(sc[h], sc[h]);
          if (bfs) {  // (128 + u) - zb is exact in bf16; one rounding for the product
#pragma unroll
            for (int i = 0; i < 16; ++i) {  // pair i: k-step i/4 of the stage, register i%4
              const uint32_t v = chunk_pair<B>(w, i);
              const int kk = i >> 2, r = i & 3;
              uint32_t t, out;
              asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(t) : "r"(v), "r"(0x3F803F80u), "r"(negzb2));
              asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out) : "r"(t), "r"(s2[(kk >= 2 ? 2 : 0) + (r & 1)]));
              *reinterpret_cast<uint32_t*>(((r & 1) ? r1 : r0) + offc[2 * kk + (r >> 1)]) = out;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t v = chunk_pair<B>(w, i);
              const int kk = i >> 2, r = i & 3;
              const float sv = sc[(kk >= 2 ? 2 : 0) + (r & 1)];
              const uint32_t out = pack_bf16x2((bf16f(v & 0xffffu) - zb) * sv, (__uint_as_float(v & 0xffff0000u) - zb) * sv);
              *reinterpret_cast<uint32_t*>(((r & 1) ? r1 : r0) + offc[2 * kk + (r >> 1)]) = out;
            }
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
        mbar_arrive(smem_addr(&fullb[slot]));
        // two stages ahead, into the slot the tensor core frees while this
        // stage's successor is dequantised
        if (s + 2 < S) fetch(s + 2);
      }
      gs += S;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      int gs = 0, ui = 0;
      for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++ui) {
        int e, mt, n0, nrows;
        decode_unit(u, e, mt, n0, nrows);
        const int N = (nrows + 15) & ~15;
        const uint32_t idesc = idesc_bf16(kTileM, N);
        const int buf = ui % NBUF, use = ui / NBUF;
        if (use > 0) mbar_wait(smem_addr(&tempty[buf]), (uint32_t)(use - 1) & 1u, a.err);  // accumulator free
        tc_fence_after();
        const uint32_t dacc = tmem + (uint32_t)(buf * 256);
        for (int s = 0; s < S; ++s, ++gs) {
          const int slot = gs % NS, su = gs / NS;
          mbar_wait(smem_addr(&fullb[slot]), (uint32_t)su & 1u, a.err);
          tc_fence_after();
          const uint32_t st = smem_addr(smem + (size_t)slot * kStage);
          const uint32_t bt = st + NMAT * kATile;
#pragma unroll
          for (int j = 0; j < kStageK / 16; ++j) {
#pragma unroll
            for (int mat = 0; mat < NMAT; ++mat)
              umma_bf16(dacc + mat * 256, smem_desc_sw128(st + mat * kATile + j * 32),
                        smem_desc_sw128(bt + j * 32), idesc, (s | j) ? 1u : 0u);
          }
          umma_commit(smem_addr(&emptyb[slot]));  // the stage is free once these MMAs are done
        }
        umma_commit(smem_addr(&tfull[buf]));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 4-7)
    const int quad = warp & 3;
    const int et = tid - kEpiWarp0 * 32;  // 0..127
    const int row = quad * 32 + lane;  // weight row within the unit = TMEM lane
    int ui = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++ui) {
      int e, mt, n0, nrows;
      decode_unit(u, e, mt, n0, nrows);
      const int buf = ui % NBUF, use = ui / NBUF;
      if constexpr (!GATEUP) {  // the unit's routing weights, staged while its MMAs run
        for (int c = et; c < nrows; c += 128) wslot[ui & 1][c] = a.topk_w[a.perm[n0 + c]];
        asm volatile("bar.sync 3, 128;" ::: "memory");
      }
      mbar_wait(smem_addr(&tfull[buf]), (uint32_t)use & 1u, a.err);
      tc_fence_after();
      const uint32_t ta = tmem + (uint32_t)(buf * 256) + ((uint32_t)(quad * 32) << 16);
      const int64_t ocol = (int64_t)mt * kTileM + row;
      for (int c0 = 0; c0 < nrows; c0 += 16) {
        float v0[16];
        tmem_ld16(ta + c0, v0);
        if constexpr (GATEUP) {
          float v1[16];
          tmem_ld16(ta + 256 + c0, v1);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if (c0 + c < nrows) {
              const float gv = v0[c], uv = v1[c];
              const float h = gv / (1.0f + expf(-gv)) * uv;
              a.hout[(int64_t)(n0 + c0 + c) * a.out_ld + ocol] = __bfloat16_as_ushort(__float2bfloat16_rn(h));
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if (c0 + c < nrows) {
              const float w = wslot[ui & 1][c0 + c];
              a.oout[(int64_t)(n0 + c0 + c) * a.out_ld + ocol] = __bfloat16_as_ushort(__float2bfloat16_rn(w * v0[c]));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_addr(&tempty[buf]));
    }
  }
  // teardown: the MMA warp frees TMEM once the last accumulator was read
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(512));
  }
}

// y[t][c] = sum over j ascending of o[inv[t*k + j]][c] (bf16 slot outputs, fp32 sum)
__global__ void pf_combine_kernel(const uint16_t* __restrict__ o, const int32_t* __restrict__ inv, int T,
                                  int H, int k, uint16_t* __restrict__ y) {
  const int64_t n = (int64_t)T * (H / 2);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / (H / 2)), c = (int)(i % (H / 2)) * 2;
    float s0 = 0.f, s1 = 0.f;
    for (int j = 0; j < k; ++j) {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(o + (int64_t)inv[(int64_t)t * k + j] * H + c);
      s0 += bf16f(v & 0xffffu);
      s1 += bf16f(v >> 16);
    }
    *reinterpret_cast<uint32_t*>(y + (int64_t)t * H + c) =
        (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s0)) |
        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s1)) << 16);
  }
}

// Per-forward accounting (one CTA): every expert with routed tokens is one
// access; a hit iff it is read from HBM; bytes by residence; cache counters
// (count += 1, last = step) and the miss queue as in the decode kernel.
__global__ void pf_stats_kernel(const int32_t* __restrict__ counts, int E, const uint8_t* const* blob_hbm,
                                unsigned long long* stats, int64_t expert_bytes, int64_t router_bytes,
                                int n_pairs, int lfu, int64_t ge0, uint32_t* lfu_count, int32_t* lfu_last,
                                const int* step, int32_t* miss_list, unsigned* miss_count, int miss_cap) {
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
  }
}

template <bool GATEUP>
cudaError_t launch_gemm(int bits, const GemmArgs& a, int grid, size_t smem, cudaStream_t s) {
  const void* fn = bits == 2   ? (const void*)pf_gemm_kernel<2, GATEUP>
                   : bits == 3 ? (const void*)pf_gemm_kernel<3, GATEUP>
                               : (const void*)pf_gemm_kernel<4, GATEUP>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  switch (bits) {
    case 2: pf_gemm_kernel<2, GATEUP><<<grid, kGemmThreads, smem, s>>>(a); break;
    case 3: pf_gemm_kernel<3, GATEUP><<<grid, kGemmThreads, smem, s>>>(a); break;
    default: pf_gemm_kernel<4, GATEUP><<<grid, kGemmThreads, smem, s>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t moe::prefill_forward(Plan& p, int layer, const uint16_t* x, int T, uint16_t* y,
                                 cudaStream_t s, const moe_routing_out* dbg) {
  const moe_plan_desc& d = p.d;
  const int E = d.num_experts, H = d.hidden, I = d.inter, k = d.top_k;
  const int n = T * k;
  cudaError_t e;
  {
    const dim3 grid((T + kRtTile - 1) / kRtTile, (E + kRtTile - 1) / kRtTile);
    pf_router_kernel<<<grid, 256, 0, s>>>(x, T, H, p.wr[layer], p.bias[layer], E, p.logits);
  }
  pf_topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(p.logits, T, E, k, p.topk_idx, p.topk_w);
  pf_count_kernel<<<E, 1024, 0, s>>>(p.topk_idx, n, p.counts);
  pf_scan_kernel<<<1, 32, 0, s>>>(p.counts, E, p.offsets);
  pf_place_kernel<<<E, 1024, 0, s>>>(p.topk_idx, n, p.offsets, p.perm, p.inv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const int64_t ge0 = (int64_t)layer * E;
  GemmArgs g{};
  g.E = E;
  g.k = k;
  g.bits = d.weight_bits;
  g.group = d.group_size;
  g.sdt = d.scale_dtype;
  g.blob_hbm = p.blob_hbm + ge0;
  g.blob_host = p.blob_host + ge0;
  g.offsets = p.offsets;
  g.perm = p.perm;
  g.topk_w = p.topk_w;
  g.err = p.err_dev;
  int optin = 0;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d.device)) != cudaSuccess)
    return e;
  const size_t static_guess = 8 * 1024;  // barriers, row sources, routing weights
  // gate / up -> h
  {
    GemmArgs a = g;
    a.K = H;
    a.kpad = p.lay.m[0].kpad;
    a.rows = I;
    a.codes[0] = p.lay.m[0].codes_off;
    a.scales[0] = p.lay.m[0].scales_off;
    a.codes[1] = p.lay.m[1].codes_off;
    a.scales[1] = p.lay.m[1].scales_off;
    a.x = x;
    a.hout = p.pf_h;
    a.out_ld = I;
    const size_t stage = 2 * kTileM * 128 + kTileN * 128 + 2 * 8 * 32 * 16 + 2 * 8 * 2 * 64;
    const size_t table = ((size_t)(E + 1) * 4 + 15) / 16 * 16;
    a.nstages = (int)std::min<size_t>(4, ((size_t)optin - static_guess - 1024 - table) / stage);
    if (a.nstages < 3) return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)a.nstages * stage + 1024 + table;
    if ((e = launch_gemm<true>(d.weight_bits, a, p.sms, smem, s)) != cudaSuccess) return e;
  }
  // down -> weighted o per slot
  {
    GemmArgs a = g;
    a.K = I;
    a.kpad = p.lay.m[2].kpad;
    a.rows = H;
    a.codes[0] = p.lay.m[2].codes_off;
    a.scales[0] = p.lay.m[2].scales_off;
    a.hin = p.pf_h;
    a.oout = p.pf_o;
    a.out_ld = H;
    const size_t stage = kTileM * 128 + kTileN * 128 + 8 * 32 * 16 + 8 * 2 * 64;
    const size_t table = ((size_t)(E + 1) * 4 + 15) / 16 * 16;
    a.nstages = (int)std::min<size_t>(4, ((size_t)optin - static_guess - 1024 - table) / stage);
    if (a.nstages < 3) return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)a.nstages * stage + 1024 + table;
    if ((e = launch_gemm<false>(d.weight_bits, a, p.sms, smem, s)) != cudaSuccess) return e;
  }
  pf_combine_kernel<<<4 * p.sms, 256, 0, s>>>(p.pf_o, p.inv, T, H, k, y);
  pf_stats_kernel<<<1, 512, 0, s>>>(p.counts, E, p.blob_hbm + ge0, p.stats + (int64_t)layer * kNumStats,
                                    p.lay.algo_bytes, (int64_t)E * H * 2, n,
                                    d.cache_policy == MOE_POLICY_LFU, ge0, p.lfu_count, p.lfu_last,
                                    &p.ctl->step, p.miss_list, p.miss_count, d.num_layers * p.max_distinct);
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
