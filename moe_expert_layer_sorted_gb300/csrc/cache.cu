// Frequency-admitted HBM expert cache ("Running a 24k-expert MoE on a single
// 32 GB card", sections 2-3: the hot experts live in a VRAM cache filled by
// access frequency, the rest are read in place from pinned host memory).
//
// Every expert's master copy is in pinned host memory; a global pool of C
// HBM slots holds the cached ones.  The forward kernel counts accesses
// (count += 1, last = step for every distinct routed (layer, expert)) and
// queues the misses.  At step end:
//   1. lfu_decide_kernel (one CTA) takes the step's misses in ascending global
//      id = (layer, expert) order.  An expert already admitted this step is
//      skipped.  A free slot (the lowest one) admits it; otherwise the victim
//      is the resident expert not accessed this step with the smallest
//      (count, last, id), and the miss is admitted iff its count exceeds the
//      victim's (ties keep the incumbent).  Tables (slot_of, owner, the
//      forward's residence pointers) and per-layer statistics are updated in
//      place; optional count halving every aging_period steps.
//   2. lfu_fill_kernel copies each admitted expert from its pinned host copy
//      into its slot.  Both run on the caller's stream before the next
//      step's forwards, so an admission takes effect from the next step.
#include "internal.h"

using namespace moe;

namespace {

constexpr int kDecideThreads = 1024;

struct StepEndArgs {
  int E;
  int64_t LE, C;
  int* step;  // device step counter: this step's number, advanced at the end
  int aging_period;
  uint32_t* count;
  int32_t* last;
  int32_t* slot_of;
  int32_t* owner;
  const int32_t* miss_list;
  unsigned* miss_count;
  int miss_cap;
  unsigned* adm;  // [0] admissions this step, [1] slots handed out so far (free = [used, C))
  unsigned* adm_list;  // (global id, slot) pairs of this step's admissions
  const uint8_t** blob_hbm;
  uint8_t* arena;
  int64_t blob_bytes, expert_bytes;
  unsigned long long* stats;  // [L][kNumStats]
};

// eviction order: smaller count, then older last access, then smaller id
struct Cand {
  uint32_t count;
  int32_t last;
  int32_t id;  // -1: none
};
__device__ __forceinline__ bool before(const Cand& x, const Cand& y) {
  if (x.id < 0) return false;
  if (y.id < 0) return true;
  if (x.count != y.count) return x.count < y.count;
  if (x.last != y.last) return x.last < y.last;
  return x.id < y.id;
}

__global__ void __launch_bounds__(kDecideThreads) lfu_decide_kernel(StepEndArgs a) {
  extern __shared__ int32_t mq[];  // [miss_cap] the step's misses, sorted
  __shared__ Cand wbest[kDecideThreads / 32];
  __shared__ Cand victim;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nm = (int)min((unsigned)a.miss_cap, *a.miss_count);
  const int step = *a.step;
  // the step's misses in ascending global id (stable among repeats: the key
  // is (id, queue position))
  for (int i = tid; i < nm; i += blockDim.x) {
    const int32_t g = a.miss_list[i];
    int r = 0;
    for (int j = 0; j < nm; ++j) {
      const int32_t h = a.miss_list[j];
      r += (h < g) || (h == g && j < i);
    }
    mq[r] = g;
  }
  if (tid == 0) a.adm[0] = 0u;
  __syncthreads();
  unsigned nadm = 0;
  for (int q = 0; q < nm; ++q) {
    const int32_t g = mq[q];
    if (a.slot_of[g] >= 0) {  // already admitted (repeated access this step)
      __syncthreads();
      continue;
    }
    const unsigned used = a.adm[1];
    int32_t slot = -1, v = -1;
    if ((int64_t)used < a.C) {
      slot = (int32_t)used;
    } else {
      // block argmin over the resident experts not accessed this step
      Cand best{0u, 0, -1};
      for (int64_t c = tid; c < a.C; c += blockDim.x) {
        const int32_t o = a.owner[c];
        if (o < 0) continue;
        const int32_t lo = a.last[o];
        if (lo == step) continue;
        const Cand x{a.count[o], lo, o};
        if (before(x, best)) best = x;
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        Cand y;
        y.count = __shfl_xor_sync(0xffffffffu, best.count, off);
        y.last = __shfl_xor_sync(0xffffffffu, best.last, off);
        y.id = __shfl_xor_sync(0xffffffffu, best.id, off);
        if (before(y, best)) best = y;
      }
      if (lane == 0) wbest[warp] = best;
      __syncthreads();
      if (tid == 0) {
        Cand b = wbest[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
          if (before(wbest[w], b)) b = wbest[w];
        victim = b;
      }
      __syncthreads();
      if (victim.id >= 0 && a.count[g] > victim.count) {
        v = victim.id;
        slot = a.slot_of[v];
      }
    }
    if (tid == 0 && slot >= 0) {
      if (v >= 0) {
        a.slot_of[v] = -1;
        a.blob_hbm[v] = nullptr;
      } else {
        a.adm[1] = used + 1u;
      }
      a.owner[slot] = g;
      a.slot_of[g] = slot;
      a.blob_hbm[g] = a.arena + (int64_t)slot * a.blob_bytes;
      a.adm_list[2 * nadm] = (unsigned)g;
      a.adm_list[2 * nadm + 1] = (unsigned)slot;
      unsigned long long* st = a.stats + (int64_t)(g / a.E) * kNumStats;
      st[kStatAdmissions] += 1ull;
      st[kStatFillBytes] += (unsigned long long)a.expert_bytes;
      if (v >= 0) st[kStatEvictions] += 1ull;
    }
    if (slot >= 0) ++nadm;
    __syncthreads();  // tables settled before the next miss
  }
  if (a.aging_period > 0 && (step + 1) % a.aging_period == 0)
    for (int64_t i = tid; i < a.LE; i += blockDim.x) a.count[i] >>= 1;
  if (tid == 0) {
    a.adm[0] = nadm;
    *a.miss_count = 0u;
    *a.step = step + 1;
  }
}

// Admitted experts: pinned host copy -> HBM slot, 16 bytes per thread per step.
__global__ void lfu_fill_kernel(const unsigned* __restrict__ adm, const unsigned* __restrict__ adm_list,
                                const uint8_t* const* __restrict__ blob_host, uint8_t* arena,
                                int64_t blob_bytes) {
  const int64_t n = adm[0];
  const int64_t per = blob_bytes / 16;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n * per;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = i / per, c = i % per;
    const unsigned g = adm_list[2 * j], slot = adm_list[2 * j + 1];
    const uint4 v = reinterpret_cast<const uint4*>(blob_host[g])[c];
    reinterpret_cast<uint4*>(arena + (int64_t)slot * blob_bytes)[c] = v;
  }
}

// The chunked prefill's residence of one layer ("Running a 24k-expert MoE on a
// single 32 GB card", section 2: slots kept for a prompt's experts): an expert
// with an HBM copy keeps it; the others, in ascending expert order, take the
// prefill slots while they last (the rest stay host-only).  stage[0] = number
// staged; stage[2 + 2i], stage[3 + 2i] = (global id, slot) of the i-th, for
// the fill kernel.  The staged bytes count as fill bytes of the layer.
__global__ void __launch_bounds__(1024) pf_stage_kernel(const uint8_t* const* __restrict__ blob_hbm, int E,
                                                        int64_t ge0, int64_t nslots, uint8_t* arena,
                                                        int64_t blob_bytes, const uint8_t** pf_blob,
                                                        unsigned* stage, unsigned long long* stats,
                                                        int64_t expert_bytes) {
  __shared__ unsigned wsum[32];
  __shared__ unsigned carry_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  if (tid == 0) carry_s = 0u;
  __syncthreads();
  for (int base = 0; base < E; base += blockDim.x) {
    const int e = base + tid;
    const uint8_t* hb = e < E ? blob_hbm[e] : nullptr;
    const bool flag = e < E && hb == nullptr;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    if (lane == 0) wsum[warp] = __popc(bal);
    __syncthreads();
    unsigned before = carry_s;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    const unsigned rank = before + __popc(bal & ((1u << lane) - 1u));
    if (e < E) {
      if (!flag) {
        pf_blob[e] = hb;
      } else if ((int64_t)rank < nslots) {
        pf_blob[e] = arena + (int64_t)rank * blob_bytes;
        stage[2 + 2 * rank] = (unsigned)(ge0 + e);
        stage[3 + 2 * rank] = rank;
      } else {
        pf_blob[e] = nullptr;
      }
    }
    __syncthreads();
    if (tid == 0) {
      unsigned tot = 0;
      for (int w = 0; w < nw; ++w) tot += wsum[w];
      carry_s += tot;
    }
    __syncthreads();
  }
  if (tid == 0) {
    const unsigned n = (unsigned)min((int64_t)carry_s, nslots);
    stage[0] = n;
    stats[kStatFillBytes] += (unsigned long long)n * (unsigned long long)expert_bytes;
  }
}

}  // namespace

cudaError_t moe::prefill_stage(Plan& p, int layer, cudaStream_t s) {
  const int E = p.d.num_experts;
  const int64_t ge0 = (int64_t)layer * E;
  pf_stage_kernel<<<1, 1024, 0, s>>>(p.blob_hbm + ge0, E, ge0, p.d.prefill_slots, p.pf_arena, p.lay.blob_bytes,
                                     p.pf_blob, p.pf_stage, p.stats + (int64_t)layer * kNumStats,
                                     p.lay.algo_bytes);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.d.prefill_slots == 0) return e;
  lfu_fill_kernel<<<2 * p.sms, 512, 0, s>>>(p.pf_stage, p.pf_stage + 2, p.blob_host, p.pf_arena, p.lay.blob_bytes);
  return cudaGetLastError();
}

cudaError_t moe::lfu_step_end(Plan& p, cudaStream_t s) {
  const moe_plan_desc& d = p.d;
  StepEndArgs a{};
  a.E = d.num_experts;
  a.LE = (int64_t)d.num_layers * d.num_experts;
  a.C = d.cache_slots;
  a.step = &p.ctl->step;
  a.aging_period = d.aging_period;
  a.count = p.lfu_count;
  a.last = p.lfu_last;
  a.slot_of = p.slot_of;
  a.owner = p.slot_owner;
  a.miss_list = p.miss_list;
  a.miss_count = p.miss_count;
  a.miss_cap = d.num_layers * p.max_distinct;
  a.adm = p.adm_count;
  a.adm_list = p.adm_list;
  a.blob_hbm = p.blob_hbm;
  a.arena = p.hbm_arena;
  a.blob_bytes = p.lay.blob_bytes;
  a.expert_bytes = p.lay.algo_bytes;
  a.stats = p.stats;
  const size_t smem = (size_t)a.miss_cap * 4;
  cudaError_t e = cudaSuccess;
  if (smem > 48 * 1024 && (e = ensure_dynamic_smem((const void*)lfu_decide_kernel, smem)) != cudaSuccess)
    return e;
  lfu_decide_kernel<<<1, kDecideThreads, smem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.C > 0) {
    lfu_fill_kernel<<<2 * p.sms, 512, 0, s>>>(p.adm_count, p.adm_list, p.blob_host, p.hbm_arena,
                                               p.lay.blob_bytes);
    e = cudaGetLastError();
  }
  return e;
}
