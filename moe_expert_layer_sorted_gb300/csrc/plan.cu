// Plan lifetime, placement of experts (canonical format -> device layout in
// HBM or pinned host memory), router upload, statistics, the quantiser and
// the link probe.  The forward passes live in decode.cu / prefill.cu and the
// cache policy in cache.cu.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <sys/syscall.h>
#include <unistd.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <new>

#include "internal.h"

using namespace moe;

namespace {

thread_local std::string g_last_error_noplan;

moe_status fail(Plan* p, moe_status s, const std::string& msg) {
  if (p) p->last_error = msg;
  else g_last_error_noplan = msg;
  return s;
}

moe_status cuda_fail(Plan* p, cudaError_t e, const char* what) {
  std::string m = std::string(what) + ": " + cudaGetErrorString(e);
  if (e == cudaErrorMemoryAllocation) return fail(p, MOE_ERR_OOM, m);
  return fail(p, MOE_ERR_CUDA, m);
}

// A forward's launch failure; a failed cuBLAS call (the prefill router's
// logits GEMM) is reported with its own status.
moe_status forward_fail(Plan* p, cudaError_t e, const char* what) {
  if (p && p->blas_status) {
    const int bs = p->blas_status;
    p->blas_status = 0;
    return fail(p, MOE_ERR_CUDA, std::string(what) + ": the router logits GEMM (cuBLAS) failed with status " +
                                     std::to_string(bs));
  }
  return cuda_fail(p, e, what);
}

#define CK(p, call)                                          \
  do {                                                       \
    cudaError_t e_ = (call);                                 \
    if (e_ != cudaSuccess) return cuda_fail((p), e_, #call); \
  } while (0)

// Makes `dev` current for the scope of a call and restores the caller's device.
struct DeviceScope {
  int prev = -1;
  bool ok = true;
  explicit DeviceScope(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceScope() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// One call at a time per plan.
struct Busy {
  Plan* p;
  bool ok;
  explicit Busy(Plan* pl) : p(pl), ok(pl->busy.exchange(1) == 0) {}
  ~Busy() {
    if (ok) p->busy.store(0);
  }
};

// Word 1 of the mapped error page: set by a forward whose step's miss queue
// was already full (its miss is not queued for the step-end admission pass).
// Taken (read and cleared) by the next call that looks.
constexpr const char* kOverflowMsg =
    "an earlier forward found this step's miss queue full (a layer forwarded more than once "
    "between step ends?); its misses were not queued for admission";
bool take_overflow(Plan* p) {
  if (!p->err_host || !p->err_host[1]) return false;
  p->err_host[1] = 0;
  return true;
}

// Host-side fault injection for the failure paths (tests): MOE_FAULT holds a
// comma-separated list; "hbm_alloc" makes the plan's HBM arena allocation
// fail, "pinned_alloc" its pinned host arena allocation.  Both then take the
// same path as a real failure: everything allocated so far is released and
// moe_plan_create returns MOE_ERR_OOM.  No device work is involved.
bool fault_injected(const char* what) {
  const char* f = getenv("MOE_FAULT");
  return f && strstr(f, what) != nullptr;
}

// NUMA node of the plan's GPU (sysfs of its PCI function), or -1.
int gpu_numa_node(int device) {
  char bus[32] = {0};
  if (cudaDeviceGetPCIBusId(bus, sizeof bus, device) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  for (char* c = bus; *c; ++c)
    if (*c >= 'A' && *c <= 'F') *c = (char)(*c - 'A' + 'a');
  char path[128];
  snprintf(path, sizeof path, "/sys/bus/pci/devices/%s/numa_node", bus);
  FILE* f = fopen(path, "r");
  if (!f) return -1;
  int node = -1;
  if (fscanf(f, "%d", &node) != 1) node = -1;
  fclose(f);
  return node;
}

// Pinned, device-mapped host memory of `bytes` from the driver's pinned
// allocator (cudaHostAlloc).  When node >= 0 the calling thread prefers that
// NUMA node for the call (set_mempolicy MPOL_PREFERRED, the thread's own policy
// restored after), so the pages come from the GPU's node where the system places them
// by the caller's policy.  The driver's allocator is used rather than
// page-locking an anonymous mapping: on a host whose memory earlier large
// pinned arenas had churned, the GPU read such a registered mapping several
// times slower (a decode step of the decode layer 0.55-0.72 ms against 0.26 ms
// from cudaHostAlloc; on a fresh host both 0.20 ms).
void* pinned_alloc(size_t bytes, int node) {
  // the calling thread's own policy, restored after the call
  int old_mode = 0;
  unsigned long old_mask[16] = {0};  // up to 1024 nodes
  bool preferred = false;
  if (node >= 0 && node < 64 && syscall(SYS_get_mempolicy, &old_mode, old_mask, 1024ul, nullptr, 0ul) == 0) {
    unsigned long mask = 1ul << node;
    preferred = syscall(SYS_set_mempolicy, 1 /* MPOL_PREFERRED */, &mask, 64ul) == 0;
  }
  void* h = nullptr;
  const cudaError_t e = cudaHostAlloc(&h, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (preferred) {
    const bool dflt = (old_mode & 0xff) == 0;  // MPOL_DEFAULT (mode flags in the high bits)
    syscall(SYS_set_mempolicy, old_mode, dflt ? nullptr : old_mask, dflt ? 0ul : 1024ul);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return h;
}

void pinned_free(void* p) {
  if (p) cudaFreeHost(p);
}

bool is_device_ptr(const void* ptr) {
  if (!ptr) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

int64_t align256(int64_t v) { return (v + 255) & ~int64_t(255); }

// ------------------------------------------------------------- kernels

// Code of W[row][k] from the canonical little-endian bit stream (b <= 8 bits).
__device__ __forceinline__ uint32_t canon_code(const uint8_t* __restrict__ src, int64_t idx,
                                               int bits) {
  const int64_t bit = idx * bits;
  uint32_t v = (uint32_t)src[bit >> 3];
  if ((bit & 7) + bits > 8) v |= (uint32_t)src[(bit >> 3) + 1] << 8;  // never reads past the code
  return (v >> (bit & 7)) & ((1u << bits) - 1u);
}

// One thread per (row tile, column block, lane): gathers the 128 codes of the
// lane's A-fragment elements and writes its 4*b words (layout in internal.h).
// Pair P = 4*kt + r of the block holds (row, k) and (row, k + 1) with
// kt = 16-column step, r = fragment register: row = 16 mt + l/4 + 8 (r & 1),
// k = 256 kb + 16 kt + 2 (l % 4) + 8 (r >> 1).  Field placement per b:
//   b = 4: word P/4, field j = P%4 at bits [4j, 4j+4) (low code) and [16+4j, ...) (high)
//   b = 2: word P/8, field j = P%8 at bits [2j, 2j+2) and [16+2j, ...)
//   b = 3: words in triples 3t..3t+2 per 16 pairs (t = P/16, m = P%16); m < 15:
//          word 3t + m/5, field j = m%5 at bits [3j, 3j+3) and [16+3j, ...);
//          m = 15: bit i of the low / high code in bit 15 / 31 of word 3t + i.
// Columns k >= K (padding) get the zero point 2^(b-1).
__global__ void repack_codes_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                    int rows, int K, int kpad, int bits) {
  const int nkb = kpad / kBlockK;
  const int64_t n = (int64_t)rows / kTileRows * nkb * 32;
  const uint32_t zp = 1u << (bits - 1);
  for (int64_t p = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; p < n;
       p += (int64_t)gridDim.x * blockDim.x) {
    const int lane = (int)(p % 32);
    const int64_t r = p / 32;
    const int kb = (int)(r % nkb);
    const int64_t mt = r / nkb;
    const int g = lane >> 2, tig = lane & 3;
    uint32_t w[16];
    for (int q = 0; q < 16; ++q) w[q] = 0u;
    for (int P = 0; P < 64; ++P) {
      const int kt = P >> 2, reg = P & 3;
      const int64_t row = mt * kTileRows + g + 8 * (reg & 1);
      const int k = kb * kBlockK + kt * 16 + 2 * tig + 8 * (reg >> 1);
      const uint32_t lo = k < K ? canon_code(src, row * K + k, bits) : zp;
      const uint32_t hi = k + 1 < K ? canon_code(src, row * K + k + 1, bits) : zp;
      if (bits == 4) {
        const int j = P & 3;
        w[P >> 2] |= (lo << (4 * j)) | (hi << (16 + 4 * j));
      } else if (bits == 2) {
        const int j = P & 7;
        w[P >> 3] |= (lo << (2 * j)) | (hi << (16 + 2 * j));
      } else {
        const int t = P >> 4, m = P & 15;
        if (m < 15) {
          const int j = m % 5;
          w[3 * t + m / 5] |= (lo << (3 * j)) | (hi << (16 + 3 * j));
        } else {
          for (int i = 0; i < 3; ++i)
            w[3 * t + i] |= (((lo >> i) & 1u) << 15) | (((hi >> i) & 1u) << 31);
        }
      }
    }
    for (int q = 0; q < 4 * bits; ++q)
      *reinterpret_cast<uint32_t*>(dst + ((r * bits + q / 4) * 512) + lane * 16 + (q % 4) * 4) = w[q];
  }
}

__global__ void repack_scales_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                     int rows, int ng, int ngpad, int esize) {
  const int64_t n = (int64_t)rows * ngpad;
  for (int64_t p = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; p < n;
       p += (int64_t)gridDim.x * blockDim.x) {
    const int rr = (int)(p % kTileRows);
    const int64_t q = p / kTileRows;
    const int g = (int)(q % ngpad);
    const int64_t mt = q / ngpad;
    const int64_t row = mt * kTileRows + rr;
    uint8_t* d = dst + p * esize;
    if (g >= ng) {
      if (esize == 4) *reinterpret_cast<uint32_t*>(d) = 0u;
      else *reinterpret_cast<uint16_t*>(d) = 0;
      continue;
    }
    const uint8_t* s = src + (row * ng + g) * esize;
    if (esize == 4) *reinterpret_cast<uint32_t*>(d) = *reinterpret_cast<const uint32_t*>(s);
    else *reinterpret_cast<uint16_t*>(d) = *reinterpret_cast<const uint16_t*>(s);
  }
}

// Symmetric int-b group quantiser: one warp per (row, group); group % 32 == 0.
__global__ void quantize_kernel(const float* __restrict__ w, int rows, int cols, int bits,
                                int group, int sdt, uint32_t* __restrict__ codes,
                                uint8_t* __restrict__ scales) {
  extern __shared__ uint32_t qs_words[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int nw = group * bits / 32;
  uint32_t* sw = qs_words + wib * nw;
  const int ng = cols / group;
  const int64_t ngroups = (int64_t)rows * ng;
  const int qmax = (1 << (bits - 1)) - 1;
  const int off = 1 << (bits - 1);
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t gi = blockIdx.x * (int64_t)(blockDim.x >> 5) + wib; gi < ngroups; gi += warps) {
    const int64_t r = gi / ng;
    const int g = (int)(gi % ng);
    const float* src = w + r * cols + (int64_t)g * group;
    float amax = 0.0f;
    for (int j = lane; j < group; j += 32) amax = fmaxf(amax, fabsf(src[j]));
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    float s = __fdiv_rn(amax, (float)qmax);
    if (sdt == MOE_SCALE_BF16) s = __bfloat162float(__float2bfloat16_rn(s));
    else if (sdt == MOE_SCALE_F16) s = __half2float(__float2half_rn(s));
    for (int j = lane; j < nw; j += 32) sw[j] = 0u;
    __syncwarp();
    for (int j = lane; j < group; j += 32) {
      int q = 0;
      if (s != 0.0f) {
        float v = rintf(__fdiv_rn(src[j], s));
        v = fminf(fmaxf(v, (float)-qmax), (float)qmax);
        q = (int)v;
      }
      const uint32_t u = (uint32_t)(q + off);
      const int bit = j * bits;
      atomicOr(&sw[bit >> 5], u << (bit & 31));
      if ((bit & 31) + bits > 32) atomicOr(&sw[(bit >> 5) + 1], u >> (32 - (bit & 31)));
    }
    __syncwarp();
    const int64_t word0 = (r * cols + (int64_t)g * group) * bits / 32;
    for (int j = lane; j < nw; j += 32) codes[word0 + j] = sw[j];
    if (lane == 0) {
      if (sdt == MOE_SCALE_F32) reinterpret_cast<float*>(scales)[gi] = s;
      else if (sdt == MOE_SCALE_BF16)
        reinterpret_cast<__nv_bfloat16*>(scales)[gi] = __float2bfloat16_rn(s);
      else reinterpret_cast<__half*>(scales)[gi] = __float2half_rn(s);
    }
    __syncwarp();
  }
}

// dst[i] = src[i] for n16 16-byte words, one per thread (src: the device
// mapping of a page-locked host buffer)
__global__ void copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int n16) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n16) dst[i] = src[i];
}

// Streaming read of n16 16-byte words; the XOR of everything goes to *sink so
// the loads cannot be removed.
__global__ void read_probe_kernel(const uint4* __restrict__ p, int64_t n16, unsigned* sink) {
  uint32_t acc = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p + i));
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9e3779b9u) atomicAdd(sink, 1u);
}

}  // namespace

cudaError_t moe::ensure_dynamic_smem(const void* fn, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> set;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  size_t& cur = set[{dev, fn}];
  if (bytes <= cur) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

// --------------------------------------------------------------- layout

ExpertLayout moe::make_layout(int H, int I, int bits, int group, int sdt) {
  ExpertLayout L{};
  int64_t off = 0;
  const int rows[3] = {I, I, H}, cols[3] = {H, H, I};
  for (int m = 0; m < 3; ++m) {
    L.m[m].rows = rows[m];
    L.m[m].cols = cols[m];
    L.m[m].kpad = (cols[m] + kBlockK - 1) / kBlockK * kBlockK;
    L.m[m].codes_bytes = (int64_t)rows[m] * L.m[m].kpad * bits / 8;
    L.m[m].codes_off = off;
    off = align256(off + L.m[m].codes_bytes);
  }
  for (int m = 0; m < 3; ++m) {
    L.m[m].scales_bytes = (int64_t)rows[m] * (L.m[m].kpad / group) * scale_size(sdt);
    L.m[m].scales_off = off;
    off = align256(off + L.m[m].scales_bytes);
  }
  L.blob_bytes = off;
  L.algo_bytes = 0;
  for (int m = 0; m < 3; ++m)
    L.algo_bytes += (int64_t)rows[m] * cols[m] * bits / 8 +
                    (int64_t)rows[m] * (cols[m] / group) * scale_size(sdt);
  return L;
}

// src_codes / src_scales: the canonical (unpadded) matrix; the device copy is
// written into dst_blob at the matrix's offsets.
cudaError_t moe::launch_repack(const uint8_t* src_codes, const void* src_scales, uint8_t* dst_blob,
                               const MatLayout& m, int bits, int group, int sdt, cudaStream_t s) {
  const int64_t threads = (int64_t)m.rows / kTileRows * (m.kpad / kBlockK) * 32;
  int blocks = (int)std::min<int64_t>((threads + 127) / 128, 8192);
  repack_codes_kernel<<<blocks, 128, 0, s>>>(src_codes, dst_blob + m.codes_off, m.rows, m.cols,
                                              m.kpad, bits);
  const int ng = m.cols / group, ngpad = m.kpad / group;
  const int64_t ns = (int64_t)m.rows * ngpad;
  blocks = (int)std::min<int64_t>((ns + 255) / 256, 4096);
  repack_scales_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint8_t*>(src_scales),
                                               dst_blob + m.scales_off, m.rows, ng, ngpad,
                                               scale_size(sdt));
  return cudaGetLastError();
}

cudaError_t moe::launch_quantize(const float* w, int rows, int cols, int bits, int group, int sdt,
                                 uint8_t* codes, void* scales, cudaStream_t s) {
  const int64_t ngroups = (int64_t)rows * (cols / group);
  const int wpb = 8;
  const int blocks = (int)std::min<int64_t>((ngroups + wpb - 1) / wpb, 8192);
  const size_t smem = (size_t)wpb * (group * bits / 32) * sizeof(uint32_t);
  quantize_kernel<<<blocks, wpb * 32, smem, s>>>(w, rows, cols, bits, group, sdt,
                                                 reinterpret_cast<uint32_t*>(codes),
                                                 static_cast<uint8_t*>(scales));
  return cudaGetLastError();
}

// ------------------------------------------------------------------ ABI

namespace {

moe_status validate(const moe_plan_desc* d, std::string& why) {
  if (!d) { why = "desc is NULL"; return MOE_ERR_INVALID; }
  if (d->struct_size != sizeof(moe_plan_desc)) {
    why = "struct_size != sizeof(moe_plan_desc)";
    return MOE_ERR_INVALID;
  }
  for (int i = 0; i < 3; ++i)
    if (d->reserved[i]) { why = "reserved fields must be zero"; return MOE_ERR_INVALID; }
  if (d->prefill_slots < 0 || d->prefill_slots > d->num_experts) {
    why = "prefill_slots must be in [0, num_experts]";
    return MOE_ERR_INVALID;
  }
  if (d->num_layers < 1 || d->num_experts < 1 || d->num_experts > 4096) {
    why = "need num_layers >= 1 and 1 <= num_experts <= 4096";
    return MOE_ERR_INVALID;
  }
  if (d->hidden < 256 || d->hidden % 256) { why = "hidden must be a positive multiple of 256"; return MOE_ERR_INVALID; }
  if (d->inter < 128 || d->inter % 128) { why = "inter must be a positive multiple of 128"; return MOE_ERR_INVALID; }
  if (d->top_k < 1 || d->top_k > kMaxTopK || d->top_k > d->num_experts) {
    why = "top_k must be in [1, min(E, 8)]";
    return MOE_ERR_INVALID;
  }
  if (d->weight_bits < 2 || d->weight_bits > 4) { why = "weight_bits must be 2, 3 or 4"; return MOE_ERR_INVALID; }
  if (d->group_size != 32 && d->group_size != 64 && d->group_size != 128) {
    why = "group_size must be 32, 64 or 128";
    return MOE_ERR_INVALID;
  }
  if (d->scale_dtype < MOE_SCALE_F32 || d->scale_dtype > MOE_SCALE_F16) { why = "bad scale_dtype"; return MOE_ERR_INVALID; }
  if (d->max_tokens < 1 || d->max_tokens > (1 << 20)) { why = "max_tokens must be in [1, 2^20]"; return MOE_ERR_INVALID; }
  if (d->cache_policy != MOE_POLICY_STATIC && d->cache_policy != MOE_POLICY_LFU) { why = "bad cache_policy"; return MOE_ERR_INVALID; }
  const int64_t total = (int64_t)d->num_layers * d->num_experts;
  if (d->cache_policy == MOE_POLICY_STATIC && (d->hbm_experts < 0 || d->hbm_experts > total)) {
    why = "hbm_experts must be in [0, L*E]";
    return MOE_ERR_INVALID;
  }
  if (d->cache_policy == MOE_POLICY_LFU && (d->cache_slots < 0 || d->cache_slots > total)) {
    why = "cache_slots must be in [0, L*E]";
    return MOE_ERR_INVALID;
  }
  if (d->cache_policy == MOE_POLICY_LFU &&
      (int64_t)d->num_layers * std::min<int64_t>(d->num_experts, (int64_t)d->max_tokens * d->top_k) > 50000) {
    why = "LFU cache: num_layers * min(E, max_tokens * top_k) must be <= 50000 (misses queued per step)";
    return MOE_ERR_INVALID;
  }
  if (d->reserved0 != 0) { why = "reserved0 must be zero"; return MOE_ERR_INVALID; }
  if (d->aging_period < 0) { why = "aging_period must be >= 0"; return MOE_ERR_INVALID; }
  return MOE_OK;
}

template <class T>
cudaError_t dalloc(T** p, size_t n) {
  return cudaMalloc(reinterpret_cast<void**>(p), std::max<size_t>(n, 1) * sizeof(T));
}

void release(Plan* p) {
  if (!p) return;
  cudaDeviceSynchronize();
  for (auto* w : p->wr) cudaFree(w);
  cudaFree(p->bias_all);
  cudaFree(p->wnorm_all);
  if (p->blas) cublasDestroy(p->blas);
  cudaFree(p->blas_ws);
  void* dev[] = {p->hbm_arena, p->pf_arena, p->pf_blob, p->pf_stage, p->blob_hbm, p->blob_host, p->logits, p->topk_idx, p->topk_w,
                 p->counts, p->offsets, p->perm, p->inv, p->wl_expert, p->wl_off, p->wl_cnt,
                 p->wl_blob, p->ctl, p->hbuf, p->obuf, p->pf_h, p->pf_o, p->pf_bucket, p->xsum, p->x_stage,
                 p->y_stage, p->slot_of, p->slot_owner, p->lfu_count, p->lfu_last, p->miss_list,
                 p->miss_count, p->adm_list, p->adm_count, p->stats};
  for (void* v : dev)
    if (v) cudaFree(v);
  pinned_free(p->host_arena);
  if (p->err_host) cudaFreeHost((void*)p->err_host);
  if (p->aux) cudaStreamDestroy(p->aux);
  if (p->ev_fork) cudaEventDestroy(p->ev_fork);
  if (p->ev_join) cudaEventDestroy(p->ev_join);
  if (p->ev_done) cudaEventDestroy(p->ev_done);
  delete p;
}

// Cross-stream ordering of a plan's forwards (they share its scratch): a
// forward on another stream than the previous one waits for it.  While the
// stream is being captured into a graph nothing is waited on or recorded --
// the graph's edges order its nodes, and an event recorded inside a capture
// could not be waited on by a later forward outside it.
cudaError_t order_before(Plan* p, cudaStream_t s, bool& capturing) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &st);
  if (e != cudaSuccess) return e;
  capturing = st != cudaStreamCaptureStatusNone;
  if (!capturing && p->have_last && p->last_stream != s) return cudaStreamWaitEvent(s, p->ev_done, 0);
  return cudaSuccess;
}

cudaError_t order_after(Plan* p, cudaStream_t s, bool capturing) {
  if (capturing) return cudaSuccess;
  const cudaError_t e = cudaEventRecord(p->ev_done, s);
  if (e == cudaSuccess) {
    p->last_stream = s;
    p->have_last = true;
  }
  return e;
}

}  // namespace

extern "C" moe_status moe_plan_create(const moe_plan_desc* desc, moe_plan** out) {
  std::string why;
  if (!out) return fail(nullptr, MOE_ERR_INVALID, "out is NULL");
  *out = nullptr;
  moe_status st = validate(desc, why);
  if (st != MOE_OK) return fail(nullptr, st, why);
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || desc->device < 0 || desc->device >= ndev) {
    cudaGetLastError();
    return fail(nullptr, MOE_ERR_INVALID, "no such CUDA device");
  }
  DeviceScope ds(desc->device);
  if (!ds.ok) return fail(nullptr, MOE_ERR_CUDA, "cudaSetDevice failed");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, desc->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, desc->device);
  if (major != 10 || minor != 3)
    return fail(nullptr, MOE_ERR_UNSUPPORTED, "the library targets sm_103a (GB300) only");

  Plan* p = new (std::nothrow) Plan();
  if (!p) return fail(nullptr, MOE_ERR_OOM, "host allocation failed");
  p->d = *desc;
  const moe_plan_desc& d = p->d;
  p->lay = make_layout(d.hidden, d.inter, d.weight_bits, d.group_size, d.scale_dtype);
  cudaDeviceGetAttribute(&p->sms, cudaDevAttrMultiProcessorCount, d.device);
  const int64_t LE = (int64_t)d.num_layers * d.num_experts;
  const int64_t E = d.num_experts, H = d.hidden, I = d.inter, k = d.top_k;
  const int64_t maxT = d.max_tokens;
  const int64_t decT = std::min<int64_t>(maxT, kDecodeMaxTokens);
  p->max_distinct = (int)std::min<int64_t>(E, maxT * k);
  const int64_t maxD = p->max_distinct;
  const int64_t slots = d.cache_policy == MOE_POLICY_LFU ? d.cache_slots : d.hbm_experts;
  const int64_t host_n = d.cache_policy == MOE_POLICY_LFU ? LE : LE - d.hbm_experts;
  p->hbm_cap = slots;
  p->host_cap = host_n;

  // HBM need: arena + routers + tables + scratch, against free memory minus headroom
  const int64_t scratch = maxT * E * 4 + maxT * k * 16 + (E + 1) * 8 + maxD * 32 +
                          maxD * decT * (I + 256) * 5 + decT * k * H * 8 +
                          (maxT > kDecodeMaxTokens ? maxT * k * (I + H) * 2 : 0) + 2 * maxT * H * 2 + 4096;
  const int64_t lfu = d.cache_policy == MOE_POLICY_LFU
                          ? LE * 12 + slots * 8 + (int64_t)d.num_layers * maxD * 8
                          : 0;
  const int64_t need = (slots + d.prefill_slots) * p->lay.blob_bytes + E * 8 * 3 +
                       (int64_t)d.num_layers * E * (H * 2 + 4) +
                       LE * 16 + scratch + lfu + (int64_t)d.num_layers * kNumStats * 8 + LE * 4 +
                       (maxT > kDecodeMaxTokens ? (int64_t)Plan::kBlasWorkspace : 0);
  size_t free_b = 0, total_b = 0;
  if (cudaMemGetInfo(&free_b, &total_b) != cudaSuccess) {
    release(p);
    return fail(nullptr, MOE_ERR_CUDA, "cudaMemGetInfo failed");
  }
  const int64_t headroom = std::max<int64_t>(int64_t(1) << 30, (int64_t)(total_b / 50));
  if (need > (int64_t)free_b - headroom) {
    char buf[256];
    snprintf(buf, sizeof buf, "plan needs %.2f GiB of HBM, %.2f GiB free minus %.2f GiB headroom",
             need / 1073741824.0, free_b / 1073741824.0, headroom / 1073741824.0);
    release(p);
    return fail(nullptr, MOE_ERR_OOM, buf);
  }

#define ALLOC(ptr, n)                                        \
  do {                                                       \
    cudaError_t e_ = dalloc(&(ptr), (size_t)(n));            \
    if (e_ != cudaSuccess) {                                 \
      cudaGetLastError();                                    \
      release(p);                                            \
      return fail(nullptr, MOE_ERR_OOM, "cudaMalloc " #ptr); \
    }                                                        \
  } while (0)

  if (slots > 0 && fault_injected("hbm_alloc")) {
    release(p);
    return fail(nullptr, MOE_ERR_OOM, "cudaMalloc p->hbm_arena (injected by MOE_FAULT=hbm_alloc)");
  }
  if (slots > 0) ALLOC(p->hbm_arena, (size_t)(slots * p->lay.blob_bytes));
  if (d.prefill_slots > 0) ALLOC(p->pf_arena, (size_t)(d.prefill_slots * p->lay.blob_bytes));
  ALLOC(p->pf_blob, E);
  ALLOC(p->pf_stage, 2 * E + 2);
  if (host_n > 0) {
    // on the GPU's own NUMA node ("763B MoE in two 96 GB cards", section "PCIe
    // topology": host memory across the socket interconnect slows every link read)
    p->numa_node = gpu_numa_node(d.device);
    p->host_arena = fault_injected("pinned_alloc")
                        ? nullptr
                        : static_cast<uint8_t*>(pinned_alloc((size_t)(host_n * p->lay.blob_bytes), p->numa_node));
    if (!p->host_arena) {
      release(p);
      return fail(nullptr, MOE_ERR_OOM, fault_injected("pinned_alloc")
                                            ? "pinned host arena allocation failed (injected by MOE_FAULT=pinned_alloc)"
                                            : "pinned host arena allocation failed");
    }
    if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&p->host_arena_dev), p->host_arena, 0) !=
        cudaSuccess) {
      release(p);
      return fail(nullptr, MOE_ERR_CUDA, "cudaHostGetDevicePointer failed");
    }
  }
  {
    void* eh = nullptr;
    if (cudaHostAlloc(&eh, 64, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
      release(p);
      return fail(nullptr, MOE_ERR_OOM, "error word allocation failed");
    }
    memset(eh, 0, 64);
    p->err_host = reinterpret_cast<volatile uint32_t*>(eh);
    cudaHostGetDevicePointer(reinterpret_cast<void**>(&p->err_dev), eh, 0);
  }
  ALLOC(p->blob_hbm, LE);
  ALLOC(p->blob_host, LE);
  ALLOC(p->logits, maxT * E);
  ALLOC(p->topk_idx, maxT * k);
  ALLOC(p->topk_w, maxT * k);
  ALLOC(p->counts, E);
  ALLOC(p->offsets, E + 1);
  ALLOC(p->perm, maxT * k);
  ALLOC(p->inv, maxT * k);
  ALLOC(p->wl_expert, maxD);
  ALLOC(p->wl_off, maxD);
  ALLOC(p->wl_cnt, maxD);
  ALLOC(p->wl_blob, maxD);
  ALLOC(p->ctl, 1);
  const int64_t KPI = p->lay.m[2].kpad;
  ALLOC(p->hbuf, maxD * decT * (KPI / 2));
  ALLOC(p->obuf, decT * k * H);
  ALLOC(p->xsum, decT * (H / d.group_size));
  if (maxT > kDecodeMaxTokens) {
    ALLOC(p->pf_h, maxT * k * I);
    ALLOC(p->pf_o, maxT * k * H);
    ALLOC(p->pf_bucket, E * ((maxT * k + kGroupChunk - 1) / kGroupChunk));
  }
  ALLOC(p->x_stage, maxT * H);
  ALLOC(p->y_stage, maxT * H);
  ALLOC(p->stats, (int64_t)d.num_layers * kNumStats);
  ALLOC(p->wnorm_all, LE);
  if (d.cache_policy == MOE_POLICY_LFU) {
    ALLOC(p->slot_of, LE);
    ALLOC(p->slot_owner, std::max<int64_t>(slots, 1));
    ALLOC(p->lfu_count, LE);
    ALLOC(p->lfu_last, LE);
    ALLOC(p->miss_list, (int64_t)d.num_layers * maxD);
    ALLOC(p->miss_count, 1);
    ALLOC(p->adm_list, 2 * (int64_t)d.num_layers * maxD + 2);
    ALLOC(p->adm_count, 4);
  }
  if (maxT > kDecodeMaxTokens) {  // prefill routing's tensor-core logits
    uint8_t* ws = nullptr;
    ALLOC(ws, Plan::kBlasWorkspace);
    p->blas_ws = ws;
    if (cublasCreate(&p->blas) != CUBLAS_STATUS_SUCCESS) {
      p->blas = nullptr;
      cudaGetLastError();
      release(p);
      return fail(nullptr, MOE_ERR_CUDA, "cublasCreate failed");
    }
    if (cublasSetWorkspace(p->blas, p->blas_ws, Plan::kBlasWorkspace) != CUBLAS_STATUS_SUCCESS ||
        cublasSetPointerMode(p->blas, CUBLAS_POINTER_MODE_HOST) != CUBLAS_STATUS_SUCCESS) {
      release(p);
      return fail(nullptr, MOE_ERR_CUDA, "cuBLAS workspace set-up failed");
    }
  }
#undef ALLOC
  p->wr.assign(d.num_layers, nullptr);
  p->bias.assign(d.num_layers, nullptr);
  if (dalloc(&p->bias_all, (int64_t)d.num_layers * E) != cudaSuccess) {
    cudaGetLastError();
    release(p);
    return fail(nullptr, MOE_ERR_OOM, "router allocation failed");
  }
  cudaMemset(p->bias_all, 0, (size_t)d.num_layers * E * 4);
  for (int l = 0; l < d.num_layers; ++l) {
    p->bias[l] = p->bias_all + (int64_t)l * E;
    if (dalloc(&p->wr[l], E * H) != cudaSuccess) {
      cudaGetLastError();
      release(p);
      return fail(nullptr, MOE_ERR_OOM, "router allocation failed");
    }
    cudaMemset(p->wr[l], 0, E * H * 2);
  }
  cudaMemset(p->blob_hbm, 0, LE * sizeof(void*));
  cudaMemset(p->blob_host, 0, LE * sizeof(void*));
  cudaMemset(p->ctl, 0, sizeof(Ctl));
  cudaMemset(p->hbuf, 0, (size_t)maxD * decT * (KPI / 2) * 8);  // epoch 0: never current
  cudaMemset(p->obuf, 0, (size_t)decT * k * H * 8);
  cudaMemset(p->stats, 0, (size_t)d.num_layers * kNumStats * 8);
  cudaMemset(p->wnorm_all, 0, LE * 4);  // the routers start as zeros
  if (d.cache_policy == MOE_POLICY_LFU) {
    cudaMemset(p->slot_of, 0xff, LE * 4);
    cudaMemset(p->slot_owner, 0xff, std::max<int64_t>(slots, 1) * 4);
    cudaMemset(p->lfu_count, 0, LE * 4);
    cudaMemset(p->lfu_last, 0xff, LE * 4);
    cudaMemset(p->miss_count, 0, 4);
    cudaMemset(p->adm_count, 0, 16);
  }
  p->hbm_pos.assign(LE, -1);
  p->host_pos.assign(LE, -1);
  p->placed.assign(LE, 0);
  p->tab_hbm.assign(LE, nullptr);
  p->tab_host.assign(LE, nullptr);
  if (cudaStreamCreateWithFlags(&p->aux, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_done, cudaEventDisableTiming) != cudaSuccess) {
    release(p);
    return fail(nullptr, MOE_ERR_CUDA, "stream/event creation failed");
  }
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    release(p);
    return fail(nullptr, MOE_ERR_CUDA, std::string("plan init: ") + cudaGetErrorString(e));
  }
  *out = reinterpret_cast<moe_plan*>(p);
  return MOE_OK;
}

extern "C" moe_status moe_plan_destroy(moe_plan* plan) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  DeviceScope ds(p->d.device);
  release(p);
  return MOE_OK;
}

extern "C" moe_status moe_set_router(moe_plan* plan, int layer, const uint16_t* wr,
                                     const float* bias) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  Busy b(p);
  if (!b.ok) return fail(p, MOE_ERR_STATE, "plan is in use by another thread");
  if (layer < 0 || layer >= p->d.num_layers || !wr) return fail(p, MOE_ERR_INVALID, "bad layer or wr");
  DeviceScope ds(p->d.device);
  const size_t E = p->d.num_experts, H = p->d.hidden;
  CK(p, cudaMemcpy(p->wr[layer], wr, E * H * 2, cudaMemcpyDefault));
  if (bias) CK(p, cudaMemcpy(p->bias[layer], bias, E * 4, cudaMemcpyDefault));
  else CK(p, cudaMemset(p->bias[layer], 0, E * 4));
  CK(p, router_norms(p->wr[layer], (int)E, (int)H, p->wnorm_all + layer * E, nullptr));
  CK(p, cudaDeviceSynchronize());
  return MOE_OK;
}

extern "C" moe_status moe_update_router_bias(moe_plan* plan, int layer, const float* bias,
                                             void* stream) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  Busy b(p);
  if (!b.ok) return fail(p, MOE_ERR_STATE, "plan is in use by another thread");
  if (layer < 0 || layer >= p->d.num_layers || !bias) return fail(p, MOE_ERR_INVALID, "bad layer or bias");
  DeviceScope ds(p->d.device);
  CK(p, cudaMemcpyAsync(p->bias[layer], bias, (size_t)p->d.num_experts * 4, cudaMemcpyDefault,
                        (cudaStream_t)stream));
  return MOE_OK;
}

extern "C" moe_status moe_debug_fail_next_forward(moe_plan* plan) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  p->fail_next = true;
  return MOE_OK;
}

extern "C" moe_status moe_update_router_biases(moe_plan* plan, int first, int count, const float* bias,
                                               void* stream) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  Busy b(p);
  if (!b.ok) return fail(p, MOE_ERR_STATE, "plan is in use by another thread");
  if (first < 0 || count < 0 || first > p->d.num_layers - count || !bias)
    return fail(p, MOE_ERR_INVALID, "bad layer range or bias");
  if (count == 0) return MOE_OK;
  DeviceScope ds(p->d.device);
  CK(p, cudaMemcpyAsync(p->bias[first], bias, (size_t)count * p->d.num_experts * 4, cudaMemcpyDefault,
                        (cudaStream_t)stream));
  return MOE_OK;
}

extern "C" moe_status moe_place_experts(moe_plan* plan, int layer, int first, int count,
                                        const uint8_t* residence, const moe_expert_weights* w) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  Busy b(p);
  if (!b.ok) return fail(p, MOE_ERR_STATE, "plan is in use by another thread");
  const moe_plan_desc& d = p->d;
  if (layer < 0 || layer >= d.num_layers || first < 0 || count < 0 ||
      first + count > d.num_experts || (count > 0 && !w))
    return fail(p, MOE_ERR_INVALID, "bad layer/first/count or weights");
  DeviceScope ds(p->d.device);
  const bool lfu = d.cache_policy == MOE_POLICY_LFU;
  const ExpertLayout& L = p->lay;
  // canonical (unpadded) sizes; staging for inputs on the host or misaligned
  int64_t canon_codes[3], canon_scales[3], stage_bytes = 0;
  for (int m = 0; m < 3; ++m) {
    canon_codes[m] = (int64_t)L.m[m].rows * L.m[m].cols * d.weight_bits / 8;
    canon_scales[m] = (int64_t)L.m[m].rows * (L.m[m].cols / d.group_size) * scale_size(d.scale_dtype);
    stage_bytes += align256(canon_codes[m]) + align256(canon_scales[m]);
  }
  uint8_t* stage = nullptr;
  cudaStream_t s = p->aux;
  moe_status st = MOE_OK;
  for (int i = 0; i < count && st == MOE_OK; ++i) {
    const int64_t g = (int64_t)layer * d.num_experts + first + i;
    const int res = lfu ? MOE_RES_HOST : (residence ? residence[i] : MOE_RES_HBM);
    if (res != MOE_RES_HBM && res != MOE_RES_HOST) { st = fail(p, MOE_ERR_INVALID, "bad residence"); break; }
    uint8_t* dst = nullptr;
    if (res == MOE_RES_HBM) {
      if (p->hbm_pos[g] < 0) {
        int64_t pos;
        if (!p->hbm_free.empty()) {  // a position freed by an expert that moved to host memory
          pos = p->hbm_free.back();
          p->hbm_free.pop_back();
        } else {
          if (p->hbm_used >= p->hbm_cap) { st = fail(p, MOE_ERR_OOM, "HBM expert arena is full"); break; }
          pos = p->hbm_used++;
        }
        p->hbm_pos[g] = pos;
      }
      dst = p->hbm_arena + p->hbm_pos[g] * L.blob_bytes;
    } else {
      if (p->host_pos[g] < 0) {
        if (p->host_used >= p->host_cap) { st = fail(p, MOE_ERR_OOM, "host expert arena is full"); break; }
        p->host_pos[g] = p->host_used++;
      }
      dst = p->host_arena_dev + p->host_pos[g] * L.blob_bytes;
    }
    uint8_t* sp = stage;
    bool staged = false;
    for (int m = 0; m < 3 && st == MOE_OK; ++m) {
      const void* c = w[i].codes[m];
      const void* sc = w[i].scales[m];
      if (!c || !sc) { st = fail(p, MOE_ERR_INVALID, "NULL codes or scales"); break; }
      const bool need_c = !is_device_ptr(c);
      const bool need_s = !is_device_ptr(sc) || (reinterpret_cast<uintptr_t>(sc) & 3);
      if ((need_c || need_s) && !stage) {
        cudaError_t e = cudaMalloc(&stage, (size_t)stage_bytes);
        if (e != cudaSuccess) { st = cuda_fail(p, e, "staging buffer"); break; }
        sp = stage;
        for (int q = 0; q < m; ++q) sp += align256(canon_codes[q]) + align256(canon_scales[q]);
      }
      const uint8_t* cd = static_cast<const uint8_t*>(c);
      if (need_c) {
        cudaError_t e = cudaMemcpyAsync(sp, c, (size_t)canon_codes[m], cudaMemcpyDefault, s);
        if (e != cudaSuccess) { st = cuda_fail(p, e, "stage codes"); break; }
        cd = sp;
        staged = true;
      }
      if (stage) sp += align256(canon_codes[m]);
      const uint8_t* sd = static_cast<const uint8_t*>(sc);
      if (need_s) {
        cudaError_t e = cudaMemcpyAsync(sp, sc, (size_t)canon_scales[m], cudaMemcpyDefault, s);
        if (e != cudaSuccess) { st = cuda_fail(p, e, "stage scales"); break; }
        sd = sp;
        staged = true;
      }
      if (stage) sp += align256(canon_scales[m]);
      cudaError_t e = launch_repack(cd, sd, dst, L.m[m], d.weight_bits, d.group_size, d.scale_dtype, s);
      if (e != cudaSuccess) { st = cuda_fail(p, e, "repack"); break; }
    }
    if (st != MOE_OK) break;
    if (res == MOE_RES_HOST && p->hbm_pos[g] >= 0) {  // moved out of HBM: free its position
      p->hbm_free.push_back(p->hbm_pos[g]);
      p->hbm_pos[g] = -1;
    }
    p->tab_hbm[g] = res == MOE_RES_HBM ? dst : nullptr;
    p->tab_host[g] = res == MOE_RES_HOST ? dst : nullptr;
    p->placed[g] = 1;
    if (staged) {  // the staging buffer is reused by the next expert
      cudaError_t e = cudaStreamSynchronize(s);
      if (e != cudaSuccess) { st = cuda_fail(p, e, "placement"); break; }
    }
  }
  if (st == MOE_OK && count > 0) {
    const int64_t g0 = (int64_t)layer * d.num_experts + first;
    cudaError_t e1 = cudaMemcpyAsync(p->blob_hbm + g0, p->tab_hbm.data() + g0,
                                     count * sizeof(void*), cudaMemcpyHostToDevice, s);
    cudaError_t e2 = cudaMemcpyAsync(p->blob_host + g0, p->tab_host.data() + g0,
                                     count * sizeof(void*), cudaMemcpyHostToDevice, s);
    if (e1 != cudaSuccess || e2 != cudaSuccess)
      st = cuda_fail(p, e1 != cudaSuccess ? e1 : e2, "tables");
  }
  {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess && st == MOE_OK) st = cuda_fail(p, e, "placement");
  }
  if (stage) cudaFree(stage);
  return st;
}

namespace {
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}

// moe_layer_forward, and with res / ysum (both non-NULL) the fused residual update
moe_status layer_forward(moe_plan* plan, int layer, const void* x, int T, void* y, const float* res,
                         void* ysum, void* stream, const moe_routing_out* dbg) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  Busy b(p);
  if (!b.ok) return fail(p, MOE_ERR_STATE, "plan is in use by another thread");
  const moe_plan_desc& d = p->d;
  if (layer < 0 || layer >= d.num_layers) return fail(p, MOE_ERR_INVALID, "bad layer");
  if (T < 0 || T > d.max_tokens) return fail(p, MOE_ERR_INVALID, "T outside [0, max_tokens]");
  if (T == 0) return MOE_OK;
  if (!x || !y || x == y) return fail(p, MOE_ERR_INVALID, "x and y must be distinct non-NULL device buffers");
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(y) & 3))
    return fail(p, MOE_ERR_INVALID, "x must be 16-byte aligned and y 4-byte aligned");
  if (ysum) {
    const size_t nb = (size_t)T * d.hidden * 2;
    if (!res) return fail(p, MOE_ERR_INVALID, "residual is NULL");
    if ((reinterpret_cast<uintptr_t>(res) & 15) || (reinterpret_cast<uintptr_t>(ysum) & 15))
      return fail(p, MOE_ERR_INVALID, "residual and out must be 16-byte aligned");
    if (overlap(ysum, nb, x, nb) || overlap(ysum, nb, y, nb) || overlap(ysum, nb, res, 2 * nb) ||
        overlap(res, 2 * nb, y, nb))
      return fail(p, MOE_ERR_INVALID, "out must not overlap x, y or residual, nor residual y");
  }
  const int64_t base = (int64_t)layer * d.num_experts;
  for (int e = 0; e < d.num_experts; ++e)
    if (!p->placed[base + e]) return fail(p, MOE_ERR_STATE, "every expert of the layer must be placed first");
  DeviceScope ds(p->d.device);
  if (*p->err_host) {
    cudaDeviceSynchronize();
    p->err_host[0] = 0;
    // epoch 0 and every hand-off word at epoch 0 again: no word written by an
    // earlier forward can be taken as current by a later one
    const int64_t decT = std::min<int64_t>(d.max_tokens, kDecodeMaxTokens);
    cudaMemset(&p->ctl->epoch, 0, sizeof(unsigned));
    cudaMemset(p->hbuf, 0, (size_t)p->max_distinct * decT * (p->lay.m[2].kpad / 2) * 8);
    cudaMemset(p->obuf, 0, (size_t)decT * d.top_k * d.hidden * 8);
    cudaDeviceSynchronize();
    return fail(p, MOE_ERR_TIMEOUT, "a bounded device-side wait of an earlier forward gave up");
  }
  if (take_overflow(p)) return fail(p, MOE_ERR_STATE, kOverflowMsg);
  cudaStream_t s = (cudaStream_t)stream;
  bool capturing = false;
  CK(p, order_before(p, s, capturing));
  cudaError_t e;
  if (T <= kDecodeMaxTokens)
    e = decode_forward(*p, layer, (const uint16_t*)x, T, (uint16_t*)y, s, dbg, res, (uint16_t*)ysum);
  else
    e = prefill_forward(*p, layer, (const uint16_t*)x, T, (uint16_t*)y, s, dbg, true, nullptr, res,
                        (uint16_t*)ysum);
  if (e != cudaSuccess) return forward_fail(p, e, "forward launch");
  CK(p, order_after(p, s, capturing));
  return MOE_OK;
}
}  // namespace

extern "C" moe_status moe_layer_forward(moe_plan* plan, int layer, const void* x, int T, void* y,
                                        void* stream, const moe_routing_out* dbg) {
  return layer_forward(plan, layer, x, T, y, nullptr, nullptr, stream, dbg);
}

extern "C" moe_status moe_layer_forward_residual(moe_plan* plan, int layer, const void* x, int T, void* y,
                                                 const float* residual, void* out, void* stream) {
  if (T > 0 && !out) return fail(reinterpret_cast<Plan*>(plan), MOE_ERR_INVALID, "out is NULL");
  return layer_forward(plan, layer, x, T, y, residual, out, stream, nullptr);
}

extern "C" moe_status moe_prefill_forward(moe_plan* plan, int layer, const void* x, int64_t T, void* y,
                                          void* stream) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  Busy b(p);
  if (!b.ok) return fail(p, MOE_ERR_STATE, "plan is in use by another thread");
  const moe_plan_desc& d = p->d;
  if (layer < 0 || layer >= d.num_layers) return fail(p, MOE_ERR_INVALID, "bad layer");
  if (T < 0) return fail(p, MOE_ERR_INVALID, "T < 0");
  if (T == 0) return MOE_OK;
  if (d.max_tokens <= kDecodeMaxTokens)
    return fail(p, MOE_ERR_UNSUPPORTED, "chunked prefill needs max_tokens > 8 (prefill-path chunks)");
  if (!x || !y || x == y) return fail(p, MOE_ERR_INVALID, "x and y must be distinct non-NULL device buffers");
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(y) & 15))
    return fail(p, MOE_ERR_INVALID, "x and y must be 16-byte aligned");
  const int64_t base = (int64_t)layer * d.num_experts;
  for (int e = 0; e < d.num_experts; ++e)
    if (!p->placed[base + e]) return fail(p, MOE_ERR_STATE, "every expert of the layer must be placed first");
  DeviceScope ds(p->d.device);
  if (*p->err_host) return fail(p, MOE_ERR_STATE, "a latched device error is pending: call moe_layer_forward");
  if (take_overflow(p)) return fail(p, MOE_ERR_STATE, kOverflowMsg);
  cudaStream_t s = (cudaStream_t)stream;
  bool capturing = false;
  CK(p, order_before(p, s, capturing));
  const int64_t chunk = std::min<int64_t>(8192, d.max_tokens), H = d.hidden;
  // Staging pays back only over several chunks (it moves each host expert
  // over the link once instead of once per chunk): with one chunk every
  // expert is read in place.  The copies precede the first chunk; overlapping
  // them with a first chunk that reads the same experts in place was measured
  // slower, both sharing the link.
  const bool stage = T > chunk && d.prefill_slots > 0;
  cudaError_t e = cudaSuccess;
  if (stage && (e = prefill_stage(*p, layer, s)) != cudaSuccess) return cuda_fail(p, e, "prefill staging");
  for (int64_t off = 0; off < T; off += chunk) {
    const int tc = (int)std::min<int64_t>(chunk, T - off);
    e = prefill_forward(*p, layer, static_cast<const uint16_t*>(x) + off * H, tc,
                        static_cast<uint16_t*>(y) + off * H, s, nullptr, /*lfu=*/false,
                        stage ? p->pf_blob : nullptr);
    if (e != cudaSuccess) return forward_fail(p, e, "prefill chunk");
  }
  CK(p, order_after(p, s, capturing));
  return MOE_OK;
}

namespace {
// The address through which `device` reaches a page-locked host buffer that
// was allocated or registered for it (nullptr otherwise: pageable memory, or
// another device's)
void* device_mapping(const void* h, int device) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost && at.device == device ? at.devicePointer : nullptr;
}
}  // namespace

extern "C" moe_status moe_layer_forward_host(moe_plan* plan, int layer, const void* x_host, int T,
                                             void* y_host, void* stream) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  if (T < 0 || T > p->d.max_tokens) return fail(p, MOE_ERR_INVALID, "T outside [0, max_tokens]");
  if (T == 0) return MOE_OK;
  if (!x_host || !y_host) return fail(p, MOE_ERR_INVALID, "NULL host buffer");
  const size_t bytes = (size_t)T * p->d.hidden * 2;
  if (T <= kDecodeMaxTokens) {
    // Page-locked buffers of a decode-sized batch: x comes in by a copy kernel
    // through its device mapping and the forward's combine writes y straight
    // into y_host's (a copy-engine operation costs ~7.6 us of stream latency
    // at these sizes, the kernel ~4.1 us, the direct writes nothing extra).
    const void* xd = device_mapping(x_host, p->d.device);
    void* yd = device_mapping(y_host, p->d.device);
    if (xd && yd && !(reinterpret_cast<uintptr_t>(xd) & 15) && !(reinterpret_cast<uintptr_t>(yd) & 3)) {
      const int n16 = (int)(bytes / 16);
      {
        DeviceScope ds(p->d.device);
        copy16_kernel<<<(n16 + 255) / 256, 256, 0, (cudaStream_t)stream>>>(static_cast<const uint4*>(xd),
                                                                          reinterpret_cast<uint4*>(p->x_stage), n16);
        CK(p, cudaGetLastError());
      }
      return moe_layer_forward(plan, layer, p->x_stage, T, yd, stream, nullptr);
    }
  }
  {
    DeviceScope ds(p->d.device);
    CK(p, cudaMemcpyAsync(p->x_stage, x_host, bytes, cudaMemcpyHostToDevice, (cudaStream_t)stream));
  }
  moe_status st = moe_layer_forward(plan, layer, p->x_stage, T, p->y_stage, stream, nullptr);
  if (st != MOE_OK) return st;
  DeviceScope ds(p->d.device);
  CK(p, cudaMemcpyAsync(y_host, p->y_stage, bytes, cudaMemcpyDeviceToHost, (cudaStream_t)stream));
  return MOE_OK;
}

extern "C" moe_status moe_step_end(moe_plan* plan, void* stream) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  Busy b(p);
  if (!b.ok) return fail(p, MOE_ERR_STATE, "plan is in use by another thread");
  DeviceScope ds(p->d.device);
  if (p->d.cache_policy == MOE_POLICY_LFU) {
    cudaError_t e = lfu_step_end(*p, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(p, e, "step end");
  }
  p->step += 1;
  // the step end ran (on the queued misses); an overflow seen by now is reported
  if (take_overflow(p)) return fail(p, MOE_ERR_STATE, kOverflowMsg);
  return MOE_OK;
}

extern "C" moe_status moe_cache_stats(moe_plan* plan, int layer, moe_cache_stats_t* out, int reset) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  Busy b(p);
  if (!b.ok) return fail(p, MOE_ERR_STATE, "plan is in use by another thread");
  if (!out || layer < -1 || layer >= p->d.num_layers) return fail(p, MOE_ERR_INVALID, "bad layer or out");
  DeviceScope ds(p->d.device);
  const int L = p->d.num_layers;
  std::vector<unsigned long long> h((size_t)L * kNumStats);
  CK(p, cudaDeviceSynchronize());
  CK(p, cudaMemcpy(h.data(), p->stats, h.size() * 8, cudaMemcpyDeviceToHost));
  const bool overflow = take_overflow(p);
  uint64_t acc[kNumStats] = {0};
  for (int l = 0; l < L; ++l)
    if (layer < 0 || l == layer)
      for (int i = 0; i < kNumStats; ++i) acc[i] += h[(size_t)l * kNumStats + i];
  out->accesses = acc[kStatAccesses];
  out->hits = acc[kStatHits];
  out->misses = acc[kStatMisses];
  out->admissions = acc[kStatAdmissions];
  out->evictions = acc[kStatEvictions];
  out->hbm_bytes = acc[kStatHbmBytes];
  out->host_bytes = acc[kStatHostBytes];
  out->fill_bytes = acc[kStatFillBytes];
  out->pairs = acc[kStatPairs];
  out->forwards = acc[kStatForwards];
  out->router_exact = acc[kStatRouterExact];
  if (reset) {
    if (layer < 0) CK(p, cudaMemset(p->stats, 0, h.size() * 8));
    else CK(p, cudaMemset(p->stats + (size_t)layer * kNumStats, 0, kNumStats * 8));
    CK(p, cudaDeviceSynchronize());
  }
  if (overflow) return fail(p, MOE_ERR_STATE, kOverflowMsg);  // *out is filled all the same
  return MOE_OK;
}

extern "C" moe_status moe_residence_table(moe_plan* plan, int layer, int32_t* out_host) {
  Plan* p = reinterpret_cast<Plan*>(plan);
  if (!p) return fail(nullptr, MOE_ERR_INVALID, "plan is NULL");
  Busy b(p);
  if (!b.ok) return fail(p, MOE_ERR_STATE, "plan is in use by another thread");
  if (!out_host || layer < 0 || layer >= p->d.num_layers) return fail(p, MOE_ERR_INVALID, "bad layer or out");
  DeviceScope ds(p->d.device);
  const int E = p->d.num_experts;
  const int64_t base = (int64_t)layer * E;
  if (p->d.cache_policy == MOE_POLICY_LFU) {
    CK(p, cudaDeviceSynchronize());
    CK(p, cudaMemcpy(out_host, p->slot_of + base, (size_t)E * 4, cudaMemcpyDeviceToHost));
  } else {
    for (int e = 0; e < E; ++e) out_host[e] = (int32_t)p->hbm_pos[base + e];
  }
  return MOE_OK;
}

extern "C" moe_status moe_quantize(const float* w, int rows, int cols, int bits, int group,
                                   int sdt, void* codes, void* scales, void* stream) {
  if (!w || !codes || !scales || rows <= 0 || cols <= 0 || bits < 2 || bits > 8 || group <= 0 ||
      (group % 32) || cols % group || sdt < 0 || sdt > 2)
    return fail(nullptr, MOE_ERR_INVALID,
                "bad quantiser arguments (group must be a multiple of 32 dividing cols)");
  if ((reinterpret_cast<uintptr_t>(codes) & 3) || (reinterpret_cast<uintptr_t>(w) & 3))
    return fail(nullptr, MOE_ERR_INVALID, "w and codes must be 4-byte aligned");
  cudaError_t e = launch_quantize(w, rows, cols, bits, group, sdt, static_cast<uint8_t*>(codes),
                                  scales, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "quantize");
  return MOE_OK;
}

extern "C" moe_status moe_probe_bandwidth(int device, size_t bytes, int iters, double* host_gbs,
                                          double* hbm_gbs) {
  if (bytes < (1u << 20) || iters < 1)
    return fail(nullptr, MOE_ERR_INVALID, "bytes >= 1 MiB and iters >= 1");
  DeviceScope ds(device);
  bytes &= ~size_t(15);
  void* h = nullptr;
  void* hd = nullptr;
  void* dv = nullptr;
  unsigned* sink = nullptr;
  cudaEvent_t a, b;
  moe_status st = MOE_OK;
  if (cudaHostAlloc(&h, bytes, cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    return fail(nullptr, MOE_ERR_OOM, "pinned probe buffer");
  }
  memset(h, 1, bytes);
  cudaHostGetDevicePointer(&hd, h, 0);
  if (cudaMalloc(&dv, bytes) != cudaSuccess || cudaMalloc(&sink, 4) != cudaSuccess) {
    cudaGetLastError();
    cudaFreeHost(h);
    if (dv) cudaFree(dv);
    return fail(nullptr, MOE_ERR_OOM, "device probe buffer");
  }
  cudaMemset(dv, 1, bytes);
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  const int64_t n16 = (int64_t)(bytes / 16);
  for (int which = 0; which < 2; ++which) {
    const uint4* src = reinterpret_cast<const uint4*>(which == 0 ? hd : dv);
    float best = 1e30f;
    for (int it = 0; it < iters + 1; ++it) {
      cudaEventRecord(a);
      read_probe_kernel<<<sms * 8, 512>>>(src, n16, sink);
      cudaEventRecord(b);
      if (cudaEventSynchronize(b) != cudaSuccess) { st = fail(nullptr, MOE_ERR_CUDA, "probe kernel"); break; }
      float ms = 0;
      cudaEventElapsedTime(&ms, a, b);
      if (it > 0) best = std::min(best, ms);
    }
    const double gbs = bytes / (best * 1e-3) / 1e9;
    if (which == 0 && host_gbs) *host_gbs = gbs;
    if (which == 1 && hbm_gbs) *hbm_gbs = gbs;
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  cudaFree(dv);
  cudaFree(sink);
  cudaFreeHost(h);
  return st;
}

extern "C" const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID: return "MOE_ERR_INVALID";
    case MOE_ERR_OOM: return "MOE_ERR_OOM";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_STATE: return "MOE_ERR_STATE";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
  }
  return "MOE_ERR_UNKNOWN";
}

extern "C" const char* moe_last_error(const moe_plan* plan) {
  const Plan* p = reinterpret_cast<const Plan*>(plan);
  return p ? p->last_error.c_str() : g_last_error_noplan.c_str();
}
