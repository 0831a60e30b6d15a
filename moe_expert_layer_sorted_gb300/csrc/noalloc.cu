// Routing that allocates nothing: router logits and top-k for callers that
// cannot call cudaMalloc.  The logits live in a fixed device array of this
// library; its memory is committed in a CUDA context when the library's
// module is loaded there (with lazy module loading, at this entry point's
// first call on that device, which also looks up the array's address); see
// moe_route_noalloc in moe.h.
#include <mutex>

#include "internal.h"

using namespace moe;

namespace {

// Largest T * E this entry point accepts (1 MiB of fp32 logits).
constexpr int64_t kNoAllocMaxLogits = int64_t(1) << 18;

// Every GPU that loads the library holds this array until the process exits.
// Host code must not pass its name to a kernel: on the host it is only a
// stand-in; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_route_scratch[kNoAllocMaxLogits];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch[kMaxDevices] = {};  // device address of g_route_scratch, per device

__device__ __forceinline__ float bf16bits(uint32_t h) { return __uint_as_float(h << 16); }

// Logits in the library's fixed summation order (the same order as the
// plan-based forward): lane j accumulates fmaf over i = 256m + 8j + r,
// m then r ascending, from +0; xor-butterfly adds 16, 8, 4, 2, 1; bias last.
// One warp per (token, expert).
__global__ void noalloc_logits_kernel(const uint16_t* __restrict__ x, int T, int H,
                                      const uint16_t* __restrict__ wr,
                                      const float* __restrict__ bias, int E,
                                      float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= (int64_t)T * E) return;
  const int t = (int)(wid / E), e = (int)(wid % E);
  const uint4* xv = reinterpret_cast<const uint4*>(x + (int64_t)t * H);
  const uint4* wv = reinterpret_cast<const uint4*>(wr + (int64_t)e * H);
  float acc = 0.0f;
  for (int m = 0; m < H / 256; ++m) {
    const uint4 a = __ldg(xv + m * 32 + lane), b = __ldg(wv + m * 32 + lane);
    const uint32_t aq[4] = {a.x, a.y, a.z, a.w}, bq[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t ab = (r & 1) ? (aq[r >> 1] >> 16) : (aq[r >> 1] & 0xffffu);
      const uint32_t bb = (r & 1) ? (bq[r >> 1] >> 16) : (bq[r >> 1] & 0xffffu);
      acc = fmaf(bf16bits(ab), bf16bits(bb), acc);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) acc = acc + __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) logits[wid] = acc + (bias ? bias[e] : 0.0f);
}

// Order-preserving integer key of a logit (-0 folded to +0): larger float,
// larger key; the same key the plan's forward paths select on.
__device__ __forceinline__ uint32_t logit_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one token per warp: k rounds, each taking every lane's best
// untaken logit (largest key; lanes scan experts in ascending order, so the
// lower index wins a tie within a lane), then the warp's largest key and,
// among the lanes holding it, the lowest expert index (ties to the lower
// index); then the softmax renormalised over the k chosen, summed in j order.
__global__ void noalloc_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                    int32_t* __restrict__ idx, float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* l = logits + (int64_t)t * E;
  int chosen[kMaxTopK];
  float cv[kMaxTopK];
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;  // below every real key
    int bi = -1;
    for (int e = lane; e < E; e += 32) {
      bool taken = false;
      for (int q = 0; q < j; ++q) taken |= chosen[q] == e;
      const uint32_t key = logit_key(l[e]);
      if (!taken && (bi < 0 || key > bk)) {
        bk = key;
        bi = e;
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bi >= 0 ? bk : 0u);
    const uint32_t mine = (bi >= 0 && bk == kmax) ? (uint32_t)bi : 0xffffffffu;
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
      w[(int64_t)t * k + j] = ex[j] / z;
    }
  }
}

}  // namespace

// Address of the fixed array on the current device, looked up once per device
// (the lookup loads the module into the context if it is not yet loaded).
static moe_status scratch_for_current_device(float** out, int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();  // leave no error behind for the caller's next check
      return MOE_ERR_CUDA;
    }
    g_scratch[dev] = static_cast<float*>(p);
  }
  *out = g_scratch[dev];
  *dev_out = dev;
  return MOE_OK;
}

extern "C" moe_status moe_route_noalloc(const void* x_bf16, int T, int H, const void* wr_bf16,
                                        const float* bias, int E, int k, int32_t* topk_idx,
                                        float* topk_w, void* stream) {
  if (T < 0 || H < 256 || H % 256 || E < 1 || k < 1 || k > kMaxTopK || k > E) {
    return MOE_ERR_INVALID;
  }
  if ((int64_t)T * E > kNoAllocMaxLogits) {
    return MOE_ERR_INVALID;
  }
  // buffers are only read or written when there are tokens (T = 0 may pass NULL)
  if (T > 0 && (!x_bf16 || !wr_bf16 || !topk_idx || !topk_w)) {
    return MOE_ERR_INVALID;
  }
  if (T > 0 && ((reinterpret_cast<uintptr_t>(x_bf16) & 15) || (reinterpret_cast<uintptr_t>(wr_bf16) & 15))) {
    return MOE_ERR_INVALID;
  }
  // set-up first, so that a call with T = 0 can serve as the warm-up
  float* logits = nullptr;
  int dev = -1;
  const moe_status st = scratch_for_current_device(&logits, &dev);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int sdev = -1;  // the array's address is per device: the stream must be the current device's
  if (cudaStreamGetDevice(s, &sdev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_INVALID;
  }
  if (sdev != dev) return MOE_ERR_INVALID;
  if (T == 0) return MOE_OK;
  const int64_t warps = (int64_t)T * E;
  noalloc_logits_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(
      static_cast<const uint16_t*>(x_bf16), T, H, static_cast<const uint16_t*>(wr_bf16), bias, E,
      logits);
  noalloc_topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
