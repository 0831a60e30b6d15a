/*
 * Device twin of synth.c's normal draws, for inputs too large to generate on
 * the host in reasonable time (the 40-layer and 24k-expert stacks).  Same
 * counter-based SplitMix64 stream and the same Irwin-Hall sum of the four
 * 16-bit fields of a draw, scaled by the same fp32 multiplier computed the
 * same way on the host, so every value is bit-identical to synth_normal_f32 /
 * synth_normal_bf16.  Random draws only: no MoE arithmetic lives here.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#define GAMMA 0x9E3779B97F4A7C15ULL
#define IH4_SD 37837.22723720648
#define IH4_MEAN 131070

__device__ __forceinline__ uint64_t fin64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float draw_normal(uint64_t key, uint64_t i, float mul) {
  const uint64_t u = fin64(key + (i + 1) * GAMMA);
  const int32_t s = (int32_t)(u & 0xFFFF) + (int32_t)((u >> 16) & 0xFFFF) +
                    (int32_t)((u >> 32) & 0xFFFF) + (int32_t)(u >> 48) - IH4_MEAN;
  return __fmul_rn((float)s, mul);
}

__global__ void normal_f32_kernel(uint64_t key, uint64_t start, int64_t n, float mul, float* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = draw_normal(key, start + (uint64_t)i, mul);
}

__global__ void normal_bf16_kernel(uint64_t key, uint64_t start, int64_t n, float mul, uint16_t* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    uint32_t u = __float_as_uint(draw_normal(key, start + (uint64_t)i, mul));
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) {
      out[i] = 0x7FC0;
      continue;
    }
    u += 0x7FFFu + ((u >> 16) & 1u);
    out[i] = (uint16_t)(u >> 16);
  }
}

static float multiplier(float sigma) { return (float)((double)sigma / IH4_SD); }

/* out (device) [i] = sigma * N01(key, start + i), i in [0, n), on `stream` */
extern "C" int synth_gpu_normal_f32(uint64_t key, uint64_t start, int64_t n, float sigma, float* out,
                                    void* stream) {
  if (n <= 0) return 0;
  const int64_t blocks = (n + 255) / 256 < 65536 ? (n + 255) / 256 : 65536;
  normal_f32_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(key, start, n, multiplier(sigma), out);
  return (int)cudaGetLastError();
}

extern "C" int synth_gpu_normal_bf16(uint64_t key, uint64_t start, int64_t n, float sigma, uint16_t* out,
                                     void* stream) {
  if (n <= 0) return 0;
  const int64_t blocks = (n + 255) / 256 < 65536 ? (n + 255) / 256 : 65536;
  normal_bf16_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(key, start, n, multiplier(sigma), out);
  return (int)cudaGetLastError();
}

/* Stacked-layer input: out[i] = bf16(float(y[i]) + noise[i]) (fp32 add, round to
   nearest even; NaN to the canonical quiet NaN), the next layer's input in the
   chained-layer workloads. */
__global__ void residual_bf16_kernel(const uint16_t* y, const float* noise, int64_t n, uint16_t* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    uint32_t u = __float_as_uint(__fadd_rn(__uint_as_float((uint32_t)y[i] << 16), noise[i]));
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) {
      out[i] = 0x7FC0;
      continue;
    }
    u += 0x7FFFu + ((u >> 16) & 1u);
    out[i] = (uint16_t)(u >> 16);
  }
}

extern "C" int synth_gpu_residual_bf16(const uint16_t* y, const float* noise, int64_t n, uint16_t* out,
                                       void* stream) {
  if (n <= 0) return 0;
  const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
  residual_bf16_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(y, noise, n, out);
  return (int)cudaGetLastError();
}
