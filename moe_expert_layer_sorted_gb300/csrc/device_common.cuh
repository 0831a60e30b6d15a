// Device helpers shared by the decode and prefill kernels (included into an
// anonymous namespace of each translation unit).
#pragma once

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ float scale_at(const uint8_t* base, int idx, int sdt) {
  if (sdt == MOE_SCALE_F32) return reinterpret_cast<const float*>(base)[idx];
  const unsigned short h = reinterpret_cast<const unsigned short*>(base)[idx];
  if (sdt == MOE_SCALE_BF16) return __uint_as_float((uint32_t)h << 16);
  return __half2float(__ushort_as_half(h));
}

// ---- mbarrier-tracked ring slots.  Each slot has a "full" barrier (one
// arrival per use: the producer's expect_tx for an HBM unit, whose bulk
// copies complete the bytes; for a host unit, lane 0 after every producer
// lane has tied its cp.async copies to the barrier) and an "empty" barrier
// (one arrival per consumer warp once it no longer reads the slot).  Pinned
// host memory is read with plain 16-byte cp.async, as everywhere else in
// this library.
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// this thread's earlier cp.async copies arrive on bar when they land (the
// pending count is raised now, so the phase cannot complete before that)
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// barrier among the consumer warps only (the producer warp never joins it)
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
}
// bytes (a multiple of 16, both addresses 16-byte aligned) HBM -> shared, completing on bar
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Bounded wait for phase `parity` of bar: ~2^20 tries, each suspending the
// thread until the phase completes or a time limit passes -- a 1 us hint, or
// (kHint false) the system's own limit, which measured about as long and wakes
// the thread sooner after the phase completes (the prefill GEMM's pipeline runs
// a few percent faster with it); latches a timeout (and gives up at once once
// one is latched).
template <bool kHint = true>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err) {
  for (uint32_t it = 0; it < (1u << 20); ++it) {
    uint32_t ok;
    if constexpr (kHint)
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n"
          " selp.u32 %0, 1, 0, p;\n}"
          : "=r"(ok)
          : "r"(bar), "r"(parity)
          : "memory");
    else
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
          " selp.u32 %0, 1, 0, p;\n}"
          : "=r"(ok)
          : "r"(bar), "r"(parity)
          : "memory");
    if (ok) return true;
    if ((it & 255u) == 255u && *reinterpret_cast<volatile uint32_t*>(err)) return false;
  }
  *reinterpret_cast<volatile uint32_t*>(err) = kErrTimeout;
  __threadfence_system();
  return false;
}

// Bounded wait used before a CTA exits: the copies or MMAs that complete the
// phase were issued by this CTA and finish by themselves, so it waits even
// after an error was latched (at most ~2^16 tries).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < (1u << 16); ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return;
  }
}

// (a & m) | c in one instruction.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
  return d;
}

// (128 + c u) -> (128 + u) in both bf16 halves, c = 1/mul: exact (a power-of-two
// scale and a sum that bf16 represents)
__device__ __forceinline__ uint32_t rescale_bf16x2(uint32_t v, uint32_t mul2, uint32_t add2) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(v), "r"(mul2), "r"(add2));
  return d;
}

// bf16x2 register (128 + u_lo, 128 + u_hi) of pair P (0..63) of a lane's
// 256-column block held in w (its 4*B words); P is a compile-time constant
// after unrolling.  Field placement: see repack_codes_kernel in plan.cu.
// A field in bits 0..6 of a half-word can be masked straight into the bf16
// mantissa of 128 (value 128 + 2^s u for a field at bit s), so only every
// second or third field needs a shift; those at s > 0 are rescaled by one
// bf16x2 fma (u < 2^b, so every intermediate is exact).
template <int B>
__device__ __forceinline__ uint32_t pair_of(const uint32_t (&w)[4 * B], int P) {
  constexpr uint32_t kMagic = 0x43004300u;  // bf16 128.0 in both halves
  if constexpr (B == 4) {
    return and_or(w[P >> 2] >> (4 * (P & 3)), 0x000F000Fu, kMagic);
  } else if constexpr (B == 2) {  // fields at bits 0, 2, 4 | 6, 8, 10 | 12, 14
    const uint32_t x = w[P >> 3] >> (6 * ((P & 7) / 3));
    switch ((P & 7) % 3) {
      case 0: return and_or(x, 0x00030003u, kMagic);
      case 1: return rescale_bf16x2(and_or(x, 0x000C000Cu, kMagic), 0x3E803E80u, 0x42C042C0u);  // 0.25, 96
      default: return rescale_bf16x2(and_or(x, 0x00300030u, kMagic), 0x3D803D80u, 0x42F042F0u);  // 1/16, 120
    }
  } else {
    const int t = P >> 4, m = P & 15;
    if (m < 15) {  // fields at bits 0, 3 | 6, 9 | 12
      const uint32_t x = w[3 * t + m / 5] >> (6 * ((m % 5) / 2));
      if ((m % 5) % 2 == 0) return and_or(x, 0x00070007u, kMagic);
      return rescale_bf16x2(and_or(x, 0x00380038u, kMagic), 0x3E003E00u, 0x42E042E0u);  // 0.125, 112
    }
    const uint32_t v = and_or(w[3 * t] >> 15, 0x00010001u, kMagic);
    const uint32_t u = and_or(w[3 * t + 1] >> 14, 0x00020002u, v);
    return and_or(w[3 * t + 2] >> 13, 0x00040004u, u);
  }
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

