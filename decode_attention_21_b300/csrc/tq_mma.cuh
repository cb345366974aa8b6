// Device helpers shared by the scoring kernels: legacy tensor-core MMA,
// fp16 splitting, and the expansion of packed bit words into subnormal fp16
// tensor-core operands.
#pragma once
#include <cuda_fp16.h>

#include "tq_internal.cuh"

namespace tq {
namespace mma {

constexpr unsigned kFull = 0xffffffffu;

// Odd subsets of the code planes (bit p <-> plane p) in increasing order; the
// first 2^(b'-1) entries are exactly the odd subsets of b' planes.
__device__ constexpr uint32_t kOddMask[8] = {1u, 2u, 4u, 7u, 8u, 11u, 13u, 14u};

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// fp16 piece of x: 0 -> round(x), 1 -> round(x - round(x)).
__device__ __forceinline__ float piece16(float x, int which) {
  const float hi = __half2float(__float2half_rn(x));
  return which == 0 ? hi : x - hi;
}

// The 16 fp16 operand registers of one packed word: register beta holds bits
// beta and beta+16 (low and high half) at mantissa position 6 + (beta mod 4).
__device__ __forceinline__ void expand16(uint32_t w, uint32_t (&r)[16]) {
  const uint32_t t0 = w << 6, t1 = w << 2, t2 = w >> 2, t3 = w >> 6;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t m = 0x00400040u << e;
    r[e] = t0 & m;
    r[4 + e] = t1 & m;
    r[8 + e] = t2 & m;
    r[12 + e] = t3 & m;
  }
}

// Power of two s with amax / s <= target (1 for amax = 0).
__device__ __forceinline__ float pow2_scale(float amax, float target) {
  if (!(amax > 0.f)) return 1.f;
  int e;
  frexpf(amax / target, &e);
  return ldexpf(1.f, e);
}

}  // namespace mma
}  // namespace tq
