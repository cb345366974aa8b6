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

// m16n8k8: A rows g, g + 8 at k = 2c, 2c + 1 (a0, a1); B at k = 2c, 2c + 1.
__device__ __forceinline__ void mma_f16_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
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

// fp16 hi and lo pieces of two floats, packed: hi = pack(round(x0), round(x1)),
// lo = pack(round(x0 - hi0), round(x1 - hi1)); the same bits as
// pack_half2(piece16(x0, w), piece16(x1, w)) for w = 0, 1, in three
// conversions instead of six.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 f = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - f.x, x1 - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Piece `which` (0 = hi, 1 = lo) of two floats, packed: the same bits as
// pack_half2(piece16(x0, which), piece16(x1, which)).
__device__ __forceinline__ uint32_t piece2(float x0, float x1, int which) {
  uint32_t hi, lo;
  split2(x0, x1, hi, lo);
  return which ? lo : hi;
}

// Packed bits as fp16 tensor-core operands.  A half whose only set bit is
// bit p <= 11 is exactly 2^(p - 24) (bits 0..9 are subnormal mantissa bits,
// bits 10 and 11 the two lowest exponent bits).  Operand register beta holds
// bits beta and beta + 16 of a word w: in place for beta < 12, from w >> 4
// (so at position beta - 4) for beta >= 12.  The other side of the product
// carries bit_factor(beta) = 1 / (value of the set bit).
__host__ __device__ constexpr float bit_factor(int beta) {
  return beta < 12 ? (float)(1u << (24 - beta)) : (float)(1u << (28 - beta));
}
constexpr float kMaxBitFactor = 16777216.f;  // bit_factor(0) = 2^24

// Operand register beta of word w (w4 = w >> 4).
__device__ __forceinline__ uint32_t bit_operand(uint32_t w, uint32_t w4, int beta) {
  return beta < 12 ? (w & (0x00010001u << beta)) : (w4 & (0x00010001u << (beta - 4)));
}

// All 16 operand registers of one word.
__device__ __forceinline__ void expand16(uint32_t w, uint32_t (&r)[16]) {
  const uint32_t w4 = w >> 4;
#pragma unroll
  for (int beta = 0; beta < 16; ++beta) r[beta] = bit_operand(w, w4, beta);
}

// Variant for operands multiplied by small values (softmax weights): chained
// fp16 MMAs accumulate products of the deepest subnormals (bits 0..5) less
// accurately, so bits 0..5 move up by 6 (from w << 6).  Every set bit is then
// worth 2^-18 .. 2^-13 and value_factor(beta) = 1 / (value of the set bit).
__host__ __device__ constexpr float value_factor(int beta) {
  return beta < 6 ? (float)(1u << (18 - beta)) : bit_factor(beta);
}

__device__ __forceinline__ void expand16_v(uint32_t w, uint32_t (&r)[16]) {
  const uint32_t w6 = w << 6, w4 = w >> 4;
#pragma unroll
  for (int beta = 0; beta < 16; ++beta)
    r[beta] = beta < 6 ? (w6 & (0x00010001u << (beta + 6))) : bit_operand(w, w4, beta);
}

// Two-level sum of the PV products of a warp.  An mma.sync chain adds each
// tile's products into its fp32 accumulator inside the tensor core, which
// drops low-order bits of small addends against a large running sum; over a
// long context (thousands of tiles per warp) that drifts by ~1e-4 relative.
// So the chain runs over a few tiles only, and flush() moves its sum into
// fp32 registers with ordinary adds.  t[mt][0/1] = the two coordinates of the
// thread's C fragment, hi and lo weight pieces already combined.
struct PvTotal {
  float t[8][2];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) t[mt][0] = t[mt][1] = 0.f;
  }
  __device__ __forceinline__ void scale(float a) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      t[mt][0] *= a;
      t[mt][1] *= a;
    }
  }
  __device__ __forceinline__ void flush(float (&acc)[8][4]) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      t[mt][0] += acc[mt][0] + acc[mt][1];
      t[mt][1] += acc[mt][2] + acc[mt][3];
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
    }
  }
};
constexpr int kPvFlushStages = 4;   // stages (2 tiles per warp each) per mma chain

// Power of two s with amax / s <= target (1 for amax = 0).
__device__ __forceinline__ float pow2_scale(float amax, float target) {
  if (!(amax > 0.f)) return 1.f;
  int e;
  frexpf(amax / target, &e);
  return ldexpf(1.f, e);
}

}  // namespace mma
}  // namespace tq
