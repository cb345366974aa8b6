// Recursive-polar stage 1 inside the tensor-core quantize kernels: the
// epilogue between the rotation GEMM and the sketch GEMM.
//
// [xujun] note-189244, 第一步：PolarQuant (pairs of coordinates, then pairs
// of radii, each angle coded on its own law); [suzuke] "TurboQuant:
// compressing AI consciousness", 第二步 (polar coordinates + Max-Lloyd).
//
// A row y (d = 128 or 256, in tensor memory: lane = row, column = coordinate)
// is coded by the threads that own its 32-coordinate blocks.  Angle slots
// follow the polar record layout: inside block k, level-1 angles at bits
// 0..15, level 2 at 16..23, level 3 at 24..27, level 4 at 28..29, level 5
// at 30; the angles of levels 6..log2 d sit at bit 31 of the word columns in
// heap order (root first).
#pragma once
#include <cstdint>

#include "tq_internal.cuh"
#include "tq_tc.cuh"

namespace tq {
namespace polar {

// Per level l (index l): the cell thresholds (level 1: tan t of the
// boundaries inside the first quadrant; levels >= 2: tan^2 t) and the
// centroids' cos and sin.
struct Tables {
  float thr[kMaxLevels][kMaxL], cc[kMaxLevels][kMaxL], cs[kMaxLevels][kMaxL];
};

__device__ __forceinline__ void load_tables(const Dev& cb, Tables& tb, int tid, int nthreads) {
  for (int i = tid; i < kMaxLevels * kMaxL; i += nthreads) {
    const int l = i / kMaxL, t = i % kMaxL;
    const float tn = cb.pb_cos[l][t] != 0.f ? cb.pb_sin[l][t] / cb.pb_cos[l][t] : 0.f;
    tb.thr[l][t] = l == 1 ? tn : tn * tn;
    tb.cc[l][t] = cb.pc_cos[l][t];
    tb.cs[l][t] = cb.pc_sin[l][t];
  }
}

// Polar angle cells in fp32.  An angle psi of level >= 2 with squared child
// radii (Ra, Rb) is >= a boundary t in (0, pi/2) iff Rb >= Ra tan^2 t, so the
// tree runs on squared radii (R = Ra + Rb, no square root) against tan^2
// thresholds; inside a level-1 quadrant the test is br >= ar tan t.  These are
// the exact decisions up to fp32 rounding (points within about 1e-6 of a
// boundary, relative).  The cell is the number of boundaries at or below the
// angle, by bisection over the increasing thresholds.
template <int N>
__device__ __forceinline__ int cell_sq(const float* thr, float Ra, float Rb) {
  int c = 0;
#pragma unroll
  for (int step = N >> 1; step; step >>= 1)
    if (Rb >= Ra * thr[c + step - 1]) c += step;
  return c;
}

// Level-1 cell of the pair (p, q) on the full circle: the quadrant from the
// signs, then the cell inside the quadrant (L / 4 cells per quadrant).
template <int L>
__device__ __forceinline__ int level1_cell(const float* tan1, float p, float q) {
  int Q = 0;
  if (p <= 0.f && q > 0.f) Q = 1;
  else if (p < 0.f && q <= 0.f) Q = 2;
  else if (p >= 0.f && q < 0.f) Q = 3;
  if constexpr (L <= 4) {
    return L == 2 ? Q >> 1 : Q;
  } else {
    const float ar = Q == 0 ? p : (Q == 1 ? q : (Q == 2 ? -p : -q));
    const float br = Q == 0 ? q : (Q == 1 ? -p : (Q == 2 ? -q : p));
    int c = 0;
#pragma unroll
    for (int step = L >> 3; step; step >>= 1)
      if (br >= ar * tan1[c + step - 1]) c += step;
    return Q * (L >> 2) + c;
  }
}

// Bit k of each of the 8 nibbles of w, packed into bits 0..7.
__device__ __forceinline__ uint32_t nibble_bits(uint32_t w, int k) {
  uint32_t x = (w >> k) & 0x11111111u;
  x = (x | (x >> 3)) & 0x03030303u;
  x = (x | (x >> 6)) & 0x000F000Fu;
  return (x | (x >> 12)) & 0xFFu;
}


// The polar codes (and, for PROD, the residual operand) of the blocks
// blk0 .. blk0 + NCH - 1 of row m.
//   y_tmem: tensor-memory address (with the lane offset) of column 0 of Y;
//   rhi_tmem, rlo_tmem: where the residual goes as bf16 pairs (column
//     16 k + i of block k holds coordinates 32 k + 2 i and 2 i + 1);
//   inv: 1 / ||y||; red3: [d / 32][128] floats of shared memory for the
//   block radii; sync(): a barrier over every thread of the tile;
//   words[h][p]: code plane p of block blk0 + h; gs: += ||r||^2 (PROD).
template <int D, int NCH, int B1, bool PROD, int NWD, class Sync>
__device__ __forceinline__ void epilogue(const Tables& tb, uint32_t y_tmem, uint32_t rhi_tmem, uint32_t rlo_tmem,
                                         int blk0, float inv, float* red3, int m, uint32_t (&words)[NCH][NWD],
                                         float& gs, Sync&& sync) {
  using namespace tc;
  constexpr int NB = D / 32;                       // 32-coordinate blocks of the row
  constexpr int LOGD = D == 128 ? 7 : 8;
  constexpr int L = 1 << B1;
  static_assert(NWD >= B1, "code planes");
  // levels 1..5 inside this thread's blocks: the 4-bit codes of slots
  // 0..30 of each word column, packed 8 to a word (slot s: nibble s % 8
  // of cn[h][s / 8])
  uint32_t cn[NCH][4];
#pragma unroll
  for (int h = 0; h < NCH; ++h) {
    float y[32];
    tmem_ld32(y_tmem + 32 * (blk0 + h), y);
    float R[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) cn[h][k] = 0u;
#pragma unroll
    for (int a = 0; a < 16; ++a) {
      const float p = y[2 * a] * inv, q = y[2 * a + 1] * inv;
      cn[h][a >> 3] |= (uint32_t)level1_cell<L>(tb.thr[1], p, q) << (4 * (a & 7));
      R[a] = fmaf(q, q, p * p);
    }
#pragma unroll
    for (int lev = 2; lev <= 5; ++lev) {
#pragma unroll
      for (int j = 0; j < (32 >> lev); ++j) {
        const int slot = 32 - (64 >> lev) + j;
        cn[h][slot >> 3] |= (uint32_t)cell_sq<L>(tb.thr[lev], R[2 * j], R[2 * j + 1]) << (4 * (slot & 7));
        R[j] = R[2 * j] + R[2 * j + 1];
      }
    }
    red3[(blk0 + h) * 128 + m] = R[0];
  }
  sync();
  // levels 6..log2 d over the squared block radii; the code of level l,
  // angle j sits at heap index 2^(log2 d - l) - 1 + j (slot 31 of that
  // word column); kept packed, 4 bits per heap index
  float rr[NB];
  uint32_t hcw = 0u;
#pragma unroll
  for (int k = 0; k < NB; ++k) rr[k] = red3[k * 128 + m];
#pragma unroll
  for (int lev = 6; lev <= LOGD; ++lev) {
#pragma unroll
    for (int j = 0; j < (D >> lev); ++j) {
      hcw |= (uint32_t)cell_sq<L>(tb.thr[lev], rr[2 * j], rr[2 * j + 1]) << (4 * ((1 << (LOGD - lev)) - 1 + j));
      rr[j] = rr[2 * j] + rr[2 * j + 1];
    }
  }
#pragma unroll
  for (int h = 0; h < NCH; ++h) {
    const int wc = blk0 + h;
    if (wc < NB - 1) cn[h][3] |= ((hcw >> (4 * wc)) & 15u) << 28;
    // plane p of the word column: bit b' - 1 - p of every slot's code
#pragma unroll
    for (int p = 0; p < B1; ++p) {
      words[h][p] = 0u;
#pragma unroll
      for (int k = 0; k < 4; ++k) words[h][p] |= nibble_bits(cn[h][k], B1 - 1 - p) << (8 * k);
    }
  }
  if constexpr (PROD) {
    // the reproduction from root radius 1: down the heap to this
    // thread's block radius, then inside the block to the coordinates;
    // residual r = y / n - yhat
#pragma unroll
    for (int h = 0; h < NCH; ++h) {
      const int wc = blk0 + h;
      float t[16];
      t[0] = 1.f;
#pragma unroll
      for (int lev = LOGD; lev >= 6; --lev) {
        const int j = wc >> (lev - 5);                 // node of level lev above block wc
        const int c = (int)((hcw >> (4 * ((1 << (LOGD - lev)) - 1 + j))) & 15u);
        t[0] *= ((wc >> (lev - 6)) & 1) ? tb.cs[lev][c] : tb.cc[lev][c];
      }
#pragma unroll
      for (int lev = 5; lev >= 2; --lev) {
#pragma unroll
        for (int j = (32 >> lev) - 1; j >= 0; --j) {
          const int slot = 32 - (64 >> lev) + j;
          const int c = (int)((cn[h][slot >> 3] >> (4 * (slot & 7))) & 15u);
          const float r0 = t[j];
          t[2 * j + 1] = r0 * tb.cs[lev][c];
          t[2 * j] = r0 * tb.cc[lev][c];
        }
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[16];
        tmem_ld16(y_tmem + 32 * (blk0 + h) + 16 * half, v);
        uint32_t rh2[8], rl2[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const int a = 8 * half + (e >> 1);
          const int c = (int)((cn[h][a >> 3] >> (4 * (a & 7))) & 15u);
          const float r0 = v[e] * inv - t[a] * tb.cc[1][c];
          const float r1 = v[e + 1] * inv - t[a] * tb.cs[1][c];
          gs = fmaf(r0, r0, gs);
          gs = fmaf(r1, r1, gs);
          const uint32_t hb = bf16x2(r0, r1);
          rh2[e >> 1] = hb;
          rl2[e >> 1] = bf16x2(r0 - __uint_as_float(hb << 16), r1 - __uint_as_float(hb & 0xFFFF0000u));
        }
        const uint32_t col = (uint32_t)(16 * (blk0 + h) + 8 * half);
        tmem_st8(rhi_tmem + col, rh2);
        tmem_st8(rlo_tmem + col, rl2);
      }
    }
  }
}

}  // namespace polar
}  // namespace tq
