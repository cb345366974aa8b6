// Scoring of recursive-polar caches ([xujun] note-189244, 第一步 recursive
// pairing of radii; [suzuke] 第二步 polar coordinates + Max-Lloyd angles):
// the stage-1 reproduction is a product of cosines and sines down the tree,
// so it is decoded to fp32 per key (or value) and fed to the tensor cores as
// fp16 hi + lo operands; the QJL term is the same sign-plane contraction as
// in scalar mode.  d = 128, tree of 7 levels, subtrees of 32 leaves per
// packed word (see the polar layout in tq.h).
//
//   logits: A = decoded keys (16 keys x 16 coordinates, hi then lo; a
//           thread's k slots 2c, 2c + 1, 2c + 8, 2c + 9 of k block kb are
//           coordinates 4 kb .. 4 kb + 3 of its subtree c, so each half of
//           the subtree is decoded and consumed on its own),
//           B = q' (fp16 hi/lo columns of the G <= 4 heads);
//   attention PV: A = decoded values (16 coordinates x 8 tokens per m16n8k8,
//           the two tokens of a pair in the two fp16 halves: tokens 2c,
//           2c + 1, then 2c + 8, 2c + 9 of the tile), B = p_t n_v,t.
// The query fragments are read from shared memory where they are used.
#include <cuda_fp16.h>

#include "tq_internal.cuh"
#include "tq_mma.cuh"
#include "tq_stage.cuh"

namespace tq {

using namespace mma;
using namespace stage;

namespace {

constexpr int kLevels = 7;   // log2(128)

// (cos, sin) of the centroid of code k at tree level l, in shared memory.
struct PolarTab {
  float2 t[kLevels + 1][16];
};

__device__ __forceinline__ void load_tab(const Dev& cb, PolarTab& tab) {
  for (int e = threadIdx.x; e < (kLevels + 1) * 16; e += blockDim.x) {
    const int l = e >> 4, k = e & 15;
    tab.t[l][k] = make_float2(cb.pc_cos[l][k], cb.pc_sin[l][k]);
  }
}

// Code of the angle stored at bit `bit` of the B planes' words (plane 0 = MSB).
template <int B>
__device__ __forceinline__ int code_at(const uint32_t (&w)[B], int bit) {
  int c = 0;
#pragma unroll
  for (int p = 0; p < B; ++p) c = (c << 1) | ((w[p] >> bit) & 1u);
  return c;
}

// Radius of subtree s (32 leaves) of a unit row: root angle (bit 31 of word 0)
// and the level-6 angle (bit 31 of word 1 + s/2).
template <int B>
__device__ __forceinline__ float subtree_radius(const PolarTab& tab, const uint32_t (&w0)[B],
                                                const uint32_t (&w6)[B], int s) {
  const float2 r7 = tab.t[7][code_at<B>(w0, 31)];
  const float rho6 = (s >> 1) ? r7.y : r7.x;
  const float2 r6 = tab.t[6][code_at<B>(w6, 31)];
  return rho6 * ((s & 1) ? r6.y : r6.x);
}

// Codes at bit positions pos .. pos + 7 of the B plane words (plane 0 = the
// code's most significant bit), gathered into the nibbles of one word:
// nibble i = the code at position pos + i.  Each plane's byte is spread to
// nibble spacing by three shift-and-mask steps, so eight codes cost about
// 8 B instructions instead of about 3 B each.
template <int B>
__device__ __forceinline__ uint32_t codes_x8(const uint32_t (&w)[B], int pos) {
  uint32_t r = 0;
#pragma unroll
  for (int p = 0; p < B; ++p) {
    uint32_t x = (w[p] >> pos) & 0xFFu;
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    x = (x | (x << 3)) & 0x11111111u;
    r = (r << 1) | x;
  }
  return r;
}

// (cos, sin) of the level-l centroid whose code is nibble i of r: the
// nibble shifted straight to its byte offset in the table row (code x 8).
__device__ __forceinline__ float2 tab_nib(const PolarTab& tab, int l, uint32_t r, int i) {
  const uint32_t off = i == 0 ? (r << 3) & 0x78u : (r >> (4 * i - 3)) & 0x78u;
  return *reinterpret_cast<const float2*>(reinterpret_cast<const char*>(&tab.t[l][0]) + off);
}

// The 16 leaves of half h of subtree s, starting from the subtree radius.
// Angle codes of a subtree word: level 1 at bits 0..15, level 2 at 16..23,
// level 3 at 24..27, level 4 at 28..29, level 5 at 30.
template <int B>
__device__ __forceinline__ void decode_half(const PolarTab& tab, const uint32_t (&ws)[B], float rho5, int h,
                                            float (&y)[16]) {
  const uint32_t n1 = codes_x8<B>(ws, 8 * h);        // level 1: codes 8h .. 8h + 7
  const uint32_t n2 = codes_x8<B>(ws, 16 + 4 * h);   // level 2: nibbles 0..3
  const uint32_t n3 = codes_x8<B>(ws, 24);           // level 3: nibbles 0..3, level 4: 4, 5, level 5: 6
  const float2 a5 = tab_nib(tab, 5, n3, 6);
  const float rho4 = rho5 * (h ? a5.y : a5.x);
  const float2 a4 = tab_nib(tab, 4, n3, 4 + h);
  float r3[2] = {rho4 * a4.x, rho4 * a4.y};
  float r2[4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float2 a = tab_nib(tab, 3, n3, 2 * h + i);
    r2[2 * i] = r3[i] * a.x;
    r2[2 * i + 1] = r3[i] * a.y;
  }
  float r1[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = tab_nib(tab, 2, n2, i);
    r1[2 * i] = r2[i] * a.x;
    r1[2 * i + 1] = r2[i] * a.y;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 a = tab_nib(tab, 1, n1, i);
    y[2 * i] = r1[i] * a.x;
    y[2 * i + 1] = r1[i] * a.y;
  }
}

__device__ __forceinline__ float dot32p(const float* __restrict__ MT, const float* xs, int i, int qt) {
  constexpr int d = 128;
  const float* col = MT + (size_t)(32 * qt) * d + i;
  float m[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) m[j] = __ldg(col + (size_t)j * d);
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) acc = fmaf(m[j], xs[32 * qt + j], acc);
  return acc;
}

}  // namespace

// Query preparation for polar keys: plane 0 = q' (plain fp16 hi/lo, the key
// side is decoded to normal fp16 values), plane 1 = the QJL plane exactly as
// in scalar mode.  Header: S1[4], S2[4], K1[4] = 0, K2[4] = -sum q''.
__global__ void __launch_bounds__(512) k_prep_polar(const Dev cb, const float* __restrict__ q, int Hq, int Hkv,
                                                    uint8_t* __restrict__ prep) {
  constexpr int d = 128;
  const int G = Hq / Hkv;
  const int kvh = blockIdx.x >> 2, slot = blockIdx.x & 3, b = blockIdx.y;
  const bool live = slot < G;
  __shared__ float sq[d], sq1[d], sq2[d], part[4][d], part2[4][d];
  __shared__ float red[3];
  const int tid = threadIdx.x;
  const int i = tid & 127, qt = tid >> 7;
  if (tid < d) sq[tid] = live ? q[((size_t)b * Hq + kvh * G + slot) * d + tid] : 0.f;
  __syncthreads();
  // q' = Pi q and q'' = (S Pi) q in the same pass
  part[qt][i] = dot32p(cb.PiT, sq, i, qt);
  part2[qt][i] = dot32p(cb.SPT, sq, i, qt);
  __syncthreads();
  if (tid < d) {
    sq1[tid] = (part[0][tid] + part[1][tid]) + (part[2][tid] + part[3][tid]);
    sq2[tid] = (part2[0][tid] + part2[1][tid]) + (part2[2][tid] + part2[3][tid]);
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < 3) {
    float v = 0.f;
    for (int k = lane; k < d; k += 32) {
      if (warp == 0) v = fmaxf(v, fabsf(sq1[k]));
      else if (warp == 1) v = fmaxf(v, 2.f * fabsf(sq2[k]));
      else v += sq2[k];
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float u = __shfl_xor_sync(kFull, v, o);
      v = warp < 2 ? fmaxf(v, u) : v + u;
    }
    if (lane == 0) red[warp] = v;
  }
  __syncthreads();
  const float S1 = pow2_scale(red[0], 16384.f), S2 = pow2_scale(red[1] * kMaxBitFactor, 16384.f);
  uint8_t* blk = prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(d);
  float* hdr = reinterpret_cast<float*>(blk);
  if (tid == 0) {
    hdr[slot] = live ? S1 : 0.f;
    hdr[4 + slot] = live ? S2 : 0.f;
    hdr[8 + slot] = 0.f;
    hdr[12 + slot] = live ? -red[2] : 0.f;
  }
  uint2* frag = reinterpret_cast<uint2*>(blk + kPrepHeader);
  for (int e = tid; e < 2 * 8 * 8; e += blockDim.x) {
    const int sub = e & 7, kb = (e >> 3) & 7, v = e >> 6;
    const int pc = sub >> 2, c = sub & 3;
    const int g = 2 * slot + pc;
    float vals[4] = {0.f, 0.f, 0.f, 0.f};
    if (live) {
      for (int t = 0; t < 4; ++t) {
        // stage 1: k slots 2c, 2c + 1, 2c + 8, 2c + 9 = coordinates
        // 4 kb + t of subtree c; QJL: bits beta and beta + 16 of the sign
        // word (the bit-operand layout of scalar mode)
        const int beta = 2 * kb + (t >> 1);
        const int k = v == 0 ? 32 * c + 4 * kb + t : 32 * c + beta + 16 * (t & 1);
        const float x = v == 0 ? sq1[k] / S1 : 2.f * sq2[k] * bit_factor(beta) / S2;
        vals[t] = piece16(x, pc);
      }
    }
    frag[(v * 8 + kb) * 32 + g * 4 + c] = make_uint2(pack_half2(vals[0], vals[1]), pack_half2(vals[2], vals[3]));
  }
}

// Words of one key the thread needs: its own column c (all P planes) and
// the top-path words 0 and 1 + c/2 of the B code planes.
template <int B>
struct PKey {
  uint32_t ws[B + 1], w0[B], w6[B];
  uint32_t nrm;
  __device__ __forceinline__ void load(const uint32_t* rec, const uint32_t* nrm_p, int64_t row, int W, int c,
                                       bool valid) {
    constexpr int P = B + 1;
    if (!valid) {
#pragma unroll
      for (int p = 0; p < P; ++p) ws[p] = 0;
#pragma unroll
      for (int p = 0; p < B; ++p) w0[p] = w6[p] = 0;
      nrm = 0;
      return;
    }
    const uint32_t* r = rec + row * W;
#pragma unroll
    for (int p = 0; p < P; ++p) ws[p] = __ldg(r + c * P + p);
#pragma unroll
    for (int p = 0; p < B; ++p) {
      w0[p] = __ldg(r + p);
      w6[p] = __ldg(r + (1 + (c >> 1)) * P + p);
    }
    nrm = __ldg(nrm_p + row);
  }
  // the same words from a record already in shared memory (r = record start)
  __device__ __forceinline__ void load_row(const uint32_t* r, uint32_t nrm_bits, int c, bool valid) {
    constexpr int P = B + 1;
#pragma unroll
    for (int p = 0; p < P; ++p) ws[p] = valid ? r[c * P + p] : 0u;
#pragma unroll
    for (int p = 0; p < B; ++p) {
      w0[p] = valid ? r[p] : 0u;
      w6[p] = valid ? r[(1 + (c >> 1)) * P + p] : 0u;
    }
    nrm = valid ? nrm_bits : 0u;
  }
  // leaves 16 h .. 16 h + 15 of subtree c (unit row), from its radius rho5
  __device__ __forceinline__ void decode_h(const PolarTab& tab, float rho5, int h, float (&y)[16]) const {
    uint32_t cw[B];
#pragma unroll
    for (int p = 0; p < B; ++p) cw[p] = ws[p];
    decode_half<B>(tab, cw, rho5, h, y);
  }
};

// The query fragments of one (sequence, kv head) from the prep block into
// shared memory: [plane][k block][lane].
__device__ __forceinline__ void load_frags(const uint8_t* blk, uint2* sfrag) {
  const uint2* frag = reinterpret_cast<const uint2*>(blk + kPrepHeader);
  for (int e = threadIdx.x; e < 2 * 8 * 32; e += blockDim.x) sfrag[e] = frag[e];
}

// inner products (stage 1, QJL) of keys g and g+8 for head slot c
template <int B>
__device__ __forceinline__ void polar_qk(const PolarTab& tab, const uint2* sfrag, int lane, const PKey<B>& ka,
                                         const PKey<B>& kb_, int c, float& s1a, float& s1b, float& s2a,
                                         float& s2b) {
  float acc1[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    uint32_t ra[16], rb[16];
    expand16(ka.ws[B], ra);
    expand16(kb_.ws[B], rb);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint2 bq = sfrag[(8 + k) * 32 + lane];
      mma_f16(acc2[k & 1], ra[2 * k], rb[2 * k], ra[2 * k + 1], rb[2 * k + 1], bq.x, bq.y);
    }
  }
  const float rha = subtree_radius<B>(tab, ka.w0, ka.w6, c), rhb = subtree_radius<B>(tab, kb_.w0, kb_.w6, c);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float ya[16], yb[16];
    ka.decode_h(tab, rha, h, ya);
    kb_.decode_h(tab, rhb, h, yb);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint2 bq = sfrag[(4 * h + kk) * 32 + lane];
      uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
      split2(ya[4 * kk], ya[4 * kk + 1], h0, l0);
      split2(yb[4 * kk], yb[4 * kk + 1], h1, l1);
      split2(ya[4 * kk + 2], ya[4 * kk + 3], h2, l2);
      split2(yb[4 * kk + 2], yb[4 * kk + 3], h3, l3);
      mma_f16(acc1[0], h0, h1, h2, h3, bq.x, bq.y);
      mma_f16(acc1[1], l0, l1, l2, l3, bq.x, bq.y);
    }
  }
  s1a = (acc1[0][0] + acc1[0][1]) + (acc1[1][0] + acc1[1][1]);
  s1b = (acc1[0][2] + acc1[0][3]) + (acc1[1][2] + acc1[1][3]);
  s2a = (acc2[0][0] + acc2[0][1]) + (acc2[1][0] + acc2[1][1]);
  s2b = (acc2[0][2] + acc2[0][3]) + (acc2[1][2] + acc2[1][3]);
}

// PV of one k8 half of a tile: yv[j][i] = coordinate i of the thread's 16
// for token 2c + j (+ 8 for the second half), bw = the weights of those two
// tokens (this thread's fp16 piece); hi pieces, then lo, per accumulator.
__device__ __forceinline__ void pv_pair(float (&acc)[8][4], const float (&yv)[2][16], uint32_t bw) {
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t h0, l0, h1, l1;
    split2(yv[0][2 * mt], yv[1][2 * mt], h0, l0);
    split2(yv[0][2 * mt + 1], yv[1][2 * mt + 1], h1, l1);
    mma_f16_k8(acc[mt], h0, h1, bw);
    mma_f16_k8(acc[mt], l0, l1, bw);
  }
}

__device__ __forceinline__ float est_polar(uint32_t nrm_bits, float s1, float s2, float kq) {
  const __half2 h = *reinterpret_cast<const __half2*>(&nrm_bits);
  return __low2float(h) * fmaf(__high2float(h) * kq, s2, s1);
}

template <int B>
__global__ void __launch_bounds__(128) k_logits_polar(const Dev cb, const uint8_t* __restrict__ kcache, int Hq,
                                                      int Hkv, int64_t capacity, int64_t cache_rows, const RowMap map,
                                                      const int32_t* __restrict__ seq_lens,
                                                      const uint8_t* __restrict__ prep, float* __restrict__ logits,
                                                      int tiles_per_cta, int* __restrict__ status) {
  __shared__ PolarTab tab;
  __shared__ uint2 sfrag[2 * 8 * 32];
  load_tab(cb, tab);
  const int kvh = blockIdx.y, b = blockIdx.z;
  const uint8_t* blk = prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(128);
  load_frags(blk, sfrag);
  __syncthreads();
  const int G = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t L = seq_lens[b];
  const int64_t ntiles = (L + 15) / 16;
  const int64_t tile0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t tend = min(tile0 + tiles_per_cta, ntiles);
  if (tile0 + warp >= tend) return;
  const float* hdr = reinterpret_cast<const float*>(blk);
  const float S1 = hdr[c], S2 = hdr[4 + c], K2 = hdr[12 + c];
  const uint32_t* recs = reinterpret_cast<const uint32_t*>(kcache);
  const uint32_t* nrm = reinterpret_cast<const uint32_t*>(kcache + norm_offset(cb, cache_rows));
  const float kq = cb.qjl_const;
  float* out = logits + ((size_t)b * Hq + (size_t)kvh * G + c) * capacity;
  for (int64_t tile = tile0 + warp; tile < tend; tile += 4) {
    const int64_t ta = tile * 16 + g, tb = ta + 8;
    const int64_t row0 = tile_row(map, b, kvh, Hkv, capacity, tile * 16, status);   // cache row of the tile's token 0
    PKey<B> ka, kb_;
    ka.load(recs, nrm, row0 + g, cb.W, c, ta < L);
    kb_.load(recs, nrm, row0 + g + 8, cb.W, c, tb < L);
    float s1a, s1b, s2a, s2b;
    polar_qk<B>(tab, sfrag, lane, ka, kb_, c, s1a, s1b, s2a, s2b);
    if (c < G) {
      if (ta < L) out[ta] = est_polar(ka.nrm, S1 * s1a, fmaf(S2, s2a, K2), kq);
      if (tb < L) out[tb] = est_polar(kb_.nrm, S1 * s1b, fmaf(S2, s2b, K2), kq);
    }
  }
}

template <int BK, int BV>
__global__ void __launch_bounds__(128, 3) k_attn_polar(const Dev kcb, const Dev vcb, const uint8_t* __restrict__ kcache,
                                                       const uint8_t* __restrict__ vcache, int Hq, int Hkv,
                                                       int64_t capacity, int64_t cache_rows,
                                                       const int32_t* __restrict__ seq_lens,
                                                       const uint8_t* __restrict__ prep, float scale_log2,
                                                       float* __restrict__ partials, int tiles_per_cta) {
  __shared__ PolarTab ktab, vtab;
  __shared__ uint2 sfrag[2 * 8 * 32];
  load_tab(kcb, ktab);
  load_tab(vcb, vtab);
  const int kvh = blockIdx.y, b = blockIdx.z;
  const uint8_t* blk = prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(128);
  load_frags(blk, sfrag);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t L = seq_lens[b];
  const int64_t ntiles = (L + 15) / 16;
  const int64_t tile0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t tend = min(tile0 + tiles_per_cta, ntiles);
  float m_run = -INFINITY, l_run = 0.f;
  float acc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
  PvTotal tot;
  tot.zero();
  if (tile0 + warp < tend) {
    const float* hdr = reinterpret_cast<const float*>(blk);
    const float S1 = hdr[c], S2 = hdr[4 + c], K2 = hdr[12 + c];
    const uint32_t* krec = reinterpret_cast<const uint32_t*>(kcache);
    const uint32_t* knrm = reinterpret_cast<const uint32_t*>(kcache + norm_offset(kcb, cache_rows));
    const uint32_t* vrec = reinterpret_cast<const uint32_t*>(vcache);
    const __half* vnrm = reinterpret_cast<const __half*>(vcache + norm_offset(vcb, cache_rows));
    const int64_t rowbase = ((int64_t)b * Hkv + kvh) * capacity;
    const float kq = kcb.qjl_const;
    const int hh = g >> 1, pc = g & 1;
    const int src0 = (2 * c) * 4 + hh, src1 = (2 * c + 1) * 4 + hh;
    const int vs = g >> 1, vh = g & 1;   // value subtree and half of this thread's 16 coordinates
    int chain = 0;    // tiles in the current mma chain
    for (int64_t tile = tile0 + warp; tile < tend; tile += 4) {
      const int64_t t0 = tile * 16, ta = t0 + g, tb = ta + 8;
      PKey<BK> ka, kb_;
      ka.load(krec, knrm, rowbase + ta, kcb.W, c, ta < L);
      kb_.load(krec, knrm, rowbase + tb, kcb.W, c, tb < L);
      float s1a, s1b, s2a, s2b;
      polar_qk<BK>(ktab, sfrag, lane, ka, kb_, c, s1a, s1b, s2a, s2b);
      const float sa = ta < L ? est_polar(ka.nrm, S1 * s1a, fmaf(S2, s2a, K2), kq) * scale_log2 : -INFINITY;
      const float sb = tb < L ? est_polar(kb_.nrm, S1 * s1b, fmaf(S2, s2b, K2), kq) * scale_log2 : -INFINITY;
      float mx = fmaxf(sa, sb);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      if (__any_sync(kFull, mx > m_run)) {
        const float m_new = fmaxf(m_run, mx);
        const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
        l_run *= alpha;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mt][e] *= alpha;
        tot.scale(alpha);
        m_run = m_new;
      }
      const float pa = sa == -INFINITY ? 0.f : exp2f(sa - m_run);
      const float pb = sb == -INFINITY ? 0.f : exp2f(sb - m_run);
      const float vn0 = ta < L ? __half2float(vnrm[rowbase + ta]) : 0.f;
      const float vn1 = tb < L ? __half2float(vnrm[rowbase + tb]) : 0.f;
      const float wA = pa * vn0, wB = pb * vn1;
      float ps = pa + pb;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) ps += __shfl_xor_sync(kFull, ps, o);
      l_run += ps;
      const float w0 = __shfl_sync(kFull, wA, src0);
      const float w1 = __shfl_sync(kFull, wA, src1);
      const float w8 = __shfl_sync(kFull, wB, src0);
      const float w9 = __shfl_sync(kFull, wB, src1);
      const uint32_t b0 = piece2(w0, w1, pc);
      const uint32_t b1 = piece2(w8, w9, pc);
      // this thread's 16 value coordinates of tokens 2c, 2c+1 (the first
      // k8 half of the tile), then of tokens 2c+8, 2c+9
#pragma unroll
      for (int hk = 0; hk < 2; ++hk) {
        float yv[2][16];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int64_t t = t0 + 2 * c + j + 8 * hk;
          uint32_t wsv[BV], w0v[BV], w6v[BV];
          if (t < L) {
            const uint32_t* r = vrec + (rowbase + t) * vcb.W;
#pragma unroll
            for (int p = 0; p < BV; ++p) {
              wsv[p] = __ldg(r + vs * BV + p);
              w0v[p] = __ldg(r + p);
              w6v[p] = __ldg(r + (1 + (vs >> 1)) * BV + p);
            }
            const float rho5 = subtree_radius<BV>(vtab, w0v, w6v, vs);
            decode_half<BV>(vtab, wsv, rho5, vh, yv[j]);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) yv[j][i] = 0.f;
          }
        }
        pv_pair(acc, yv, hk ? b1 : b0);
      }
      if (++chain == 2 * kPvFlushStages) {
        tot.flush(acc);
        chain = 0;
      }
    }
  }
  tot.flush(acc);
  const int nchunks = gridDim.x;
  float* part = partials + ((((size_t)b * Hkv + kvh) * nchunks + blockIdx.x) * kAttnWarps + warp) * partial_floats(128);
  float* ph = part + c * (2 + 128);
  if (g == 0) {
    ph[0] = m_run;
    ph[1] = l_run;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    ph[2 + 16 * g + 2 * mt] = tot.t[mt][0];
    ph[2 + 16 * g + 2 * mt + 1] = tot.t[mt][1];
  }
}

// Polar-mode decode attention with bulk-copy staging (capacity a multiple of
// 16): the key and value records and norms of each stage of kStageTiles
// tiles arrive by cp.async.bulk in a ring of kRing slots, so the tree decode
// reads shared memory instead of waiting on global loads.  Arithmetic as in
// k_attn_polar.
template <int BK, int BV>
__global__ void __launch_bounds__(128, 3) k_attn_polar_staged(const Dev kcb, const Dev vcb,
                                                           const uint8_t* __restrict__ kcache,
                                                           const uint8_t* __restrict__ vcache, int Hq, int Hkv,
                                                           int64_t capacity, int64_t cache_rows, const RowMap map,
                                                           const int32_t* __restrict__ seq_lens,
                                                           const uint8_t* __restrict__ prep, float scale_log2,
                                                           float* __restrict__ partials, int tiles_per_cta,
                                                           int* __restrict__ status) {
  constexpr int PK = BK + 1, PV = BV;
  constexpr int RBK = 16 * PK, RBV = 16 * PV;    // record bytes at d = 128
  constexpr int kSK = kStageTiles * 16 * RBK, kSKN = kStageTiles * 16 * 4;
  constexpr int kSV = kStageTiles * 16 * RBV, kSVN = kStageTiles * 16 * 2;
  constexpr int kSlot = kSK + kSKN + kSV + kSVN;
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ __align__(8) uint64_t bars[kRing];
  __shared__ PolarTab ktab, vtab;
  __shared__ uint2 sfrag[2 * 8 * 32];
  load_tab(kcb, ktab);
  load_tab(vcb, vtab);
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t tile0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t tcap = min(tile0 + tiles_per_cta, capacity / 16);
  const uint8_t* gkn = kcache + norm_offset(kcb, cache_rows);
  const uint8_t* gvn = vcache + norm_offset(vcb, cache_rows);
  // Stage st into ring slot st % kRing.  Every thread calls this and warp 0
  // issues the copies: one per array for a contiguous cache, one per array
  // and page touched for a paged one.
  auto request = [&](int st, int t_n) {
    const int slot = st % kRing;
    const uint32_t bar = su32(&bars[slot]);
    uint8_t* base = sm + (size_t)slot * kSlot;
    if (warp == 0) {
      if (lane == 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"((uint32_t)(t_n * 16 * (RBK + 4 + RBV + 2)))
                     : "memory");
      const int64_t t0 = (tile0 + (int64_t)st * kStageTiles) * 16;
      if (map.table == nullptr) {
        if (lane == 0) {
          const int64_t row = ((int64_t)b * Hkv + kvh) * capacity + t0;
          const uint32_t n = (uint32_t)(t_n * 16);
          bulk_g2s(su32(base), kcache + row * RBK, n * RBK, bar);
          bulk_g2s(su32(base + kSK), gkn + row * 4, n * 4, bar);
          bulk_g2s(su32(base + kSK + kSKN), vcache + row * RBV, n * RBV, bar);
          bulk_g2s(su32(base + kSK + kSKN + kSV), gvn + row * 2, n * 2, bar);
        }
      } else {
        // paged: lane 4r + a copies array a (key records, key norms, value
        // records, value norms) of the stage's run r (its tokens in one page),
        // so the runs' table lookups and copies are issued in parallel
        int k, cnt;
        int64_t row;
        if (page_run(map, b, kvh, Hkv, t0, t_n * 16, lane >> 2, status, k, cnt, row)) {
          const int a = lane & 3;
          const int rb = a == 0 ? RBK : a == 1 ? 4 : a == 2 ? RBV : 2;
          const int off = a == 0 ? 0 : a == 1 ? kSK : a == 2 ? kSK + kSKN : kSK + kSKN + kSV;
          const uint8_t* g = a == 0 ? kcache : a == 1 ? gkn : a == 2 ? vcache : gvn;
          bulk_g2s(su32(base + off + k * rb), g + row * rb, (uint32_t)(cnt * rb), bar);
        }
      }
    }
  };
  if (tid == 0) {
    for (int k = 0; k < kRing; ++k) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bars[k])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const int64_t L = seq_lens[b];
  const int L32 = (int)L;                    // token positions in 32 bits (capacity < 2^31)
  const int64_t tend = min(tcap, (L + 15) / 16);
  const int nt = tend > tile0 ? (int)(tend - tile0) : 0;
  const int nst = (nt + kStageTiles - 1) / kStageTiles;
  for (int st = 0; st < min(nst, kRing); ++st) request(st, min(kStageTiles, nt - st * kStageTiles));
  int issued = min(nst, kRing);
  const uint8_t* blk = prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(128);
  load_frags(blk, sfrag);
  const float* hdr = reinterpret_cast<const float*>(blk);
  const float S1 = hdr[c], S2 = hdr[4 + c], K2 = hdr[12 + c];
  __syncthreads();                           // tables and barriers ready

  float m_run = -INFINITY, l_run = 0.f;
  float acc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
  PvTotal tot;
  tot.zero();
  const float kq = kcb.qjl_const;
  const int hh = g >> 1, pc = g & 1;
  const int src0 = (2 * c) * 4 + hh, src1 = (2 * c + 1) * 4 + hh;
  const int vs = g >> 1, vh = g & 1;   // value subtree and half of this thread's 16 coordinates
  bool ok = true;
  int pending_from = 0;
  for (int st = 0; st < nst; ++st) {
    const int slot = st % kRing;
    if (!__syncthreads_and(bar_wait(su32(&bars[slot]), (uint32_t)((st / kRing) & 1), st == 0 ? kcb.first_wait : kWaitLimit))) {
      ok = false;
      pending_from = st;
      break;
    }
    const uint8_t* base = sm + (size_t)slot * kSlot;
    const uint32_t* skn = reinterpret_cast<const uint32_t*>(base + kSK);
    const uint8_t* sv = base + kSK + kSKN;
    const __half* svn = reinterpret_cast<const __half*>(base + kSK + kSKN + kSV);
    const int t_a = st * kStageTiles, n_here = min(kStageTiles, nt - t_a);
    for (int lt = warp; lt < n_here; lt += 4) {
      const int t0 = ((int)tile0 + t_a + lt) * 16;
      const int ta = t0 + g, tb = ta + 8;
      PKey<BK> ka, kb_;
      ka.load_row(reinterpret_cast<const uint32_t*>(base + ((size_t)lt * 16 + g) * RBK), skn[lt * 16 + g], c, ta < L32);
      kb_.load_row(reinterpret_cast<const uint32_t*>(base + ((size_t)lt * 16 + g + 8) * RBK), skn[lt * 16 + g + 8], c,
                   tb < L32);
      float s1a, s1b, s2a, s2b;
      polar_qk<BK>(ktab, sfrag, lane, ka, kb_, c, s1a, s1b, s2a, s2b);
      const float sa = ta < L32 ? est_polar(ka.nrm, S1 * s1a, fmaf(S2, s2a, K2), kq) * scale_log2 : -INFINITY;
      const float sb = tb < L32 ? est_polar(kb_.nrm, S1 * s1b, fmaf(S2, s2b, K2), kq) * scale_log2 : -INFINITY;
      float mx = fmaxf(sa, sb);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      if (__any_sync(kFull, mx > m_run)) {
        const float m_new = fmaxf(m_run, mx);
        const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
        l_run *= alpha;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mt][e] *= alpha;
        tot.scale(alpha);
        m_run = m_new;
      }
      const float pa = sa == -INFINITY ? 0.f : exp2f(sa - m_run);
      const float pb = sb == -INFINITY ? 0.f : exp2f(sb - m_run);
      const float vn0 = ta < L32 ? __half2float(svn[lt * 16 + g]) : 0.f;
      const float vn1 = tb < L32 ? __half2float(svn[lt * 16 + g + 8]) : 0.f;
      const float wA = pa * vn0, wB = pb * vn1;
      float ps = pa + pb;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) ps += __shfl_xor_sync(kFull, ps, o);
      l_run += ps;
      const float w0 = __shfl_sync(kFull, wA, src0);
      const float w1 = __shfl_sync(kFull, wA, src1);
      const float w8 = __shfl_sync(kFull, wB, src0);
      const float w9 = __shfl_sync(kFull, wB, src1);
      const uint32_t b0 = piece2(w0, w1, pc);
      const uint32_t b1 = piece2(w8, w9, pc);
      // this thread's 16 value coordinates of tokens 2c, 2c+1 (the first
      // k8 half of the tile), then of tokens 2c+8, 2c+9
#pragma unroll
      for (int hk = 0; hk < 2; ++hk) {
        float yv[2][16];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int tok = 2 * c + j + 8 * hk;
          if (t0 + tok < L32) {
            const uint32_t* r = reinterpret_cast<const uint32_t*>(sv + ((size_t)lt * 16 + tok) * RBV);
            uint32_t wsv[BV], w0v[BV], w6v[BV];
#pragma unroll
            for (int p = 0; p < BV; ++p) {
              wsv[p] = r[vs * BV + p];
              w0v[p] = r[p];
              w6v[p] = r[(1 + (vs >> 1)) * BV + p];
            }
            const float rho5 = subtree_radius<BV>(vtab, w0v, w6v, vs);
            decode_half<BV>(vtab, wsv, rho5, vh, yv[j]);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) yv[j][i] = 0.f;
          }
        }
        pv_pair(acc, yv, hk ? b1 : b0);
      }
    }
    if (st % kPvFlushStages == kPvFlushStages - 1) tot.flush(acc);
    if (st + kRing < nst) {
      __syncthreads();
      request(st + kRing, min(kStageTiles, nt - (st + kRing) * kStageTiles));
      issued = st + kRing + 1;
    }
  }
  if (!ok) {
    if (tid == 0) atomicOr(status, 2);
    for (int st = pending_from; st < issued; ++st) bar_wait(su32(&bars[st % kRing]), (uint32_t)((st / kRing) & 1));
  }
  tot.flush(acc);
  const int nchunks = gridDim.x;
  float* part = partials + ((((size_t)b * Hkv + kvh) * nchunks + blockIdx.x) * kAttnWarps + warp) * partial_floats(128);
  float* ph = part + c * (2 + 128);
  if (g == 0) {
    ph[0] = m_run;
    ph[1] = l_run;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    ph[2 + 16 * g + 2 * mt] = tot.t[mt][0];
    ph[2 + 16 * g + 2 * mt + 1] = tot.t[mt][1];
  }
}

template <int BK, int BV>
static cudaError_t attn_polar_staged_t(dim3 grid, cudaStream_t s, const Dev& k, const Dev& v, const uint8_t* kc,
                                       const uint8_t* vc, int Hq, int Hkv, int64_t cap, int64_t rows,
                                       const RowMap& map, const int32_t* sl, const uint8_t* prep, float sl2, float* parts, int tpc,
                                       int* status) {
  constexpr size_t smem = (size_t)kRing * kStageTiles * 16 * (16 * (BK + 1) + 4 + 16 * BV + 2);
  static cudaError_t configured = cudaFuncSetAttribute(k_attn_polar_staged<BK, BV>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (configured != cudaSuccess) return configured;
  k_attn_polar_staged<BK, BV><<<grid, 128, smem, s>>>(k, v, kc, vc, Hq, Hkv, cap, rows, map, sl, prep, sl2, parts, tpc,
                                                      status);
  return cudaGetLastError();
}

template <int BK>
static cudaError_t attn_polar_staged_v(int bv, dim3 grid, cudaStream_t s, const Dev& k, const Dev& v,
                                       const uint8_t* kc, const uint8_t* vc, int Hq, int Hkv, int64_t cap,
                                       int64_t rows, const RowMap& map, const int32_t* sl, const uint8_t* prep, float sl2,
                                       float* parts, int tpc, int* status) {
  switch (bv) {
    case 1: return attn_polar_staged_t<BK, 1>(grid, s, k, v, kc, vc, Hq, Hkv, cap, rows, map, sl, prep, sl2, parts, tpc, status);
    case 2: return attn_polar_staged_t<BK, 2>(grid, s, k, v, kc, vc, Hq, Hkv, cap, rows, map, sl, prep, sl2, parts, tpc, status);
    case 3: return attn_polar_staged_t<BK, 3>(grid, s, k, v, kc, vc, Hq, Hkv, cap, rows, map, sl, prep, sl2, parts, tpc, status);
    default: return attn_polar_staged_t<BK, 4>(grid, s, k, v, kc, vc, Hq, Hkv, cap, rows, map, sl, prep, sl2, parts, tpc, status);
  }
}

cudaError_t launch_attn_polar_staged(const Dev& kcb, const Dev& vcb, const uint8_t* kc, const uint8_t* vc, int B,
                                     int Hq, int Hkv, int64_t capacity, int64_t rows, const RowMap& map,
                                     const int32_t* seq_lens, const uint8_t* prep, float scale_log2, float* parts,
                                     int nchunks, int tpc, int* status, cudaStream_t s) {
  const dim3 grid(nchunks, Hkv, B);
  switch (kcb.b1) {
    case 1: return attn_polar_staged_v<1>(vcb.b1, grid, s, kcb, vcb, kc, vc, Hq, Hkv, capacity, rows, map, seq_lens, prep, scale_log2, parts, tpc, status);
    case 2: return attn_polar_staged_v<2>(vcb.b1, grid, s, kcb, vcb, kc, vc, Hq, Hkv, capacity, rows, map, seq_lens, prep, scale_log2, parts, tpc, status);
    default: return attn_polar_staged_v<3>(vcb.b1, grid, s, kcb, vcb, kc, vc, Hq, Hkv, capacity, rows, map, seq_lens, prep, scale_log2, parts, tpc, status);
  }
}

cudaError_t launch_prep_polar(const Dev& cb, const float* q, int B, int Hq, int Hkv, uint8_t* prep, cudaStream_t s) {
  k_prep_polar<<<dim3(Hkv * 4, B), 512, 0, s>>>(cb, q, Hq, Hkv, prep);
  return cudaGetLastError();
}

cudaError_t launch_logits_polar(const Dev& cb, const uint8_t* kc, int B, int Hq, int Hkv, int64_t capacity,
                                int64_t rows, const RowMap& map, const int32_t* seq_lens, const uint8_t* prep,
                                float* logits, int nchunks, int tpc, int* status, cudaStream_t s) {
  const dim3 grid(nchunks, Hkv, B);
  switch (cb.b1) {
    case 1: k_logits_polar<1><<<grid, 128, 0, s>>>(cb, kc, Hq, Hkv, capacity, rows, map, seq_lens, prep, logits, tpc, status); break;
    case 2: k_logits_polar<2><<<grid, 128, 0, s>>>(cb, kc, Hq, Hkv, capacity, rows, map, seq_lens, prep, logits, tpc, status); break;
    default: k_logits_polar<3><<<grid, 128, 0, s>>>(cb, kc, Hq, Hkv, capacity, rows, map, seq_lens, prep, logits, tpc, status); break;
  }
  return cudaGetLastError();
}

template <int BK>
static void attn_polar_v(int bv, dim3 grid, cudaStream_t s, const Dev& k, const Dev& v, const uint8_t* kc,
                         const uint8_t* vc, int Hq, int Hkv, int64_t cap, int64_t rows, const int32_t* sl,
                         const uint8_t* prep, float sl2, float* parts, int tpc) {
  switch (bv) {
    case 1: k_attn_polar<BK, 1><<<grid, 128, 0, s>>>(k, v, kc, vc, Hq, Hkv, cap, rows, sl, prep, sl2, parts, tpc); break;
    case 2: k_attn_polar<BK, 2><<<grid, 128, 0, s>>>(k, v, kc, vc, Hq, Hkv, cap, rows, sl, prep, sl2, parts, tpc); break;
    case 3: k_attn_polar<BK, 3><<<grid, 128, 0, s>>>(k, v, kc, vc, Hq, Hkv, cap, rows, sl, prep, sl2, parts, tpc); break;
    default: k_attn_polar<BK, 4><<<grid, 128, 0, s>>>(k, v, kc, vc, Hq, Hkv, cap, rows, sl, prep, sl2, parts, tpc); break;
  }
}

cudaError_t launch_attn_polar(const Dev& kcb, const Dev& vcb, const uint8_t* kc, const uint8_t* vc, int B, int Hq,
                              int Hkv, int64_t capacity, int64_t rows, const int32_t* seq_lens, const uint8_t* prep,
                              float scale_log2, float* parts, int nchunks, int tpc, cudaStream_t s) {
  const dim3 grid(nchunks, Hkv, B);
  switch (kcb.b1) {
    case 1: attn_polar_v<1>(vcb.b1, grid, s, kcb, vcb, kc, vc, Hq, Hkv, capacity, rows, seq_lens, prep, scale_log2, parts, tpc); break;
    case 2: attn_polar_v<2>(vcb.b1, grid, s, kcb, vcb, kc, vc, Hq, Hkv, capacity, rows, seq_lens, prep, scale_log2, parts, tpc); break;
    default: attn_polar_v<3>(vcb.b1, grid, s, kcb, vcb, kc, vc, Hq, Hkv, capacity, rows, seq_lens, prep, scale_log2, parts, tpc); break;
  }
  return cudaGetLastError();
}

}  // namespace tq
