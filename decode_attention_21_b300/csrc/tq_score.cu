// Scoring of full-precision queries against the packed bit-plane cache:
// query preparation, attention logits, fused decode attention and the
// split-KV merge.
//
// Estimator ([cnyes] hao.cnyes.com "TurboQuant", 1 bit 掃尾; [xujun]
// note-189244, 第二步; [suzuke] 第三步 "approximation + residual correction"):
//   est(q, x) = n ( <q', yhat> + gamma sqrt(pi/2)/m <q'', sigma> ),
//   q' = Pi q, q'' = S q' (once per step).
//
// Both inner products are sums over +-1 patterns: sigma is one, and a
// symmetric 2^b'-cell scalar codebook is exactly a weighted sum of the odd
// XOR-products of its code planes, yhat = sum_v coef_v s_v with
// s_v = (-1)^(xor of the planes in subset v) = 1 - 2 b_v (a Walsh-Hadamard
// expansion of the centroid table).  So every score is a constant per query
// head plus masked sums  sum_{i : b_v(i) = 1} x_i  of a query-side vector x.
//
// Those masked sums run on the tensor cores (fp16 m16n8k16, fp32
// accumulation) with the packed bits as the operand: a bit at mantissa
// position p of a subnormal fp16 element is the exact value 2^(p - 24), so a
// packed word becomes operands with one AND per 2 coordinates and one shift
// per 4 bit positions; the factor 2^-p goes into the query side (keys) or into
// a per-row scale (values).
//   * QK: A = key bits (16 keys x 16 coordinates), B = -2 coef_v q' (or 2 q'')
//     times 2^(24 - p), split into fp16 hi + lo; the G <= 4 heads x (hi, lo)
//     fill the 8 columns.
//   * PV: A = value bits (16 coordinates x 16 tokens), B = -2 coef_v p_t n_v,t
//     split into fp16 hi + lo.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tq_internal.cuh"
#include "tq_mma.cuh"
#include "tq_stage.cuh"

namespace tq {

using namespace mma;
using namespace stage;

// ---------------------------------------------------------------------------
// Query preparation: one CTA per (kv head, head slot, sequence).  q' = Pi q,
// q'' = S q', the per-slot constants and the fp16 B fragments of the two
// query-side planes:
//   plane 0 (stage 1): q'_k * bit_factor / S1, shared by every virtual plane
//     (the kernels apply -2 coef_v S1 to each virtual plane's MMA sum);
//   plane 1 (QJL):     2 q''_k * bit_factor / S2.
//   header (floats): S1[4], S2[4], K1[4] = (sum coef) sum q', K2[4] = -sum q''
//   fragments: [plane][kb][lane] uint2, column 2*slot + piece (piece 0 = hi,
//   1 = lo).
// Element k = 2c + e (b0) / 2c + 8 + e (b1) of k-block kb is coordinate
// 32c + beta + 16e with beta = 2kb (b0) or 2kb + 1 (b1); its key bit sits in
// operand register beta, whose bit value 1 / bit_factor(beta) the query side
// absorbs.
// ---------------------------------------------------------------------------
//
// One cluster of 4 CTAs per (kv head, head slot, sequence): CTA r computes
// the 32 coordinates 32r .. 32r+31 (word column r), reading only that slice
// of Pi and S Pi, and the cluster combines the per-CTA maxima and sums
// through distributed shared memory.
// ---------------------------------------------------------------------------
namespace {
// Store v at the address of p in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ void cluster_st(float* p, uint32_t rank, float v) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
}  // namespace

__device__ __forceinline__ void prep_body(const Dev& cb, const float* __restrict__ q, int Hq, int Hkv,
                                          uint8_t* __restrict__ prep) {
  constexpr int d = 128;
  const int G = Hq / Hkv;
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  const int unit = blockIdx.x >> 2;               // kv head * 4 + slot
  const int kvh = unit >> 2, slot = unit & 3, b = blockIdx.y;
  const bool live = slot < G;
  __shared__ float sq[d], part[2][4][32], sv[2][32];
  // [source rank][max |q'|, max |2 q''|, sum q', sum q'', sum of q' over extended-codebook coordinates]
  __shared__ float red[4][5];
  const int tid = threadIdx.x;
  const int mat = tid >> 7, qt = (tid >> 5) & 3, o = tid & 31;
  // Pi^T (mat 0) or (S Pi)^T (mat 1): rows 32 qt .. 32 qt + 31, column 32 r + o;
  // these loads do not depend on q, so they are issued before waiting for it
  // (MSE-only keys have no sketch: the second matrix is absent and q'' = 0)
  const bool has_s = cb.kind == 0;
  const float* col = (mat == 0 ? cb.PiT : cb.SPT) + (size_t)(32 * qt) * d + 32 * r + o;
  float m[32];
  const uint64_t keep = l2_policy_evict_last();
#pragma unroll
  for (int j = 0; j < 32; ++j) m[j] = (mat == 0 || has_s) ? ld_table(col + (size_t)j * d, keep) : 0.f;
  if (tid < d) sq[tid] = live ? q[((size_t)b * Hq + kvh * G + slot) * d + tid] : 0.f;
  __syncthreads();
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) acc = fmaf(m[j], sq[32 * qt + j], acc);
  part[mat][qt][o] = acc;
  __syncthreads();
  if (tid < 64) {
    // warp 0: q'_{32r+o}; warp 1: q''_{32r+o}.  Local max |q'| (|2 q''|) and sum.
    const int mm = tid >> 5;
    const float v = (part[mm][0][o] + part[mm][1][o]) + (part[mm][2][o] + part[mm][3][o]);
    sv[mm][o] = v;
    float mx = mm == 0 ? fabsf(v) : 2.f * fabsf(v), sm = v;
#pragma unroll
    for (int k = 16; k; k >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, k));
      sm += __shfl_xor_sync(kFull, sm, k);
    }
    // push this CTA's partials into slot r of every cluster CTA (itself included)
    if (o < 4) {
      cluster_st(&red[r][mm], (uint32_t)o, mx);
      cluster_st(&red[r][2 + mm], (uint32_t)o, sm);
      if (mm == 0) cluster_st(&red[r][4], (uint32_t)o, (int)r < cb.extra / 32 ? sm : 0.f);
    }
  }
  cluster_sync();
  // every CTA combines the four partials in rank order (identical results)
  float mx1 = 0.f, mx2 = 0.f, sm1 = 0.f, sm2 = 0.f, sm1x = 0.f;
  // outlier-channel split: the sums of q' and q'' over each group's word
  // columns (group A: columns 0 .. extra/32 - 1)
  float ga1 = 0.f, ga2 = 0.f, gb1 = 0.f, gb2 = 0.f;
  for (int k = 0; k < 4; ++k) {
    mx1 = fmaxf(mx1, red[k][0]);
    mx2 = fmaxf(mx2, red[k][1]);
    sm1 += red[k][2];
    sm2 += red[k][3];
    sm1x += red[k][4];
    if (k < cb.extra / 32) {
      ga1 += red[k][2];
      ga2 += red[k][3];
    } else {
      gb1 += red[k][2];
      gb2 += red[k][3];
    }
  }
  const int nv = cb.nv;
  float csum = 0.f, csumx = 0.f;
  for (int v = 0; v < nv; ++v) csum += cb.vcoef[v];
  for (int u = 0; u < cb.nvx; ++u) csumx += cb.vcoef_x[u];
  // keep |B| <= 2^14 at the largest bit factor
  const float S1 = pow2_scale(mx1 * kMaxBitFactor, 16384.f), S2 = pow2_scale(mx2 * kMaxBitFactor, 16384.f);
  uint8_t* blk = prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(d);
  float* hdr = reinterpret_cast<float*>(blk);
  if (r == 0 && tid == 0) {
    hdr[slot] = live ? S1 : 0.f;
    hdr[4 + slot] = live ? S2 : 0.f;
    if (cb.split) {
      // group B's constants in K1, K2 and group A's in K1x, K2x
      hdr[8 + slot] = live ? csum * gb1 : 0.f;
      hdr[12 + slot] = live ? -gb2 : 0.f;
      hdr[16 + slot] = live ? csumx * ga1 : 0.f;
      hdr[20 + slot] = live ? -ga2 : 0.f;
    } else {
      hdr[8 + slot] = live ? fmaf(csumx - csum, sm1x, csum * sm1) : 0.f;
      hdr[12 + slot] = live ? -sm2 : 0.f;
      hdr[16 + slot] = 0.f;
      hdr[20 + slot] = 0.f;
    }
  }
  // fragments of this word column (c = r) for this slot's lanes g = 2 slot + piece
  uint2* frag = reinterpret_cast<uint2*>(blk + kPrepHeader);
  if (tid < 32) {
    const int pc = tid & 1, kb = (tid >> 1) & 7, v = tid >> 4;
    const int g = 2 * slot + pc;
    float vals[4] = {0.f, 0.f, 0.f, 0.f};
    if (live) {
      for (int t = 0; t < 4; ++t) {
        const int beta = 2 * kb + (t >> 1);
        const int k = beta + 16 * (t & 1);          // local coordinate (32 r + k)
        const float x = v == 0 ? sv[0][k] * bit_factor(beta) / S1 : 2.f * sv[1][k] * bit_factor(beta) / S2;
        vals[t] = piece16(x, pc);
      }
    }
    frag[(v * 8 + kb) * 32 + g * 4 + r] = make_uint2(pack_half2(vals[0], vals[1]), pack_half2(vals[2], vals[3]));
  }
  // One CTA waiting for the kernel before this grid is enough for the grid's
  // completion to imply that kernel's; the others leave now and free their
  // SMs for the scoring kernel.
  if (blockIdx.x == 0 && blockIdx.y == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

__global__ void __launch_bounds__(256) k_prep(const Dev cb, const float* __restrict__ q, int Hq, int Hkv,
                                              uint8_t* __restrict__ prep) {
  // This grid may run alongside the kernel before it (a cache append), since
  // it reads only the queries and the codebook; one of its CTAs waits for
  // that kernel at its end, so the grid's completion implies the append's.  The scoring kernel
  // that follows may start now: it touches no cache row before it waits for
  // this grid.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  prep_body(cb, q, Hq, Hkv, prep);
}

// One key row of a decode step's cache append (scalar mode, d = 128, no
// extra-bit words), by a CTA of 256 threads: thread (i, h) owns coordinate
// i and quarters 2h, 2h + 1 of each matrix-vector product.  The arithmetic
// and its order are those of the short-batch append kernel (quarters of 32
// terms, each an fma chain, summed pairwise; warp sums of squares; codes by
// compare-count), so the stored record and norms are bit-identical.  The
// stores wait for the kernel before this grid (griddepcontrol.wait).
__device__ __forceinline__ void append_body(const Dev& cb, uint8_t* __restrict__ cache, int64_t cache_rows,
                                            const void* __restrict__ x, int x_dtype, int64_t row, int d_in,
                                            const int64_t* __restrict__ dst_rows, int* __restrict__ status) {
  constexpr int D = 128, NW = D / 32;
  __shared__ float xs[D], part[4][D], red[NW];
  __shared__ uint32_t words[4 * NW];
  const int t = threadIdx.x, i = t & (D - 1), h = t >> 7;
  const int lane = i & 31, w = i >> 5;
  const int b1 = cb.b1, P = cb.P;
  const bool prod = cb.kind == 0;
  const uint64_t keep = l2_policy_evict_last();
  if (h == 0) {
    float v = 0.f;
    if (i < d_in)
      v = x_dtype == 0 ? static_cast<const float*>(x)[row * d_in + i]
                       : __bfloat162float(static_cast<const __nv_bfloat16*>(x)[row * d_in + i]);
    xs[i] = v;
  }
  __syncthreads();
  // quarter k of (M^T)[:, i] . xs: rows 32 k .. 32 k + 31 of column i
  auto quarter = [&](const float* MT, int k) {
    const float* col = MT + (size_t)(32 * k) * D + i;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) acc = fmaf(ld_table(col + (size_t)j * D, keep), xs[32 * k + j], acc);
    return acc;
  };
  part[2 * h][i] = quarter(cb.PiT, 2 * h);
  part[2 * h + 1][i] = quarter(cb.PiT, 2 * h + 1);
  __syncthreads();
  float y = 0.f, r = 0.f;
  if (h == 0) {
    y = (part[0][i] + part[1][i]) + (part[2][i] + part[3][i]);
    float ss = y * y;
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
    if (lane == 0) red[w] = ss;
  }
  __syncthreads();
  float nrm = 0.f;
  if (h == 0) {
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < NW; ++k) ss += red[k];
    nrm = sqrtf(ss);
    y *= nrm > 0.f ? 1.f / nrm : 0.f;
    int idx = 0;
    const int nbd = (1 << b1) - 1;
    for (int k = 0; k < nbd; ++k) idx += (y >= cb.bound[k]) ? 1 : 0;
    r = y - cb.cent[idx];
    for (int p = 0; p < b1; ++p) {
      const uint32_t bw = __ballot_sync(kFull, (idx >> (b1 - 1 - p)) & 1);
      if (lane == 0) words[w * P + p] = bw;
    }
  }
  __syncthreads();                         // everyone has read red and xs
  if (prod && h == 0) {
    xs[i] = r;
    float ss = r * r;
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
    if (lane == 0) red[w] = ss;
  }
  __syncthreads();
  float gamma = 0.f;
  if (prod) {
    part[2 * h][i] = quarter(cb.ST, 2 * h);
    part[2 * h + 1][i] = quarter(cb.ST, 2 * h + 1);
    __syncthreads();
    if (h == 0) {
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < NW; ++k) ss += red[k];
      gamma = sqrtf(ss);
      const float z = (part[0][i] + part[1][i]) + (part[2][i] + part[3][i]);
      const uint32_t bw = __ballot_sync(kFull, z >= 0.f);
      if (lane == 0) words[w * P + b1] = bw;
    }
  }
  __syncthreads();
  // the kernel before this grid (a scoring kernel reading this cache) has
  // completed before any destination is looked up or written
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t dst = dst_rows ? dst_rows[row] : row;
  if (dst < 0 || dst >= cache_rows) {
    if (t == 0) atomicOr(status, kBadRow);
    return;
  }
  uint32_t* rec = reinterpret_cast<uint32_t*>(cache) + dst * cb.W;
  if (t < cb.W) rec[t] = words[t];
  if (t == 0) {
    unsigned char* norms = cache + norm_offset(cb, cache_rows);
    if (prod)
      reinterpret_cast<__half2*>(norms)[dst] = __floats2half2_rn(nrm, gamma);
    else
      reinterpret_cast<__half*>(norms)[dst] = __float2half_rn(nrm);
  }
}

// A decode step's query prep and key append in one grid: blocks
// 0 .. 16 Hkv - 1 of each grid row are the prep's (4-CTA clusters), blocks
// 16 Hkv + k of grid row 0 append row k of x (k < n).  One launch instead of
// two saves one grid-completion handoff on the step's critical path; the
// append CTAs wait for the kernel before this grid before they store.
__global__ void __launch_bounds__(256) k_prep_append(const Dev cb, const float* __restrict__ q, int Hq, int Hkv,
                                                     uint8_t* __restrict__ prep, uint8_t* __restrict__ cache,
                                                     int64_t cache_rows, const void* __restrict__ x, int x_dtype,
                                                     int64_t n, int d_in, const int64_t* __restrict__ dst_rows,
                                                     int* __restrict__ status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int nprep = Hkv * 16;
  if ((int)blockIdx.x < nprep) {
    prep_body(cb, q, Hq, Hkv, prep);
    return;
  }
  const int64_t row = (int64_t)blockIdx.x - nprep;
  if (blockIdx.y != 0 || row >= n) return;
  append_body(cb, cache, cache_rows, x, x_dtype, row, d_in, dst_rows, status);
}

// ---------------------------------------------------------------------------
// QK for T 16-key tiles at once: thread (g, c) gets the inner products of
// keys g and g+8 of each tile for head slot c.  The stage-1 virtual planes
// (odd XOR-products of the code planes) share the query operand and keep one
// accumulator each; the coefficients -2 coef_v S1 are applied to the sums.
// ---------------------------------------------------------------------------
template <int NV, int P, bool QJL = true>
struct QK16 {
  static constexpr int C1 = NV == 1 ? 2 : 1;   // accumulator chains per virtual plane
  static constexpr int PS = QJL ? P - 1 : P;   // stage-1 code planes (the QJL sign plane is last)
  static constexpr int NQ = QJL ? 1 : 0;
  uint2 bq[1 + NQ][8];
  float S2, K1, K2, K1x, K2x;
  float cv[NV];
  float cvx[2 * NV];   // coefficients of the extended (mixed-bit) codebook's planes
  int c_;

  __device__ __forceinline__ void load(const uint8_t* blk, int lane, const Dev& cb) {
    const float* hdr = reinterpret_cast<const float*>(blk);
    const uint2* frag = reinterpret_cast<const uint2*>(blk + kPrepHeader);
#pragma unroll
    for (int v = 0; v <= NQ; ++v)
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) bq[v][kb] = frag[(v * 8 + kb) * 32 + lane];
    const int c = lane & 3;
    const float S1 = hdr[c];
    S2 = hdr[4 + c];
    K1 = hdr[8 + c];
    K2 = hdr[12 + c];
    K1x = hdr[16 + c];
    K2x = hdr[20 + c];
#pragma unroll
    for (int v = 0; v < NV; ++v) cv[v] = -2.f * cb.vcoef[v] * S1;
#pragma unroll
    for (int u = 0; u < 2 * NV; ++u) cvx[u] = -2.f * cb.vcoef_x[u] * S1;
    c_ = c;
  }

  // wa[t], wb[t]: the P plane words (column c) of keys g and g+8 of tile t.
  // s1[t][0/1], s2[t][0/1]: stage-1 and QJL inner products of keys g, g+8
  // (s2 = 0 without the QJL plane).
  template <int T>
  __device__ __forceinline__ void score(const uint32_t (&wa)[T][P], const uint32_t (&wb)[T][P], float (&s1)[T][2],
                                        float (&s2)[T][2]) const {
    uint32_t z[T];
#pragma unroll
    for (int t = 0; t < T; ++t) z[t] = 0u;
    score_mixed<T, 0>(wa, wb, z, z, s1, s2);
  }

  // Mixed-bit keys: the first EXT word columns (32 EXT coordinates) use the
  // (b' + 1)-bit codebook, whose low bit is the extra word ea/eb of the
  // column.  Lanes of those columns feed the 2 NV extended virtual planes and
  // zeros to the main ones; the other lanes do the opposite.
  template <int T, int EXT>
  __device__ __forceinline__ void score_mixed(const uint32_t (&wa)[T][P], const uint32_t (&wb)[T][P],
                                              const uint32_t (&ea)[T], const uint32_t (&eb)[T], float (&s1)[T][2],
                                              float (&s2)[T][2]) const {
    float s1x[T][2], s2x[T][2];
    score_groups<T, EXT, false>(wa, wb, ea, eb, s1, s2, s1x, s2x);
  }

  // SPLIT (outlier-channel split keys): the extended columns are group A,
  // with its own norms, so its stage-1 and QJL sums come out separately
  // (s1x, s2x) and s1, s2 hold group B's; group A's sign plane gets its own
  // accumulator (lanes of the other group feed it zeros).
  template <int T, int EXT, bool SPLIT>
  __device__ __forceinline__ void score_groups(const uint32_t (&wa)[T][P], const uint32_t (&wb)[T][P],
                                               const uint32_t (&ea)[T], const uint32_t (&eb)[T], float (&s1)[T][2],
                                               float (&s2)[T][2], float (&s1x)[T][2], float (&s2x)[T][2]) const {
    static_assert(!SPLIT || (QJL && EXT > 0), "a split key has the QJL plane and extended columns");
    constexpr int NX = EXT ? 2 * NV : 0;
    const bool xl = EXT > 0 && c_ < EXT;
    float a1[T][NV][C1][4], a2[T][2][4], ax[T][NX > 0 ? NX : 1][4], a2x[T][SPLIT ? 2 : 1][4];
    uint32_t qxa[T], qxb[T], qya[T], qyb[T];    // group A's sign-plane operands (SPLIT)
    uint32_t xa[T][NV + NQ], xb[T][NV + NQ], ya[T][NV + NQ], yb[T][NV + NQ];
    uint32_t za[T][NX > 0 ? NX : 1], zb[T][NX > 0 ? NX : 1], wza[T][NX > 0 ? NX : 1], wzb[T][NX > 0 ? NX : 1];
#pragma unroll
    for (int t = 0; t < T; ++t) {
#pragma unroll
      for (int u = 0; u < NX; ++u) {
        uint32_t pa = 0, pb = 0;
#pragma unroll
        for (int p = 0; p < PS; ++p)
          if (kOddMask[u] >> p & 1u) {
            pa ^= wa[t][p];
            pb ^= wb[t][p];
          }
        if (kOddMask[u] >> PS & 1u) {
          pa ^= ea[t];
          pb ^= eb[t];
        }
        za[t][u] = xl ? pa : 0u;
        zb[t][u] = xl ? pb : 0u;
        wza[t][u] = za[t][u] >> 4;
        wzb[t][u] = zb[t][u] >> 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) ax[t][u][e] = 0.f;
      }
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        uint32_t pa = 0, pb = 0;
#pragma unroll
        for (int p = 0; p < PS; ++p)
          if (kOddMask[v] >> p & 1u) {
            pa ^= wa[t][p];
            pb ^= wb[t][p];
          }
        xa[t][v] = xl ? 0u : pa;
        xb[t][v] = xl ? 0u : pb;
#pragma unroll
        for (int ch = 0; ch < C1; ++ch)
#pragma unroll
          for (int e = 0; e < 4; ++e) a1[t][v][ch][e] = 0.f;
      }
      if constexpr (QJL) {
        xa[t][NV] = (SPLIT && xl) ? 0u : wa[t][P - 1];
        xb[t][NV] = (SPLIT && xl) ? 0u : wb[t][P - 1];
      }
      if constexpr (SPLIT) {
        qxa[t] = xl ? wa[t][P - 1] : 0u;
        qxb[t] = xl ? wb[t][P - 1] : 0u;
        qya[t] = qxa[t] >> 4;
        qyb[t] = qxb[t] >> 4;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int e = 0; e < 4; ++e) a2x[t][ch][e] = 0.f;
      }
#pragma unroll
      for (int v = 0; v < NV + NQ; ++v) {
        ya[t][v] = xa[t][v] >> 4;
        yb[t][v] = xb[t][v] >> 4;
      }
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int e = 0; e < 4; ++e) a2[t][ch][e] = 0.f;
    }
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      const int b0 = 2 * kb, b1 = 2 * kb + 1;
#pragma unroll
      for (int t = 0; t < T; ++t) {
        if constexpr (QJL)
          mma_f16(a2[t][kb & 1], bit_operand(xa[t][NV], ya[t][NV], b0), bit_operand(xb[t][NV], yb[t][NV], b0),
                  bit_operand(xa[t][NV], ya[t][NV], b1), bit_operand(xb[t][NV], yb[t][NV], b1), bq[NQ][kb].x,
                  bq[NQ][kb].y);
        if constexpr (SPLIT)
          mma_f16(a2x[t][kb & 1], bit_operand(qxa[t], qya[t], b0), bit_operand(qxb[t], qyb[t], b0),
                  bit_operand(qxa[t], qya[t], b1), bit_operand(qxb[t], qyb[t], b1), bq[NQ][kb].x, bq[NQ][kb].y);
#pragma unroll
        for (int v = 0; v < NV; ++v)
          mma_f16(a1[t][v][kb % C1], bit_operand(xa[t][v], ya[t][v], b0), bit_operand(xb[t][v], yb[t][v], b0),
                  bit_operand(xa[t][v], ya[t][v], b1), bit_operand(xb[t][v], yb[t][v], b1), bq[0][kb].x,
                  bq[0][kb].y);
#pragma unroll
        for (int u = 0; u < NX; ++u)
          mma_f16(ax[t][u], bit_operand(za[t][u], wza[t][u], b0), bit_operand(zb[t][u], wzb[t][u], b0),
                  bit_operand(za[t][u], wza[t][u], b1), bit_operand(zb[t][u], wzb[t][u], b1), bq[0][kb].x,
                  bq[0][kb].y);
      }
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float ra = K1, rb = K1;
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int ch = 0; ch < C1; ++ch) {
          ra = fmaf(cv[v], a1[t][v][ch][0] + a1[t][v][ch][1], ra);
          rb = fmaf(cv[v], a1[t][v][ch][2] + a1[t][v][ch][3], rb);
        }
      float xa_ = SPLIT ? K1x : 0.f, xb_ = SPLIT ? K1x : 0.f;
#pragma unroll
      for (int u = 0; u < NX; ++u) {
        if constexpr (SPLIT) {
          xa_ = fmaf(cvx[u], ax[t][u][0] + ax[t][u][1], xa_);
          xb_ = fmaf(cvx[u], ax[t][u][2] + ax[t][u][3], xb_);
        } else {
          ra = fmaf(cvx[u], ax[t][u][0] + ax[t][u][1], ra);
          rb = fmaf(cvx[u], ax[t][u][2] + ax[t][u][3], rb);
        }
      }
      s1[t][0] = ra;
      s1[t][1] = rb;
      if constexpr (QJL) {
        s2[t][0] = fmaf(S2, (a2[t][0][0] + a2[t][0][1]) + (a2[t][1][0] + a2[t][1][1]), K2);
        s2[t][1] = fmaf(S2, (a2[t][0][2] + a2[t][0][3]) + (a2[t][1][2] + a2[t][1][3]), K2);
      } else {
        s2[t][0] = s2[t][1] = 0.f;
      }
      if constexpr (SPLIT) {
        s1x[t][0] = xa_;
        s1x[t][1] = xb_;
        s2x[t][0] = fmaf(S2, (a2x[t][0][0] + a2x[t][0][1]) + (a2x[t][1][0] + a2x[t][1][1]), K2x);
        s2x[t][1] = fmaf(S2, (a2x[t][0][2] + a2x[t][0][3]) + (a2x[t][1][2] + a2x[t][1][3]), K2x);
      }
    }
  }
};

// The P plane words of word column c of a record.  Vector loads need the
// record start aligned to 4 P bytes (records of exactly 4 P words); records
// with extra-bit words (VEC = false) are read word by word.
template <int P, bool VEC = true>
__device__ __forceinline__ void load_words(const uint32_t* __restrict__ rec, int c, uint32_t (&w)[P]) {
  const uint32_t* p = rec + c * P;
  if constexpr (VEC && P == 4) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (VEC && P == 2) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < P; ++i) w[i] = __ldg(p + i);
  }
}

// Key words and norms of one 16-key tile for thread (g, c).  The norm entry
// is 4 bytes (n, gamma) with the QJL term, 2 bytes (n) without.
template <int P, bool QJL = true, int EXT = 0, bool SPLIT = false>
struct KTile {
  uint32_t wa[P], wb[P];
  uint32_t ea = 0, eb = 0;   // extra-bit words (word columns < EXT of mixed-bit keys)
  uint32_t na, nb;           // norm entries (a split's group B: n_B, gamma_B)
  uint32_t nxa = 0, nxb = 0; // a split's group A: n_A, gamma_A
  __device__ __forceinline__ static uint32_t norm_at(const uint32_t* nrm, int64_t row) {
    if constexpr (SPLIT) return __ldg(nrm + 2 * row + 1);
    else if constexpr (QJL) return __ldg(nrm + row);
    else return (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(nrm) + row);
  }
  __device__ __forceinline__ void load(const uint32_t* recs, const uint32_t* nrm, int W, int64_t rowbase, int64_t ta,
                                       int64_t L, int c) {
    const int64_t tb = ta + 8;
    if (ta < L) {
      load_words<P, EXT == 0>(recs + (rowbase + ta) * W, c, wa);
      if (EXT && c < EXT) ea = __ldg(recs + (rowbase + ta) * W + 4 * P + c);
      na = norm_at(nrm, rowbase + ta);
      if (SPLIT) nxa = __ldg(nrm + 2 * (rowbase + ta));
    } else {
#pragma unroll
      for (int p = 0; p < P; ++p) wa[p] = 0;
      na = 0;
    }
    if (tb < L) {
      load_words<P, EXT == 0>(recs + (rowbase + tb) * W, c, wb);
      if (EXT && c < EXT) eb = __ldg(recs + (rowbase + tb) * W + 4 * P + c);
      nb = norm_at(nrm, rowbase + tb);
      if (SPLIT) nxb = __ldg(nrm + 2 * (rowbase + tb));
    } else {
#pragma unroll
      for (int p = 0; p < P; ++p) wb[p] = 0;
      nb = 0;
    }
  }
};

// Estimate from the norm entry: fp16 (n, gamma) for keys with the QJL term,
// fp16 n (low half) for MSE-only keys.
template <bool QJL>
__device__ __forceinline__ float est_key(uint32_t nrm_bits, float s1, float s2, float kq);

__device__ __forceinline__ float est_from(uint32_t nrm_bits, float s1, float s2, float kq) {
  const __half2 h = *reinterpret_cast<const __half2*>(&nrm_bits);
  return __low2float(h) * fmaf(__high2float(h) * kq, s2, s1);
}

template <bool QJL>
__device__ __forceinline__ float est_key(uint32_t nrm_bits, float s1, float s2, float kq) {
  if constexpr (QJL) {
    return est_from(nrm_bits, s1, s2, kq);
  } else {
    return __half2float(__ushort_as_half((unsigned short)(nrm_bits & 0xffffu))) * s1;
  }
}

// Outlier-channel split key: group A's estimate (n_A, gamma_A in nx; sums
// s1x, s2x; QJL constant kqx) plus group B's (n_B, gamma_B in n).
template <bool QJL, bool SPLIT>
__device__ __forceinline__ float est_groups(uint32_t nx, uint32_t n, float s1x, float s2x, float s1, float s2,
                                            float kqx, float kq) {
  if constexpr (SPLIT) return est_from(nx, s1x, s2x, kqx) + est_from(n, s1, s2, kq);
  else return est_key<QJL>(n, s1, s2, kq);
}

// ---------------------------------------------------------------------------
// Logits: grid (chunks, Hkv, B), 4 warps; each warp scores 16-key tiles,
// prefetching its next tile while scoring the current one.
// ---------------------------------------------------------------------------
template <int NV, int P, bool QJL, int EXT, bool SPLIT = false>
__global__ void __launch_bounds__(128, 4) k_logits(const Dev cb, const uint8_t* __restrict__ kcache, int Hq, int Hkv,
                                                int64_t capacity, int64_t cache_rows,
                                                const int32_t* __restrict__ seq_lens,
                                                const uint8_t* __restrict__ prep, float* __restrict__ logits,
                                                int tiles_per_cta) {
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int G = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t L = seq_lens[b];
  const int64_t ntiles = (L + 15) / 16;
  const int64_t tile0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t tend = min(tile0 + tiles_per_cta, ntiles);
  if (tile0 + warp >= tend) return;
  QK16<NV, P, QJL> qk;
  qk.load(prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(128), lane, cb);
  const uint32_t* recs = reinterpret_cast<const uint32_t*>(kcache);
  const uint32_t* nrm = reinterpret_cast<const uint32_t*>(kcache + norm_offset(cb, cache_rows));
  const int64_t rowbase = ((int64_t)b * Hkv + kvh) * capacity;
  const float kq = cb.qjl_const, kqx = cb.qjl_const_x;
  const int W = cb.W;
  float* out = logits + ((size_t)b * Hq + (size_t)kvh * G + c) * capacity;
  KTile<P, QJL, EXT, SPLIT> cur, nxt;
  int64_t tile = tile0 + warp;
  cur.load(recs, nrm, W, rowbase, tile * 16 + g, L, c);
  for (; tile < tend; tile += 4) {
    const int64_t tn = tile + 4;
    if (tn < tend) nxt.load(recs, nrm, W, rowbase, tn * 16 + g, L, c);
    uint32_t wa[1][P], wb[1][P];
#pragma unroll
    for (int p = 0; p < P; ++p) {
      wa[0][p] = cur.wa[p];
      wb[0][p] = cur.wb[p];
    }
    float s1[1][2], s2[1][2], s1x[1][2], s2x[1][2];
    const uint32_t ea[1] = {cur.ea}, eb[1] = {cur.eb};
    qk.template score_groups<1, EXT, SPLIT>(wa, wb, ea, eb, s1, s2, s1x, s2x);
    const int64_t ta = tile * 16 + g, tb = ta + 8;
    if (c < G) {
      if (ta < L) out[ta] = est_groups<QJL, SPLIT>(cur.nxa, cur.na, s1x[0][0], s2x[0][0], s1[0][0], s2[0][0], kqx, kq);
      if (tb < L) out[tb] = est_groups<QJL, SPLIT>(cur.nxb, cur.nb, s1x[0][1], s2x[0][1], s1[0][1], s2[0][1], kqx, kq);
    }
    cur = nxt;
  }
}

// ---------------------------------------------------------------------------
// Logits with bulk-copy staging (capacity a multiple of 16), launched as the
// programmatic dependent of the query prep.  Grid (chunks, Hkv, B); each CTA
//   * sets up a ring of kRing stages of kStageTiles tiles (one mbarrier per
//     stage) while the prep runs, then waits for the prep grid;
//   * requests the first stage of its chunk's key records and norms
//     (cp.async.bulk), loads the query fragments while only that stage is in
//     flight (a whole chunk in flight would queue these small loads behind
//     it), then requests the next stages;
//   * scores its tiles as the stages land, refilling each ring slot once all
//     warps are done with it.
// Every wait is bounded; on a timeout the CTA records an error, waits
// (bounded) for its copies in flight and returns.
// ---------------------------------------------------------------------------

template <int NV, int P, bool QJL, int EXT, bool SPLIT = false>
__global__ void __launch_bounds__(128, 4) k_logits_staged(const Dev cb, const uint8_t* __restrict__ kcache, int Hq,
                                                       int Hkv, int64_t capacity, int64_t cache_rows,
                                                       const RowMap map, const int32_t* __restrict__ seq_lens,
                                                       const uint8_t* __restrict__ prep, float* __restrict__ logits,
                                                       int tiles_per_cta, int* __restrict__ status) {
  constexpr int RB = 16 * P + 4 * EXT;       // record bytes at d = 128 (+ extra-bit words)
  constexpr int NB = SPLIT ? 8 : QJL ? 4 : 2;  // norm entry bytes
  constexpr int kPairs = NV <= 4 && EXT == 0;  // two tiles per warp step (registers permitting)
  constexpr int kStageRec = kStageTiles * 16 * RB, kStageNrm = kStageTiles * 16 * NB;
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ __align__(8) uint64_t bars[kRing];
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int G = Hq / Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  uint8_t* srec = sm;
  uint8_t* snrm = sm + (size_t)kRing * kStageRec;
  // ---- chunk bounds
  const int64_t tile0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t tcap = min(tile0 + tiles_per_cta, capacity / 16);
  if (tile0 >= tcap) return;
  const uint8_t* gnrm = kcache + norm_offset(cb, cache_rows);
  // Stage st (tiles st*kStageTiles ..) into ring slot st % kRing; every
  // thread calls this and warp 0 issues the copies: one per array for a
  // contiguous cache, one per array and page touched for a paged one.
  auto request = [&](int st, int t_n) {
    const int slot = st % kRing;
    const uint32_t bar = su32(&bars[slot]);
    if (warp == 0) {
      if (lane == 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"((uint32_t)(t_n * 16 * (RB + NB)))
                     : "memory");
      const int64_t t0 = (tile0 + (int64_t)st * kStageTiles) * 16;
      if (map.table == nullptr) {
        if (lane == 0) {
          const int64_t row = ((int64_t)b * Hkv + kvh) * capacity + t0;
          bulk_g2s(su32(srec + (size_t)slot * kStageRec), kcache + row * RB, (uint32_t)(t_n * 16 * RB), bar);
          bulk_g2s(su32(snrm + (size_t)slot * kStageNrm), gnrm + row * NB, (uint32_t)(t_n * 16 * NB), bar);
        }
      } else {
        // paged: lane 2r + a copies array a (records, norms) of the stage's
        // run r (its tokens in one page), so the runs' table lookups and
        // copies are issued in parallel
        int k, cnt;
        int64_t row;
        if (lane < 2 * kStageTiles && page_run(map, b, kvh, Hkv, t0, t_n * 16, lane >> 1, status, k, cnt, row)) {
          if (lane & 1)
            bulk_g2s(su32(snrm + (size_t)slot * kStageNrm + (size_t)k * NB), gnrm + row * NB, (uint32_t)(cnt * NB), bar);
          else
            bulk_g2s(su32(srec + (size_t)slot * kStageRec + (size_t)k * RB), kcache + row * RB, (uint32_t)(cnt * RB), bar);
        }
      }
    }
  };
  if (tid == 0) {
    for (int k = 0; k < kRing; ++k) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bars[k])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const int64_t L = seq_lens[b];
  const int64_t tend = min(tcap, (L + 15) / 16);
  const int nt = tend > tile0 ? (int)(tend - tile0) : 0;
  const int nst = (nt + kStageTiles - 1) / kStageTiles;
  // Stream the first kPrefetchStages stages of the chunk from HBM into L2
  // while the prep (and any cache append before it) still runs.
  if (warp == 0)
    for (int st = 0; st < min(nst, kPrefetchStages); ++st) {
      const int64_t t0 = (tile0 + (int64_t)st * kStageTiles) * 16;
      const int n = min(kStageTiles, nt - st * kStageTiles) * 16;
      int k = 0, cnt = n;
      int64_t row = ((int64_t)b * Hkv + kvh) * capacity + t0;
      if (map.table ? (lane < 2 * kStageTiles && page_run(map, b, kvh, Hkv, t0, n, lane >> 1, status, k, cnt, row))
                    : lane < 2) {
        if (lane & 1)
          prefetch_l2(gnrm + row * NB, (uint32_t)(cnt * NB));
        else
          prefetch_l2(kcache + row * RB, (uint32_t)(cnt * RB));
      }
    }
  // The query fragments come from the preceding prep grid, launched as its
  // programmatic dependent; the prep's completion also implies that of any
  // cache append before it, so no cache row is read into the SM before this
  // wait.  The first stage goes out right after it, the fragment loads queue
  // behind only that stage, and the other stages follow.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (nst > 0) request(0, min(kStageTiles, nt));
  QK16<NV, P, QJL> qk;
  qk.load(prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(128), lane, cb);
  __syncthreads();                           // the barriers are initialised; the fragments are in
  for (int st = 1; st < min(nst, kRing); ++st) request(st, min(kStageTiles, nt - st * kStageTiles));
  int issued = min(nst, kRing);              // stages requested so far
  // ---- scoring
  const float kq = cb.qjl_const, kqx = cb.qjl_const_x;
  float* out = logits + ((size_t)b * Hq + (size_t)kvh * G + c) * capacity;
  bool ok = true;
  int pending_from = 0;                      // first stage whose copy may still be in flight
  uint32_t nxa = 0u, nxb = 0u;               // a split key's group A norms (single-tile steps only)
  auto tile_words = [&](const uint8_t* rec, const uint8_t* nrm, int lt, int64_t tg, uint32_t(&wa)[P],
                        uint32_t(&wb)[P], uint32_t& na, uint32_t& nb, uint32_t& ea, uint32_t& eb) {
    const uint8_t* ra = rec + ((size_t)lt * 16 + g) * RB + c * P * 4;
    const uint8_t* rbp = ra + 8 * RB;
    ea = eb = 0u;
    if (EXT && c < EXT) {
      ea = reinterpret_cast<const uint32_t*>(rec + ((size_t)lt * 16 + g) * RB + 16 * P)[c];
      eb = reinterpret_cast<const uint32_t*>(rec + ((size_t)lt * 16 + g + 8) * RB + 16 * P)[c];
    }
    if constexpr (P == 4 && EXT == 0) {
      const uint4 x = *reinterpret_cast<const uint4*>(ra);
      const uint4 y = *reinterpret_cast<const uint4*>(rbp);
      wa[0] = x.x; wa[1] = x.y; wa[2] = x.z; wa[3] = x.w;
      wb[0] = y.x; wb[1] = y.y; wb[2] = y.z; wb[3] = y.w;
    } else {
#pragma unroll
      for (int p = 0; p < P; ++p) {
        wa[p] = reinterpret_cast<const uint32_t*>(ra)[p];
        wb[p] = reinterpret_cast<const uint32_t*>(rbp)[p];
      }
    }
    if constexpr (SPLIT) {
      const uint2 x = reinterpret_cast<const uint2*>(nrm)[lt * 16 + g];
      const uint2 y = reinterpret_cast<const uint2*>(nrm)[lt * 16 + g + 8];
      nxa = x.x;
      na = x.y;
      nxb = y.x;
      nb = y.y;
    } else if constexpr (QJL) {
      na = reinterpret_cast<const uint32_t*>(nrm)[lt * 16 + g];
      nb = reinterpret_cast<const uint32_t*>(nrm)[lt * 16 + g + 8];
    } else {
      na = reinterpret_cast<const unsigned short*>(nrm)[lt * 16 + g];
      nb = reinterpret_cast<const unsigned short*>(nrm)[lt * 16 + g + 8];
    }
    // keys at or past L are scored like the others (their bytes are staged
    // cache rows of the same tile); an MMA output row depends only on its
    // own key, and emit stores only keys below L
    (void)tg;
  };
  // token positions in 32 bits (capacity < 2^31)
  const int L32 = (int)L;
  auto emit = [&](int64_t tg, uint32_t na, uint32_t nb, float s1a, float s1b, float s2a, float s2b) {
    const int ta = (int)tg * 16 + g, tb = ta + 8;
    if (c < G) {
      if (ta < L32) out[ta] = est_key<QJL>(na, s1a, s2a, kq);
      if (tb < L32) out[tb] = est_key<QJL>(nb, s1b, s2b, kq);
    }
  };
  // a split key: group A's estimate from nxa / nxb plus group B's
  auto emit_split = [&](int64_t tg, uint32_t na, uint32_t nb, const float (&s1)[1][2], const float (&s2)[1][2],
                        const float (&s1x)[1][2], const float (&s2x)[1][2]) {
    const int64_t ta = tg * 16 + g, tb = ta + 8;
    if (c < G) {
      if (ta < L) out[ta] = est_groups<QJL, true>(nxa, na, s1x[0][0], s2x[0][0], s1[0][0], s2[0][0], kqx, kq);
      if (tb < L) out[tb] = est_groups<QJL, true>(nxb, nb, s1x[0][1], s2x[0][1], s1[0][1], s2[0][1], kqx, kq);
    }
  };
  for (int st = 0; st < nst; ++st) {
    const int slot = st % kRing;
    if (!__syncthreads_and(bar_wait(su32(&bars[slot]), (uint32_t)((st / kRing) & 1), st == 0 ? cb.first_wait : kWaitLimit))) {
      ok = false;
      pending_from = st;
      break;
    }
    const uint8_t* rec = srec + (size_t)slot * kStageRec;
    const uint8_t* nrm = snrm + (size_t)slot * kStageNrm;
    const int t_a = st * kStageTiles, n_here = min(kStageTiles, nt - t_a);
    // two tiles per iteration (warp, warp + 4) for independent MMA chains;
    // a lone last tile is scored on its own
    for (int lt = warp; lt < n_here; lt += 8) {
      const int lt2 = lt + 4;
      if (kPairs && lt2 < n_here) {
        uint32_t wa[2][P], wb[2][P], na, nb, ma, mb, ea[2], eb[2];
        tile_words(rec, nrm, lt, tile0 + t_a + lt, wa[0], wb[0], na, nb, ea[0], eb[0]);
        tile_words(rec, nrm, lt2, tile0 + t_a + lt2, wa[1], wb[1], ma, mb, ea[1], eb[1]);
        float s1[2][2], s2[2][2];
        qk.template score_mixed<2, EXT>(wa, wb, ea, eb, s1, s2);
        emit(tile0 + t_a + lt, na, nb, s1[0][0], s1[0][1], s2[0][0], s2[0][1]);
        emit(tile0 + t_a + lt2, ma, mb, s1[1][0], s1[1][1], s2[1][0], s2[1][1]);
      } else if constexpr (SPLIT) {
        uint32_t wa[1][P], wb[1][P], na, nb, ea[1], eb[1];
        float s1[1][2], s2[1][2], s1x[1][2], s2x[1][2];
        tile_words(rec, nrm, lt, tile0 + t_a + lt, wa[0], wb[0], na, nb, ea[0], eb[0]);
        qk.template score_groups<1, EXT, true>(wa, wb, ea, eb, s1, s2, s1x, s2x);
        emit_split(tile0 + t_a + lt, na, nb, s1, s2, s1x, s2x);
        if (lt2 < n_here) {
          tile_words(rec, nrm, lt2, tile0 + t_a + lt2, wa[0], wb[0], na, nb, ea[0], eb[0]);
          qk.template score_groups<1, EXT, true>(wa, wb, ea, eb, s1, s2, s1x, s2x);
          emit_split(tile0 + t_a + lt2, na, nb, s1, s2, s1x, s2x);
        }
      } else {
        uint32_t wa[1][P], wb[1][P], na, nb, ea[1], eb[1];
        tile_words(rec, nrm, lt, tile0 + t_a + lt, wa[0], wb[0], na, nb, ea[0], eb[0]);
        float s1[1][2], s2[1][2];
        qk.template score_mixed<1, EXT>(wa, wb, ea, eb, s1, s2);
        emit(tile0 + t_a + lt, na, nb, s1[0][0], s1[0][1], s2[0][0], s2[0][1]);
        if (!kPairs && lt2 < n_here) {
          uint32_t xa[1][P], xb[1][P], ma, mb;
          tile_words(rec, nrm, lt2, tile0 + t_a + lt2, xa[0], xb[0], ma, mb, ea[0], eb[0]);
          qk.template score_mixed<1, EXT>(xa, xb, ea, eb, s1, s2);
          emit(tile0 + t_a + lt2, ma, mb, s1[0][0], s1[0][1], s2[0][0], s2[0][1]);
        }
      }
    }
    // The query fragments have been used (the first stage is scored), so
    // the next call's query prep, which rewrites the workspace they came
    // from, may start on SMs this grid frees; it waits for this grid before
    // its own dependent reads any cache row or writes any output.
    if (st == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // every warp is done with this ring slot: refill it with stage st + kRing
    if (st + kRing < nst) {
      __syncthreads();
      request(st + kRing, min(kStageTiles, nt - (st + kRing) * kStageTiles));
      issued = st + kRing + 1;
    }
  }
  if (!ok) {
    if (tid == 0) atomicOr(status, 2);
    // let the copies still in flight land (bounded) before the shared memory is released
    for (int st = pending_from; st < issued; ++st) bar_wait(su32(&bars[st % kRing]), (uint32_t)((st / kRing) & 1));
  }
}

// ---------------------------------------------------------------------------
// Fused decode attention: QK as above, online softmax per head slot, and the
// weighted value sum  acc[i] = sum_t p_t n_v,t yhat_v,t[i]  in the rotated
// domain on the tensor cores (A = value bits, 16 coordinates x 16 tokens, the
// two tokens of a pair in the two fp16 halves; B = -2 coef_v p_t n_v,t).
// Thread (g, c) owns head slot c and coordinates 16g .. 16g+15.
// ---------------------------------------------------------------------------
template <int PV>
struct VTile {
  uint32_t w[4][PV];
  float vn0, vn1;
  __device__ __forceinline__ void load(const uint32_t* vrec, const __half* vnrm, int VW, int64_t rowbase, int64_t t0,
                                       int64_t L, int g, int c) {
    const int vword = g >> 1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t t = t0 + 2 * c + (j & 1) + 8 * (j >> 1);
      if (t < L) {
#pragma unroll
        for (int p = 0; p < PV; ++p) w[j][p] = __ldg(vrec + (rowbase + t) * VW + vword * PV + p);
      } else {
#pragma unroll
        for (int p = 0; p < PV; ++p) w[j][p] = 0;
      }
    }
    const int64_t ta = t0 + g, tb = ta + 8;
    vn0 = ta < L ? __half2float(vnrm[rowbase + ta]) : 0.f;
    vn1 = tb < L ? __half2float(vnrm[rowbase + tb]) : 0.f;
  }
};

template <int NVK, int PK, int NVV, int PV>
__global__ void __launch_bounds__(128, 2) k_attn(const Dev kcb, const Dev vcb, const uint8_t* __restrict__ kcache,
                                              const uint8_t* __restrict__ vcache, int Hq, int Hkv, int64_t capacity,
                                              int64_t cache_rows, const int32_t* __restrict__ seq_lens,
                                              const uint8_t* __restrict__ prep, float scale_log2,
                                              float* __restrict__ partials, int tiles_per_cta) {
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t L = seq_lens[b];
  const int64_t ntiles = (L + 15) / 16;
  const int64_t tile0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t tend = min(tile0 + tiles_per_cta, ntiles);

  float m_run = -INFINITY, l_run = 0.f, wsum = 0.f;
  float acc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
  PvTotal tot;
  tot.zero();

  if (tile0 + warp < tend) {
    QK16<NVK, PK> qk;
    qk.load(prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(128), lane, kcb);
    float vcn[NVV];
#pragma unroll
    for (int u = 0; u < NVV; ++u) vcn[u] = -2.f * vcb.vcoef[u];
    const uint32_t* krec = reinterpret_cast<const uint32_t*>(kcache);
    const uint32_t* knrm = reinterpret_cast<const uint32_t*>(kcache + norm_offset(kcb, cache_rows));
    const uint32_t* vrec = reinterpret_cast<const uint32_t*>(vcache);
    const __half* vnrm = reinterpret_cast<const __half*>(vcache + norm_offset(vcb, cache_rows));
    const int64_t rowbase = ((int64_t)b * Hkv + kvh) * capacity;
    const float kq = kcb.qjl_const;
    const int KW = kcb.W, VW = vcb.W;
    const uint32_t vsel = (g & 1) ? 0x7632u : 0x5410u;
    const int hh = g >> 1, pc = g & 1;    // B-fragment column: head slot, piece
    const int src0 = (2 * c) * 4 + hh, src1 = (2 * c + 1) * 4 + hh;

    KTile<PK> kcur, knxt;
    VTile<PV> vcur, vnxt;
    int64_t tile = tile0 + warp;
    kcur.load(krec, knrm, KW, rowbase, tile * 16 + g, L, c);
    vcur.load(vrec, vnrm, VW, rowbase, tile * 16, L, g, c);
    int chain = 0;    // tiles in the current mma chain
    for (; tile < tend; tile += 4) {
      const int64_t tn = tile + 4;
      if (tn < tend) {
        knxt.load(krec, knrm, KW, rowbase, tn * 16 + g, L, c);
        vnxt.load(vrec, vnrm, VW, rowbase, tn * 16, L, g, c);
      }
      const int64_t ta = tile * 16 + g, tb = ta + 8;
      uint32_t wa[1][PK], wb[1][PK];
#pragma unroll
      for (int p = 0; p < PK; ++p) {
        wa[0][p] = kcur.wa[p];
        wb[0][p] = kcur.wb[p];
      }
      float s1[1][2], s2[1][2];
      qk.template score<1>(wa, wb, s1, s2);
      // scores in log2 units
      const float sa = ta < L ? est_from(kcur.na, s1[0][0], s2[0][0], kq) * scale_log2 : -INFINITY;
      const float sb = tb < L ? est_from(kcur.nb, s1[0][1], s2[0][1], kq) * scale_log2 : -INFINITY;
      float mx = fmaxf(sa, sb);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      if (__any_sync(kFull, mx > m_run)) {
        const float m_new = fmaxf(m_run, mx);
        const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
        l_run *= alpha;
        wsum *= alpha;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mt][e] *= alpha;
        tot.scale(alpha);
        m_run = m_new;
      }
      const float pa = sa == -INFINITY ? 0.f : exp2f(sa - m_run);
      const float pb = sb == -INFINITY ? 0.f : exp2f(sb - m_run);
      const float wA = pa * vcur.vn0, wB = pb * vcur.vn1;
      float ps = pa + pb, ws = wA + wB;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        ps += __shfl_xor_sync(kFull, ps, o);
        ws += __shfl_xor_sync(kFull, ws, o);
      }
      l_run += ps;
      wsum += ws;
      // weights of tokens 2c, 2c+1, 2c+8, 2c+9 for head slot hh, in B-fragment order
      const float w0 = __shfl_sync(kFull, wA, src0);
      const float w1 = __shfl_sync(kFull, wA, src1);
      const float w8 = __shfl_sync(kFull, wB, src0);
      const float w9 = __shfl_sync(kFull, wB, src1);
#pragma unroll
      for (int u = 0; u < NVV; ++u) {
        const float cu = vcn[u];
        const uint32_t b0 = piece2(cu * w0, cu * w1, pc);
        const uint32_t b1 = piece2(cu * w8, cu * w9, pc);
        uint32_t x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r = 0;
#pragma unroll
          for (int p = 0; p < PV; ++p)
            if (kOddMask[u] >> p & 1u) r ^= vcur.w[j][p];
          x[j] = r;
        }
        uint32_t r01[16], r89[16];
        expand16_v(__byte_perm(x[0], x[1], vsel), r01);
        expand16_v(__byte_perm(x[2], x[3], vsel), r89);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          mma_f16(acc[mt], r01[2 * mt], r01[2 * mt + 1], r89[2 * mt], r89[2 * mt + 1], b0, b1);
      }
      kcur = knxt;
      vcur = vnxt;
      if (++chain == 2 * kPvFlushStages) {
        tot.flush(acc);
        chain = 0;
      }
    }
  }
  tot.flush(acc);
  // this warp's partial: head slot c, coordinates 16g + 2mt (+1);
  // acc = C0 * wsum + value_factor(beta) * D
  float c0 = 0.f;
#pragma unroll
  for (int u = 0; u < NVV; ++u) c0 += vcb.vcoef[u];
  const int nchunks = gridDim.x;
  float* part = partials + ((((size_t)b * Hkv + kvh) * nchunks + blockIdx.x) * kAttnWarps + warp) * partial_floats(128);
  float* ph = part + c * (2 + 128);
  if (g == 0) {
    ph[0] = m_run;
    ph[1] = l_run;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int b0 = 2 * mt, b1 = 2 * mt + 1;
    const float f0 = value_factor(b0), f1 = value_factor(b1);
    ph[2 + 16 * g + b0] = fmaf(f0, tot.t[mt][0], c0 * wsum);
    ph[2 + 16 * g + b1] = fmaf(f1, tot.t[mt][1], c0 * wsum);
  }
}

// Resident CTAs per SM of the staged attention kernel: 4, or 3 where it needs
// more registers (4 key virtual planes, or extra-bit words in keys or values).
// The host sizes the grid to one wave of the same count.
constexpr int attn_min_blocks(int nvk, int extk) { return nvk >= 4 || extk > 0 ? 3 : 4; }

// ---------------------------------------------------------------------------
// Fused decode attention with bulk-copy staging (capacity a multiple of 16),
// launched as the programmatic dependent of the query prep.  Same arithmetic
// as k_attn; the key and value records and norms of each stage of
// kStageTiles tiles arrive by cp.async.bulk in a ring of kRing slots (the
// first stage is requested right after the wait for the prep, before the
// query fragments are loaded), and each warp scores tiles warp and warp + 4
// of every stage.
// ---------------------------------------------------------------------------
template <int NVK, int PK, int NVV, int PV, bool QJLK, int EXTK, int EXTV, bool SPLIT = false>
__global__ void __launch_bounds__(128, attn_min_blocks(NVK, EXTK + EXTV)) k_attn_staged(const Dev kcb, const Dev vcb,
                                                     const uint8_t* __restrict__ kcache,
                                                     const uint8_t* __restrict__ vcache, int Hq, int Hkv,
                                                     int64_t capacity, int64_t cache_rows, const RowMap map,
                                                     const int32_t* __restrict__ seq_lens,
                                                     const uint8_t* __restrict__ prep, float scale_log2,
                                                     float* __restrict__ partials, int tiles_per_cta,
                                                     int* __restrict__ status) {
  constexpr int RBK = 16 * PK + 4 * EXTK;       // key record bytes at d = 128 (+ extra-bit words)
  constexpr int RBV = 16 * PV + 4 * EXTV;       // value record bytes (+ extra-bit words)
  constexpr int NBK = SPLIT ? 8 : QJLK ? 4 : 2;  // key norm entry bytes
  constexpr int kSK = kStageTiles * 16 * RBK, kSKN = kStageTiles * 16 * NBK;
  constexpr int kSV = kStageTiles * 16 * RBV, kSVN = kStageTiles * 16 * 2;
  constexpr int kSlot = kSK + kSKN + kSV + kSVN;
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ __align__(8) uint64_t bars[kRing];
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
                     "r"((uint32_t)(t_n * 16 * (RBK + NBK + RBV + 2)))
                     : "memory");
      const int64_t t0 = (tile0 + (int64_t)st * kStageTiles) * 16;
      if (map.table == nullptr) {
        if (lane == 0) {
          const int64_t row = ((int64_t)b * Hkv + kvh) * capacity + t0;
          const uint32_t n = (uint32_t)(t_n * 16);
          bulk_g2s(su32(base), kcache + row * RBK, n * RBK, bar);
          bulk_g2s(su32(base + kSK), gkn + row * NBK, n * NBK, bar);
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
          const int rb = a == 0 ? RBK : a == 1 ? NBK : a == 2 ? RBV : 2;
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
  // the first stages stream from HBM into L2 while the prep still runs
  if (warp == 0)
    for (int st = 0; st < min(nst, kRing); ++st) {
      const int64_t t0 = (tile0 + (int64_t)st * kStageTiles) * 16;
      const int n = min(kStageTiles, nt - st * kStageTiles) * 16;
      int k = 0, cnt = n;
      int64_t row = ((int64_t)b * Hkv + kvh) * capacity + t0;
      if (map.table ? page_run(map, b, kvh, Hkv, t0, n, lane >> 2, status, k, cnt, row) : lane < 4) {
        const int a = lane & 3;
        const int rb = a == 0 ? RBK : a == 1 ? NBK : a == 2 ? RBV : 2;
        const uint8_t* g = a == 0 ? kcache : a == 1 ? gkn : a == 2 ? vcache : gvn;
        prefetch_l2(g + row * rb, (uint32_t)(cnt * rb));
      }
    }
  // query fragments come from the preceding prep grid (whose completion also
  // implies that of any cache append before it): no cache row is read into
  // the SM before this wait; the first stage goes out right after it
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (nst > 0) request(0, min(kStageTiles, nt));
  QK16<NVK, PK, QJLK> qk;
  qk.load(prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(128), lane, kcb);
  __syncthreads();
  for (int st = 1; st < min(nst, kRing); ++st) request(st, min(kStageTiles, nt - st * kStageTiles));
  int issued = min(nst, kRing);

  float m_run = -INFINITY, l_run = 0.f, wsum = 0.f;
  float acc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
  PvTotal tot;
  tot.zero();
  float vcn[NVV], vcnx[EXTV ? 2 * NVV : 1];
#pragma unroll
  for (int u = 0; u < NVV; ++u) vcn[u] = -2.f * vcb.vcoef[u];
#pragma unroll
  for (int u = 0; u < (EXTV ? 2 * NVV : 1); ++u) vcnx[u] = EXTV ? -2.f * vcb.vcoef_x[u] : 0.f;
  const float kq = kcb.qjl_const, kqx = kcb.qjl_const_x;
  const uint32_t vsel = (g & 1) ? 0x7632u : 0x5410u;
  const int hh = g >> 1, pc = g & 1;    // B-fragment column: head slot, piece
  const int src0 = (2 * c) * 4 + hh, src1 = (2 * c + 1) * 4 + hh;
  const int vword = g >> 1;
  // mixed-bit values: the first EXTV word columns use the extended codebook,
  // whose low bit is the column's extra word
  const bool vxl = EXTV > 0 && vword < EXTV;
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
    const uint8_t* sk = base;
    const uint8_t* skn = base + kSK;
    const uint8_t* sv = base + kSK + kSKN;
    const __half* svn = reinterpret_cast<const __half*>(base + kSK + kSKN + kSV);
    const int t_a = st * kStageTiles, n_here = min(kStageTiles, nt - t_a);
    for (int lt = warp; lt < n_here; lt += 4) {
      const int t0 = ((int)tile0 + t_a + lt) * 16;      // first token of the tile
      const int ta = t0 + g, tb = ta + 8;
      // keys g and g+8: column c words (+ the extra-bit word of column c)
      uint32_t wa[1][PK], wb[1][PK], ea[1] = {0u}, eb[1] = {0u};
      {
        const uint32_t* ka = reinterpret_cast<const uint32_t*>(sk + ((size_t)lt * 16 + g) * RBK);
        const uint32_t* kb2 = reinterpret_cast<const uint32_t*>(sk + ((size_t)lt * 16 + g + 8) * RBK);
#pragma unroll
        for (int p = 0; p < PK; ++p) {
          wa[0][p] = ka[c * PK + p];
          wb[0][p] = kb2[c * PK + p];
        }
        if (EXTK > 0 && c < EXTK) {
          ea[0] = ka[4 * PK + c];
          eb[0] = kb2[4 * PK + c];
        }
      }
      float s1[1][2], s2[1][2], s1x[1][2], s2x[1][2];
      qk.template score_groups<1, EXTK, SPLIT>(wa, wb, ea, eb, s1, s2, s1x, s2x);
      uint32_t na, nb, nxa = 0u, nxb = 0u;
      if constexpr (SPLIT) {
        const uint2 x = reinterpret_cast<const uint2*>(skn)[lt * 16 + g];
        const uint2 y = reinterpret_cast<const uint2*>(skn)[lt * 16 + g + 8];
        nxa = x.x;
        na = x.y;
        nxb = y.x;
        nb = y.y;
      } else if constexpr (QJLK) {
        na = reinterpret_cast<const uint32_t*>(skn)[lt * 16 + g];
        nb = reinterpret_cast<const uint32_t*>(skn)[lt * 16 + g + 8];
      } else {
        na = reinterpret_cast<const unsigned short*>(skn)[lt * 16 + g];
        nb = reinterpret_cast<const unsigned short*>(skn)[lt * 16 + g + 8];
      }
      // scores in log2 units
      const float sa =
          ta < L32 ? est_groups<QJLK, SPLIT>(nxa, na, s1x[0][0], s2x[0][0], s1[0][0], s2[0][0], kqx, kq) * scale_log2
                 : -INFINITY;
      const float sb =
          tb < L32 ? est_groups<QJLK, SPLIT>(nxb, nb, s1x[0][1], s2x[0][1], s1[0][1], s2[0][1], kqx, kq) * scale_log2
                 : -INFINITY;
      float mx = fmaxf(sa, sb);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      if (__any_sync(kFull, mx > m_run)) {
        const float m_new = fmaxf(m_run, mx);
        const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
        l_run *= alpha;
        wsum *= alpha;
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
      float ps = pa + pb, ws = wA + wB;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        ps += __shfl_xor_sync(kFull, ps, o);
        ws += __shfl_xor_sync(kFull, ws, o);
      }
      l_run += ps;
      wsum += ws;
      // weights of tokens 2c, 2c+1, 2c+8, 2c+9 for head slot hh, in B-fragment order
      const float w0 = __shfl_sync(kFull, wA, src0);
      const float w1 = __shfl_sync(kFull, wA, src1);
      const float w8 = __shfl_sync(kFull, wB, src0);
      const float w9 = __shfl_sync(kFull, wB, src1);
      // value words (word column g/2) of tokens 2c, 2c+1, 2c+8, 2c+9
      uint32_t vw[4][PV], ve[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tok = 2 * c + (j & 1) + 8 * (j >> 1);
        const uint32_t* vrow = reinterpret_cast<const uint32_t*>(sv + ((size_t)lt * 16 + tok) * RBV);
#pragma unroll
        for (int p = 0; p < PV; ++p) vw[j][p] = vrow[vword * PV + p];
        ve[j] = vxl ? vrow[4 * PV + vword] : 0u;
      }
#pragma unroll
      for (int u = 0; u < NVV; ++u) {
        const float cu = vcn[u];
        const uint32_t b0 = piece2(cu * w0, cu * w1, pc);
        const uint32_t b1 = piece2(cu * w8, cu * w9, pc);
        uint32_t x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r = 0;
#pragma unroll
          for (int p = 0; p < PV; ++p)
            if (kOddMask[u] >> p & 1u) r ^= vw[j][p];
          x[j] = vxl ? 0u : r;                    // extended-codebook columns take the planes below
        }
        uint32_t r01[16], r89[16];
        expand16_v(__byte_perm(x[0], x[1], vsel), r01);
        expand16_v(__byte_perm(x[2], x[3], vsel), r89);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          mma_f16(acc[mt], r01[2 * mt], r01[2 * mt + 1], r89[2 * mt], r89[2 * mt + 1], b0, b1);
      }
      if constexpr (EXTV > 0) {
        // the extended codebook's 2 NVV virtual planes (plane PV = extra
        // word), fed only by the extra-bit columns' lanes
#pragma unroll
        for (int u = 0; u < 2 * NVV; ++u) {
          const float cu = vcnx[u];
          const uint32_t b0 = piece2(cu * w0, cu * w1, pc);
          const uint32_t b1 = piece2(cu * w8, cu * w9, pc);
          uint32_t x[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t r = (kOddMask[u] >> PV & 1u) ? ve[j] : 0u;
#pragma unroll
            for (int p = 0; p < PV; ++p)
              if (kOddMask[u] >> p & 1u) r ^= vw[j][p];
            x[j] = vxl ? r : 0u;
          }
          uint32_t r01[16], r89[16];
          expand16_v(__byte_perm(x[0], x[1], vsel), r01);
          expand16_v(__byte_perm(x[2], x[3], vsel), r89);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
            mma_f16(acc[mt], r01[2 * mt], r01[2 * mt + 1], r89[2 * mt], r89[2 * mt + 1], b0, b1);
        }
      }
    }
    if (st % kPvFlushStages == kPvFlushStages - 1) tot.flush(acc);
    // The query fragments have been used (the first stage is scored), so
    // the next call's query prep, which rewrites the workspace they came
    // from, may start on SMs this grid frees; it waits for this grid before
    // its own dependent reads any cache row or writes any output.
    if (st == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // every warp is done with this ring slot: refill it with stage st + kRing
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
  // this warp's partial: head slot c, coordinates 16g + 2mt (+1);
  // acc = C0 * wsum + value_factor(beta) * D
  float c0 = 0.f;
#pragma unroll
  for (int u = 0; u < NVV; ++u) c0 += vcb.vcoef[u];
  if (EXTV > 0 && vxl) {
    c0 = 0.f;
#pragma unroll
    for (int u = 0; u < (EXTV ? 2 * NVV : 0); ++u) c0 += vcb.vcoef_x[u];
  }
  const int nchunks = gridDim.x;
  float* part = partials + ((((size_t)b * Hkv + kvh) * nchunks + blockIdx.x) * kAttnWarps + warp) * partial_floats(128);
  float* ph = part + c * (2 + 128);
  if (g == 0) {
    ph[0] = m_run;
    ph[1] = l_run;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int b0 = 2 * mt, b1 = 2 * mt + 1;
    const float f0 = value_factor(b0), f1 = value_factor(b1);
    ph[2 + 16 * g + b0] = fmaf(f0, tot.t[mt][0], c0 * wsum);
    ph[2 + 16 * g + b1] = fmaf(f1, tot.t[mt][1], c0 * wsum);
  }
}

// Merge the split partials of one (b, query head) and rotate back once:
// M = max m_p, o_rot = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,
// out = Pi_v^T o_rot.  The maximum, the weights and L are computed by the
// whole CTA (parts strided over threads); thread i then sums coordinate i.
// Groups larger than 4 heads per kv head are scored 4 heads at a time; the
// partials of head group g start at partials + g * group_stride floats.
constexpr int kMergeMaxParts = 4096;
__global__ void __launch_bounds__(128) k_attn_merge(const Dev vcb, const float* __restrict__ partials, int Hq, int Hkv,
                                                    int nparts, int64_t group_stride, float* __restrict__ out) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int G = Hq / Hkv, kvh = h / G, slot = h % G;
  constexpr int d = 128;
  constexpr int64_t PF = 4 * (2 + d);        // partial_floats(d)
  __shared__ float so[d], red[4], wts[kMergeMaxParts];
  const float* base =
      partials + (slot / 4) * group_stride + ((size_t)b * Hkv + kvh) * nparts * PF + (slot % 4) * (2 + d);
  const int i = threadIdx.x, warp = i >> 5, lane = i & 31;
  const bool cache_w = nparts <= kMergeMaxParts;
  float mloc = -INFINITY;
  for (int p = i; p < nparts; p += 128) mloc = fmaxf(mloc, base[(size_t)p * PF]);
#pragma unroll
  for (int o = 16; o; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, o));
  if (lane == 0) red[warp] = mloc;
  __syncthreads();
  const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float lloc = 0.f;
  for (int p = i; p < nparts; p += 128) {
    const float mp = base[(size_t)p * PF];
    const float w = (M == -INFINITY || mp == -INFINITY) ? 0.f : exp2f(mp - M);
    if (cache_w) wts[p] = w;
    lloc = fmaf(w, base[(size_t)p * PF + 1], lloc);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) lloc += __shfl_xor_sync(kFull, lloc, o);
  if (lane == 0) red[warp] = lloc;
  __syncthreads();
  const float Lsum = (red[0] + red[1]) + (red[2] + red[3]);
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  int p = 0;
  auto weight = [&](int q) {
    if (cache_w) return wts[q];
    const float mp = base[(size_t)q * PF];
    return (M == -INFINITY || mp == -INFINITY) ? 0.f : exp2f(mp - M);
  };
  for (; p + 4 <= nparts; p += 4) {
    a0 = fmaf(weight(p), base[(size_t)p * PF + 2 + i], a0);
    a1 = fmaf(weight(p + 1), base[(size_t)(p + 1) * PF + 2 + i], a1);
    a2 = fmaf(weight(p + 2), base[(size_t)(p + 2) * PF + 2 + i], a2);
    a3 = fmaf(weight(p + 3), base[(size_t)(p + 3) * PF + 2 + i], a3);
  }
  for (; p < nparts; ++p) a0 = fmaf(weight(p), base[(size_t)p * PF + 2 + i], a0);
  const float a = (a0 + a1) + (a2 + a3);
  so[i] = Lsum > 0.f ? a / Lsum : 0.f;
  __syncthreads();
  float o = 0.f;
  const uint64_t keep = l2_policy_evict_last();
  for (int k = 0; k < d; ++k) o = fmaf(ld_table(vcb.Pi + (size_t)k * d + i, keep), so[k], o);
  out[((size_t)b * Hq + h) * d + i] = o;
}

template <int NVK, int PK>
static void attn_v(int b1v, dim3 grid, cudaStream_t s, const Dev& k, const Dev& v, const uint8_t* kc,
                   const uint8_t* vc, int Hq, int Hkv, int64_t cap, int64_t rows, const int32_t* sl, const uint8_t* prep,
                   float sl2, float* parts, int tpc) {
  switch (b1v) {
    case 1: k_attn<NVK, PK, 1, 1><<<grid, 128, 0, s>>>(k, v, kc, vc, Hq, Hkv, cap, rows, sl, prep, sl2, parts, tpc); break;
    case 2: k_attn<NVK, PK, 2, 2><<<grid, 128, 0, s>>>(k, v, kc, vc, Hq, Hkv, cap, rows, sl, prep, sl2, parts, tpc); break;
    case 3: k_attn<NVK, PK, 4, 3><<<grid, 128, 0, s>>>(k, v, kc, vc, Hq, Hkv, cap, rows, sl, prep, sl2, parts, tpc); break;
    default: k_attn<NVK, PK, 8, 4><<<grid, 128, 0, s>>>(k, v, kc, vc, Hq, Hkv, cap, rows, sl, prep, sl2, parts, tpc); break;
  }
}

// The query prep, the scoring kernels and the cache append share SMs while
// their grids overlap; an SM only hosts CTAs of kernels with the same
// shared-memory carveout, so all of them ask for the largest one.
cudaError_t prefer_max_shared(const void* fn) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_prep_append(const Dev& cb, const float* q, int B, int Hq, int Hkv, uint8_t* prep, uint8_t* cache,
                               int64_t cache_rows, const void* x, int x_dtype, int64_t n, int d_in,
                               const int64_t* dst_rows, int* status, cudaStream_t s) {
  static cudaError_t configured = prefer_max_shared(reinterpret_cast<const void*>(k_prep_append));
  if (configured != cudaSuccess) return configured;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(Hkv * 16 + ((n + 3) / 4) * 4), B);   // whole 4-CTA clusters
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 4;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_prep_append, cb, q, Hq, Hkv, prep, cache, cache_rows, x, x_dtype, n, d_in,
                            dst_rows, status);
}

cudaError_t launch_prep(const Dev& cb, const float* q, int B, int Hq, int Hkv, uint8_t* prep, cudaStream_t s) {
  static cudaError_t configured = prefer_max_shared(reinterpret_cast<const void*>(k_prep));
  if (configured != cudaSuccess) return configured;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(Hkv * 16, B);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 4;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_prep, cb, q, Hq, Hkv, prep);
}

// Key caches with the QJL term (PROD) use b' = 1..3 code planes + the sign
// plane, optionally with 1 or 2 extra-bit word columns (mixed-bit caches);
// MSE-only key caches use b = 1..4 code planes.
// Outlier-channel split keys are mixed-bit records with per-group norms.
#define TQ_LOGITS_DISPATCH(CALL)                          \
  if (cb.kind == 0 && cb.split) {                         \
    switch (cb.b1 * 4 + cb.extra / 32) {                  \
      case 5: CALL(1, 2, true, 1, true);                  \
      case 6: CALL(1, 2, true, 2, true);                  \
      case 9: CALL(2, 3, true, 1, true);                  \
      case 10: CALL(2, 3, true, 2, true);                 \
      case 13: CALL(4, 4, true, 1, true);                 \
      default: CALL(4, 4, true, 2, true);                 \
    }                                                     \
  }                                                       \
  if (cb.kind == 0) {                                     \
    const int ext = cb.extra / 32;                        \
    switch (cb.b1 * 4 + ext) {                            \
      case 4: CALL(1, 2, true, 0, false);                 \
      case 5: CALL(1, 2, true, 1, false);                 \
      case 6: CALL(1, 2, true, 2, false);                 \
      case 8: CALL(2, 3, true, 0, false);                 \
      case 9: CALL(2, 3, true, 1, false);                 \
      case 10: CALL(2, 3, true, 2, false);                \
      case 13: CALL(4, 4, true, 1, false);                \
      case 14: CALL(4, 4, true, 2, false);                \
      default: CALL(4, 4, true, 0, false);                \
    }                                                     \
  }                                                       \
  switch (cb.b1) {                                        \
    case 1: CALL(1, 1, false, 0, false);                  \
    case 2: CALL(2, 2, false, 0, false);                  \
    case 3: CALL(4, 3, false, 0, false);                  \
    default: CALL(8, 4, false, 0, false);                 \
  }

cudaError_t launch_logits(const Dev& cb, const uint8_t* kc, int B, int Hq, int Hkv, int64_t capacity,
                          int64_t rows, const int32_t* seq_lens, const uint8_t* prep, float* logits, int nchunks,
                          int tpc, cudaStream_t s) {
  const dim3 grid(nchunks, Hkv, B);
#define TQ_CALL(NV, P, Q, X, S)                                                                                 \
  k_logits<NV, P, Q, X, S><<<grid, 128, 0, s>>>(cb, kc, Hq, Hkv, capacity, rows, seq_lens, prep, logits, tpc); \
  return cudaGetLastError()
  TQ_LOGITS_DISPATCH(TQ_CALL)
#undef TQ_CALL
}

template <int NV, int P, bool QJL, int EXT, bool SPLIT>
static cudaError_t logits_staged_t(const Dev& cb, const uint8_t* kc, int B, int Hq, int Hkv, int64_t capacity,
                                   int64_t rows, const RowMap& map, const int32_t* seq_lens, const uint8_t* prep,
                                   float* logits, int nchunks, int tpc, int* status, cudaStream_t s) {
  constexpr size_t smem = (size_t)kRing * kStageTiles * 16 * (16 * P + 4 * EXT + (SPLIT ? 8 : QJL ? 4 : 2));
  auto kern = k_logits_staged<NV, P, QJL, EXT, SPLIT>;
  static cudaError_t configured = [&] {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = prefer_max_shared(reinterpret_cast<const void*>(kern));
    return e;
  }();
  if (configured != cudaSuccess) return configured;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nchunks, Hkv, B);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, cb, kc, Hq, Hkv, capacity, rows, map, seq_lens, prep, logits, tpc, status);
}

cudaError_t launch_logits_staged(const Dev& cb, const uint8_t* kc, int B, int Hq, int Hkv, int64_t capacity,
                                 int64_t rows, const RowMap& map, const int32_t* seq_lens, const uint8_t* prep,
                                 float* logits, int nchunks, int tpc, int* status, cudaStream_t s) {
#define TQ_CALL(NV, P, Q, X, S)                                                                                      \
  return logits_staged_t<NV, P, Q, X, S>(cb, kc, B, Hq, Hkv, capacity, rows, map, seq_lens, prep, logits, nchunks, tpc, \
                                         status, s)
  TQ_LOGITS_DISPATCH(TQ_CALL)
#undef TQ_CALL
}
#undef TQ_LOGITS_DISPATCH

template <int NVK, int PK, int NVV, int PV, bool QJLK, int EXTK, int EXTV, bool SPLIT>
static cudaError_t attn_staged_t(dim3 grid, cudaStream_t s, const Dev& k, const Dev& v, const uint8_t* kc,
                                 const uint8_t* vc, int Hq, int Hkv, int64_t cap, int64_t rows, const RowMap& map,
                                 const int32_t* sl, const uint8_t* prep, float sl2, float* parts, int tpc,
                                 int* status) {
  constexpr size_t smem =
      (size_t)kRing * kStageTiles * 16 * (16 * PK + 4 * EXTK + (SPLIT ? 8 : QJLK ? 4 : 2) + 16 * PV + 4 * EXTV + 2);
  auto kern = k_attn_staged<NVK, PK, NVV, PV, QJLK, EXTK, EXTV, SPLIT>;
  static cudaError_t configured = [&] {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = prefer_max_shared(reinterpret_cast<const void*>(kern));
    return e;
  }();
  if (configured != cudaSuccess) return configured;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, k, v, kc, vc, Hq, Hkv, cap, rows, map, sl, prep, sl2, parts, tpc, status);
}

// Value codebooks: every b' for keys with the QJL term and no extra bits;
// b = 3 and 4 for MSE-only and mixed-bit keys; mixed-bit values (extra bit on
// d/4 coordinates) at b = 2 and 3 for keys with the QJL term and no or d/4
// extra bits (other pairs are rejected by the host before launch).
template <int NVK, int PK, bool QJLK, int EXTK, bool SPLIT>
static cudaError_t attn_staged_v(int b1v, dim3 grid, cudaStream_t s, const Dev& k, const Dev& v, const uint8_t* kc,
                                 const uint8_t* vc, int Hq, int Hkv, int64_t cap, int64_t rows, const RowMap& map,
                                 const int32_t* sl, const uint8_t* prep, float sl2, float* parts, int tpc,
                                 int* status) {
#define TQ_ATTN_V(NVV, PV, XV)                                                                                     \
  return attn_staged_t<NVK, PK, NVV, PV, QJLK, EXTK, XV, SPLIT>(grid, s, k, v, kc, vc, Hq, Hkv, cap, rows, map, sl, \
                                                                prep, sl2, parts, tpc, status)
  if (v.extra != 0) {
    if constexpr (QJLK && EXTK <= 1 && !SPLIT) {
      switch (b1v) {
        case 2: TQ_ATTN_V(2, 2, 1);
        case 3: TQ_ATTN_V(4, 3, 1);
        default: return cudaErrorInvalidValue;
      }
    }
    return cudaErrorInvalidValue;
  }
  if constexpr (QJLK && EXTK == 0) {
    switch (b1v) {
      case 1: TQ_ATTN_V(1, 1, 0);
      case 2: TQ_ATTN_V(2, 2, 0);
      case 3: TQ_ATTN_V(4, 3, 0);
      default: TQ_ATTN_V(8, 4, 0);
    }
  } else {
    switch (b1v) {
      case 3: TQ_ATTN_V(4, 3, 0);
      case 4: TQ_ATTN_V(8, 4, 0);
      default: return cudaErrorInvalidValue;
    }
  }
#undef TQ_ATTN_V
}

bool attn_staged_supports(const Dev& kcb, const Dev& vcb) {
  if (kcb.mode != 0 || vcb.mode != 0) return false;
  if (vcb.extra != 0)
    return vcb.d == 128 && vcb.extra == 32 && (vcb.b1 == 2 || vcb.b1 == 3) && kcb.kind == 0 && kcb.extra <= 32 &&
           !kcb.split;
  const bool plain_keys = kcb.kind == 0 && kcb.extra == 0;
  return plain_keys || vcb.b1 == 3 || vcb.b1 == 4;
}

cudaError_t launch_attn_staged(const Dev& kcb, const Dev& vcb, const uint8_t* kc, const uint8_t* vc, int B, int Hq,
                               int Hkv, int64_t capacity, int64_t rows, const RowMap& map, const int32_t* seq_lens,
                               const uint8_t* prep, float scale_log2, float* parts, int nchunks, int tpc, int* status,
                               cudaStream_t s) {
  const dim3 grid(nchunks, Hkv, B);
#define TQ_ATTN_K(NVK, PK, Q, X, S)                                                                                  \
  return attn_staged_v<NVK, PK, Q, X, S>(vcb.b1, grid, s, kcb, vcb, kc, vc, Hq, Hkv, capacity, rows, map, seq_lens, \
                                         prep, scale_log2, parts, tpc, status)
  if (kcb.kind == 0 && kcb.split) {
    switch (kcb.b1 * 4 + kcb.extra / 32) {
      case 5: TQ_ATTN_K(1, 2, true, 1, true);
      case 6: TQ_ATTN_K(1, 2, true, 2, true);
      case 9: TQ_ATTN_K(2, 3, true, 1, true);
      case 10: TQ_ATTN_K(2, 3, true, 2, true);
      case 13: TQ_ATTN_K(4, 4, true, 1, true);
      default: TQ_ATTN_K(4, 4, true, 2, true);
    }
  }
  if (kcb.kind == 0) {
    switch (kcb.b1 * 4 + kcb.extra / 32) {
      case 4: TQ_ATTN_K(1, 2, true, 0, false);
      case 5: TQ_ATTN_K(1, 2, true, 1, false);
      case 6: TQ_ATTN_K(1, 2, true, 2, false);
      case 8: TQ_ATTN_K(2, 3, true, 0, false);
      case 9: TQ_ATTN_K(2, 3, true, 1, false);
      case 10: TQ_ATTN_K(2, 3, true, 2, false);
      case 13: TQ_ATTN_K(4, 4, true, 1, false);
      case 14: TQ_ATTN_K(4, 4, true, 2, false);
      default: TQ_ATTN_K(4, 4, true, 0, false);
    }
  }
  switch (kcb.b1) {
    case 1: TQ_ATTN_K(1, 1, false, 0, false);
    case 2: TQ_ATTN_K(2, 2, false, 0, false);
    case 3: TQ_ATTN_K(4, 3, false, 0, false);
    default: TQ_ATTN_K(8, 4, false, 0, false);
  }
#undef TQ_ATTN_K
}

cudaError_t launch_attn(const Dev& kcb, const Dev& vcb, const uint8_t* kc, const uint8_t* vc, int B, int Hq, int Hkv,
                        int64_t capacity, int64_t rows, const int32_t* seq_lens, const uint8_t* prep,
                        float scale_log2, float* parts, int nchunks, int tpc, cudaStream_t s) {
  const dim3 grid(nchunks, Hkv, B);
  switch (kcb.b1) {
    case 1: attn_v<1, 2>(vcb.b1, grid, s, kcb, vcb, kc, vc, Hq, Hkv, capacity, rows, seq_lens, prep, scale_log2, parts, tpc); break;
    case 2: attn_v<2, 3>(vcb.b1, grid, s, kcb, vcb, kc, vc, Hq, Hkv, capacity, rows, seq_lens, prep, scale_log2, parts, tpc); break;
    default: attn_v<4, 4>(vcb.b1, grid, s, kcb, vcb, kc, vc, Hq, Hkv, capacity, rows, seq_lens, prep, scale_log2, parts, tpc); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_merge(const Dev& vcb, const float* partials, int B, int Hq, int Hkv, int nparts,
                              int64_t group_stride, float* out, cudaStream_t s) {
  k_attn_merge<<<dim3(Hq, B), 128, 0, s>>>(vcb, partials, Hq, Hkv, nparts, group_stride, out);
  return cudaGetLastError();
}

}  // namespace tq
