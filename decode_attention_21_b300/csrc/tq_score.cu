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
#include <cuda_fp16.h>

#include "tq_internal.cuh"
#include "tq_mma.cuh"

namespace tq {

using namespace mma;

// ---------------------------------------------------------------------------
// Query preparation: one CTA per (kv head, head slot, sequence).  q' = Pi q,
// q'' = S q', the per-slot constants and the fp16 B fragments of every
// stage-1 virtual plane and of the sign plane.
//   header (floats): S1[4], S2[4], K1[4], K2[4]
//   fragments: [plane][kb][lane] uint2, plane nv = QJL, kb = 0..7, column
//   2*slot + piece (piece 0 = hi, 1 = lo).
// Element k = 2c + e (b0) / 2c + 8 + e (b1) of k-block kb is coordinate
// 32c + beta + 16e with beta = 2kb (b0) or 2kb + 1 (b1); its key bit sits at
// mantissa position 6 + (beta mod 4), whose factor 2^-(pos - 24) the query
// side absorbs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float dot32(const float* __restrict__ MT, const float* xs, int i, int qt) {
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

__global__ void __launch_bounds__(512) k_prep(const Dev cb, const float* __restrict__ q, int Hq, int Hkv,
                                              uint8_t* __restrict__ prep) {
  constexpr int d = 128;
  const int G = Hq / Hkv;
  const int kvh = blockIdx.x >> 2, slot = blockIdx.x & 3, b = blockIdx.y;
  const bool live = slot < G;
  // The scoring kernel that follows may start now: it only reads the key
  // cache (written before this kernel started) until it waits for this grid.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float sq[d], sq1[d], sq2[d], part[4][d], part2[4][d];
  __shared__ float red[4];
  const int tid = threadIdx.x;
  const int i = tid & 127, qt = tid >> 7;
  if (tid < d) sq[tid] = live ? q[((size_t)b * Hq + kvh * G + slot) * d + tid] : 0.f;
  __syncthreads();
  // q' = Pi q and q'' = (S Pi) q in the same pass
  part[qt][i] = dot32(cb.PiT, sq, i, qt);
  part2[qt][i] = dot32(cb.SPT, sq, i, qt);
  __syncthreads();
  if (tid < d) {
    sq1[tid] = (part[0][tid] + part[1][tid]) + (part[2][tid] + part[3][tid]);
    sq2[tid] = (part2[0][tid] + part2[1][tid]) + (part2[2][tid] + part2[3][tid]);
  }
  __syncthreads();
  const int nv = cb.nv;
  float cmax = 0.f, csum = 0.f;
  for (int v = 0; v < nv; ++v) {
    cmax = fmaxf(cmax, fabsf(cb.vcoef[v]));
    csum += cb.vcoef[v];
  }
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < 4) {
    // warp 0: max |stage-1 B|, 1: max |QJL B| (before the mantissa factor),
    // 2: sum q', 3: sum q''
    float v = 0.f;
    for (int k = lane; k < d; k += 32) {
      if (warp == 0) v = fmaxf(v, 2.f * cmax * fabsf(sq1[k]));
      else if (warp == 1) v = fmaxf(v, 2.f * fabsf(sq2[k]));
      else if (warp == 2) v += sq1[k];
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
  // largest mantissa factor 2^(24 - 6) = 2^18; keep |B| <= 2^14
  const float S1 = pow2_scale(red[0] * 262144.f, 16384.f), S2 = pow2_scale(red[1] * 262144.f, 16384.f);
  uint8_t* blk = prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(nv, d);
  float* hdr = reinterpret_cast<float*>(blk);
  if (tid == 0) {
    hdr[slot] = live ? S1 : 0.f;
    hdr[4 + slot] = live ? S2 : 0.f;
    hdr[8 + slot] = live ? csum * red[2] : 0.f;
    hdr[12 + slot] = live ? -red[3] : 0.f;
  }
  // fragments of the 8 lanes whose column belongs to this slot (g = 2 slot + piece)
  uint2* frag = reinterpret_cast<uint2*>(blk + kPrepHeader);
  const int total = (nv + 1) * 8 * 8;
  for (int e = tid; e < total; e += blockDim.x) {
    const int sub = e & 7, kb = (e >> 3) & 7, v = e >> 6;
    const int pc = sub >> 2, c = sub & 3;
    const int g = 2 * slot + pc;
    float vals[4] = {0.f, 0.f, 0.f, 0.f};
    if (live) {
      for (int t = 0; t < 4; ++t) {
        const int beta = 2 * kb + (t >> 1);
        const int k = 32 * c + beta + 16 * (t & 1);
        const float pf = (float)(1 << (18 - (beta & 3)));
        const float x = v < nv ? -2.f * cb.vcoef[v] * sq1[k] * pf / S1 : 2.f * sq2[k] * pf / S2;
        vals[t] = piece16(x, pc);
      }
    }
    frag[(v * 8 + kb) * 32 + g * 4 + c] = make_uint2(pack_half2(vals[0], vals[1]), pack_half2(vals[2], vals[3]));
  }
}

// ---------------------------------------------------------------------------
// QK for one 16-key tile: thread (g, c) gets the two inner products of keys
// g and g+8 for head slot c.
// ---------------------------------------------------------------------------
template <int NV, int P>
struct QK16 {
  uint2 bq[NV + 1][8];
  float S1, S2, K1, K2;

  __device__ __forceinline__ void load(const uint8_t* blk, int lane) {
    const float* hdr = reinterpret_cast<const float*>(blk);
    const uint2* frag = reinterpret_cast<const uint2*>(blk + kPrepHeader);
#pragma unroll
    for (int v = 0; v <= NV; ++v)
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) bq[v][kb] = frag[(v * 8 + kb) * 32 + lane];
    const int c = lane & 3;
    S1 = hdr[c];
    S2 = hdr[4 + c];
    K1 = hdr[8 + c];
    K2 = hdr[12 + c];
  }

  // Accumulates into chains kb % 2 (two independent accumulator chains per
  // call so consecutive MMAs do not wait on each other).
  __device__ __forceinline__ void plane(uint32_t xa, uint32_t xb, int v, float (&acc)[2][4]) const {
    uint32_t ra[16], rb[16];
    expand16(xa, ra);
    expand16(xb, rb);
#pragma unroll
    for (int kb = 0; kb < 8; ++kb)
      mma_f16(acc[kb & 1], ra[2 * kb], rb[2 * kb], ra[2 * kb + 1], rb[2 * kb + 1], bq[v][kb].x, bq[v][kb].y);
  }

  // wa, wb: the P plane words (column c) of keys g and g+8
  __device__ __forceinline__ void score(const uint32_t (&wa)[P], const uint32_t (&wb)[P], float& s1a, float& s1b,
                                        float& s2a, float& s2b) const {
    float acc1[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    // sign plane first: its chain runs alongside the stage-1 planes
    plane(wa[P - 1], wb[P - 1], NV, acc2);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      uint32_t xa = 0, xb = 0;
#pragma unroll
      for (int p = 0; p < P - 1; ++p)
        if (kOddMask[v] >> p & 1u) {
          xa ^= wa[p];
          xb ^= wb[p];
        }
      plane(xa, xb, v, acc1);
    }
    s1a = fmaf(S1, (acc1[0][0] + acc1[0][1]) + (acc1[1][0] + acc1[1][1]), K1);
    s1b = fmaf(S1, (acc1[0][2] + acc1[0][3]) + (acc1[1][2] + acc1[1][3]), K1);
    s2a = fmaf(S2, (acc2[0][0] + acc2[0][1]) + (acc2[1][0] + acc2[1][1]), K2);
    s2b = fmaf(S2, (acc2[0][2] + acc2[0][3]) + (acc2[1][2] + acc2[1][3]), K2);
  }

  // Two 16-key tiles at once, plane by plane, so their MMA chains interleave.
  __device__ __forceinline__ void score2(const uint32_t (&wa)[P], const uint32_t (&wb)[P], const uint32_t (&xa)[P],
                                         const uint32_t (&xb)[P], float& s1a, float& s1b, float& s2a, float& s2b,
                                         float& u1a, float& u1b, float& u2a, float& u2b) const {
    float acc1[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float bcc1[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float bcc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    plane(wa[P - 1], wb[P - 1], NV, acc2);
    plane(xa[P - 1], xb[P - 1], NV, bcc2);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      uint32_t pa = 0, pb = 0, qa = 0, qb = 0;
#pragma unroll
      for (int p = 0; p < P - 1; ++p)
        if (kOddMask[v] >> p & 1u) {
          pa ^= wa[p];
          pb ^= wb[p];
          qa ^= xa[p];
          qb ^= xb[p];
        }
      plane(pa, pb, v, acc1);
      plane(qa, qb, v, bcc1);
    }
    s1a = fmaf(S1, (acc1[0][0] + acc1[0][1]) + (acc1[1][0] + acc1[1][1]), K1);
    s1b = fmaf(S1, (acc1[0][2] + acc1[0][3]) + (acc1[1][2] + acc1[1][3]), K1);
    s2a = fmaf(S2, (acc2[0][0] + acc2[0][1]) + (acc2[1][0] + acc2[1][1]), K2);
    s2b = fmaf(S2, (acc2[0][2] + acc2[0][3]) + (acc2[1][2] + acc2[1][3]), K2);
    u1a = fmaf(S1, (bcc1[0][0] + bcc1[0][1]) + (bcc1[1][0] + bcc1[1][1]), K1);
    u1b = fmaf(S1, (bcc1[0][2] + bcc1[0][3]) + (bcc1[1][2] + bcc1[1][3]), K1);
    u2a = fmaf(S2, (bcc2[0][0] + bcc2[0][1]) + (bcc2[1][0] + bcc2[1][1]), K2);
    u2b = fmaf(S2, (bcc2[0][2] + bcc2[0][3]) + (bcc2[1][2] + bcc2[1][3]), K2);
  }
};

template <int P>
__device__ __forceinline__ void load_words(const uint32_t* __restrict__ rec, int c, uint32_t (&w)[P]) {
  const uint32_t* p = rec + c * P;
  if constexpr (P == 4) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (P == 2) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < P; ++i) w[i] = __ldg(p + i);
  }
}

// Key words and norms of one 16-key tile for thread (g, c).
template <int P>
struct KTile {
  uint32_t wa[P], wb[P];
  uint32_t na, nb;
  __device__ __forceinline__ void load(const uint32_t* recs, const uint32_t* nrm, int W, int64_t rowbase, int64_t ta,
                                       int64_t L, int c) {
    const int64_t tb = ta + 8;
    if (ta < L) {
      load_words<P>(recs + (rowbase + ta) * W, c, wa);
      na = __ldg(nrm + rowbase + ta);
    } else {
#pragma unroll
      for (int p = 0; p < P; ++p) wa[p] = 0;
      na = 0;
    }
    if (tb < L) {
      load_words<P>(recs + (rowbase + tb) * W, c, wb);
      nb = __ldg(nrm + rowbase + tb);
    } else {
#pragma unroll
      for (int p = 0; p < P; ++p) wb[p] = 0;
      nb = 0;
    }
  }
};

__device__ __forceinline__ float est_from(uint32_t nrm_bits, float s1, float s2, float kq) {
  const __half2 h = *reinterpret_cast<const __half2*>(&nrm_bits);
  return __low2float(h) * fmaf(__high2float(h) * kq, s2, s1);
}

// ---------------------------------------------------------------------------
// Logits: grid (chunks, Hkv, B), 4 warps; each warp scores 16-key tiles,
// prefetching its next tile while scoring the current one.
// ---------------------------------------------------------------------------
template <int NV, int P>
__global__ void __launch_bounds__(128, 3) k_logits(const Dev cb, const uint8_t* __restrict__ kcache, int Hq, int Hkv,
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
  QK16<NV, P> qk;
  qk.load(prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(NV, 128), lane);
  const uint32_t* recs = reinterpret_cast<const uint32_t*>(kcache);
  const uint32_t* nrm = reinterpret_cast<const uint32_t*>(kcache + norm_offset(cb, cache_rows));
  const int64_t rowbase = ((int64_t)b * Hkv + kvh) * capacity;
  const float kq = cb.qjl_const;
  const int W = cb.W;
  float* out = logits + ((size_t)b * Hq + (size_t)kvh * G + c) * capacity;
  KTile<P> cur, nxt;
  int64_t tile = tile0 + warp;
  cur.load(recs, nrm, W, rowbase, tile * 16 + g, L, c);
  for (; tile < tend; tile += 4) {
    const int64_t tn = tile + 4;
    if (tn < tend) nxt.load(recs, nrm, W, rowbase, tn * 16 + g, L, c);
    float s1a, s1b, s2a, s2b;
    qk.score(cur.wa, cur.wb, s1a, s1b, s2a, s2b);
    const int64_t ta = tile * 16 + g, tb = ta + 8;
    if (c < G) {
      if (ta < L) out[ta] = est_from(cur.na, s1a, s2a, kq);
      if (tb < L) out[tb] = est_from(cur.nb, s1b, s2b, kq);
    }
    cur = nxt;
  }
}

// ---------------------------------------------------------------------------
// Logits with bulk-copy staging: the CTA's whole chunk of key records and
// norms (up to kStageTiles x kMaxStages tiles) is requested at once with
// cp.async.bulk into shared memory, one mbarrier per stage of kStageTiles
// tiles, and the warps score each stage as it lands.  Requires capacity to be
// a multiple of 16 (every copied tile lies inside its sequence's rows).
// ---------------------------------------------------------------------------
namespace {
constexpr int kStageTiles = 8;
constexpr int kMaxStages = 8;
constexpr long long kWaitLimit = 1ll << 26;

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  for (long long i = 0; i < kWaitLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
}  // namespace

template <int NV, int P>
__global__ void __launch_bounds__(128) k_logits_tma(const Dev cb, const uint8_t* __restrict__ kcache, int Hq, int Hkv,
                                                    int64_t capacity, int64_t cache_rows,
                                                    const int32_t* __restrict__ seq_lens,
                                                    const uint8_t* __restrict__ prep, float* __restrict__ logits,
                                                    int tiles_per_cta, int* __restrict__ status) {
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ __align__(8) uint64_t bars[kMaxStages];
  constexpr int RB = 16 * P;                 // record bytes at d = 128
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int G = Hq / Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t L = seq_lens[b];
  const int64_t ntiles = (L + 15) / 16;
  const int64_t tile0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t tend = min(tile0 + tiles_per_cta, ntiles);
  if (tile0 >= tend) return;
  const int nt = (int)(tend - tile0);
  const int nstages = (nt + kStageTiles - 1) / kStageTiles;
  uint8_t* srec = sm;
  uint8_t* snrm = sm + (size_t)tiles_per_cta * 16 * RB;
  const int64_t rowbase = ((int64_t)b * Hkv + kvh) * capacity;
  const uint8_t* grec = kcache + (rowbase + tile0 * 16) * RB;
  const uint8_t* gnrm = kcache + norm_offset(cb, cache_rows) + (rowbase + tile0 * 16) * 4;
  if (tid == 0) {
    for (int st = 0; st < nstages; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bars[st])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int st = 0; st < nstages; ++st) {
      const int t_a = st * kStageTiles, t_n = min(kStageTiles, nt - t_a);
      const uint32_t rb = (uint32_t)(t_n * 16 * RB), nb = (uint32_t)(t_n * 16 * 4);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&bars[st])), "r"(rb + nb)
                   : "memory");
      bulk_g2s(su32(srec + (size_t)t_a * 16 * RB), grec + (size_t)t_a * 16 * RB, rb, su32(&bars[st]));
      bulk_g2s(su32(snrm + (size_t)t_a * 16 * 4), gnrm + (size_t)t_a * 16 * 4, nb, su32(&bars[st]));
    }
  }
  // query fragments come from the preceding prep grid (launched as its
  // programmatic dependent): wait for it only now, after the copies are in flight
  asm volatile("griddepcontrol.wait;" ::: "memory");
  QK16<NV, P> qk;
  qk.load(prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(NV, 128), lane);
  __syncthreads();
  const float kq = cb.qjl_const;
  float* out = logits + ((size_t)b * Hq + (size_t)kvh * G + c) * capacity;
  bool ok = true;
  auto tile_words = [&](int lt, uint32_t(&wa)[P], uint32_t(&wb)[P], uint32_t& na, uint32_t& nb) {
    const uint8_t* ra = srec + ((size_t)lt * 16 + g) * RB + c * P * 4;
    const uint8_t* rbp = ra + 8 * RB;
    if constexpr (P == 4) {
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
    na = reinterpret_cast<const uint32_t*>(snrm)[lt * 16 + g];
    nb = reinterpret_cast<const uint32_t*>(snrm)[lt * 16 + g + 8];
    const int64_t ta = (tile0 + lt) * 16 + g;
    if (ta >= L) {
#pragma unroll
      for (int p = 0; p < P; ++p) wa[p] = 0;
    }
    if (ta + 8 >= L) {
#pragma unroll
      for (int p = 0; p < P; ++p) wb[p] = 0;
    }
  };
  auto emit = [&](int lt, uint32_t na, uint32_t nb, float s1a, float s1b, float s2a, float s2b) {
    const int64_t ta = (tile0 + lt) * 16 + g, tb = ta + 8;
    if (c < G) {
      if (ta < L) out[ta] = est_from(na, s1a, s2a, kq);
      if (tb < L) out[tb] = est_from(nb, s1b, s2b, kq);
    }
  };
  for (int st = 0; st < nstages && ok; ++st) {
    if (!bar_wait(su32(&bars[st]), 0)) {
      ok = false;
      break;
    }
    const int t_a = st * kStageTiles, t_e = min(t_a + kStageTiles, nt);
    // two tiles per iteration (warp, warp + 4) for independent MMA chains
    for (int lt = t_a + warp; lt < t_e; lt += 8) {
      const int lt2 = lt + 4;
      uint32_t wa[P], wb[P], xa[P], xb[P], na, nb, ma = 0, mb = 0;
      tile_words(lt, wa, wb, na, nb);
      const bool two = lt2 < t_e;
      if (two) {
        tile_words(lt2, xa, xb, ma, mb);
      } else {
#pragma unroll
        for (int p = 0; p < P; ++p) xa[p] = xb[p] = 0;
      }
      float s1a, s1b, s2a, s2b, u1a, u1b, u2a, u2b;
      qk.score2(wa, wb, xa, xb, s1a, s1b, s2a, s2b, u1a, u1b, u2a, u2b);
      emit(lt, na, nb, s1a, s1b, s2a, s2b);
      if (two) emit(lt2, ma, mb, u1a, u1b, u2a, u2b);
    }
  }
  if (!ok) {
    if (tid == 0) atomicExch(status, 2);
    // let the remaining copies land (bounded) before the CTA's shared memory is released
    for (int st = 0; st < nstages; ++st) bar_wait(su32(&bars[st]), 0);
  }
}

int logits_tma_max_tiles() { return kStageTiles * kMaxStages; }

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

  if (tile0 + warp < tend) {
    QK16<NVK, PK> qk;
    qk.load(prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(NVK, 128), lane);
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
    for (; tile < tend; tile += 4) {
      const int64_t tn = tile + 4;
      if (tn < tend) {
        knxt.load(krec, knrm, KW, rowbase, tn * 16 + g, L, c);
        vnxt.load(vrec, vnrm, VW, rowbase, tn * 16, L, g, c);
      }
      const int64_t ta = tile * 16 + g, tb = ta + 8;
      float s1a, s1b, s2a, s2b;
      qk.score(kcur.wa, kcur.wb, s1a, s1b, s2a, s2b);
      // scores in log2 units
      const float sa = ta < L ? est_from(kcur.na, s1a, s2a, kq) * scale_log2 : -INFINITY;
      const float sb = tb < L ? est_from(kcur.nb, s1b, s2b, kq) * scale_log2 : -INFINITY;
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
        const uint32_t b0 = pack_half2(piece16(cu * w0, pc), piece16(cu * w1, pc));
        const uint32_t b1 = pack_half2(piece16(cu * w8, pc), piece16(cu * w9, pc));
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
        expand16(__byte_perm(x[0], x[1], vsel), r01);
        expand16(__byte_perm(x[2], x[3], vsel), r89);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          mma_f16(acc[mt], r01[2 * mt], r01[2 * mt + 1], r89[2 * mt], r89[2 * mt + 1], b0, b1);
      }
      kcur = knxt;
      vcur = vnxt;
    }
  }
  // this warp's partial: head slot c, coordinates 16g + 2mt (+1);
  // acc = C0 * wsum + 2^(24 - pos) * D with pos = 6 + (beta mod 4)
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
    const float f0 = (float)(1 << (18 - (b0 & 3))), f1 = (float)(1 << (18 - (b1 & 3)));
    ph[2 + 16 * g + b0] = fmaf(f0, acc[mt][0] + acc[mt][1], c0 * wsum);
    ph[2 + 16 * g + b1] = fmaf(f1, acc[mt][2] + acc[mt][3], c0 * wsum);
  }
}

// Merge the split partials of one (b, query head) and rotate back once:
// M = max m_p, o_rot = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,
// out = Pi_v^T o_rot.
__global__ void __launch_bounds__(128) k_attn_merge(const Dev vcb, const float* __restrict__ partials, int Hq, int Hkv,
                                                    int nparts, float* __restrict__ out) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int G = Hq / Hkv, kvh = h / G, slot = h % G;
  constexpr int d = 128;
  __shared__ float so[d];
  const float* base = partials + ((size_t)b * Hkv + kvh) * nparts * partial_floats(d) + slot * (2 + d);
  const int i = threadIdx.x;
  float M = -INFINITY;
  for (int p = 0; p < nparts; ++p) M = fmaxf(M, base[(size_t)p * partial_floats(d)]);
  float Lsum = 0.f, a = 0.f;
  if (M != -INFINITY) {
    for (int p = 0; p < nparts; ++p) {
      const float* ph = base + (size_t)p * partial_floats(d);
      const float mp = ph[0];
      if (mp == -INFINITY) continue;
      const float w = exp2f(mp - M);
      Lsum = fmaf(w, ph[1], Lsum);
      a = fmaf(w, ph[2 + i], a);
    }
  }
  so[i] = Lsum > 0.f ? a / Lsum : 0.f;
  __syncthreads();
  float o = 0.f;
  for (int k = 0; k < d; ++k) o = fmaf(vcb.Pi[(size_t)k * d + i], so[k], o);
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

cudaError_t launch_prep(const Dev& cb, const float* q, int B, int Hq, int Hkv, uint8_t* prep, cudaStream_t s) {
  k_prep<<<dim3(Hkv * 4, B), 512, 0, s>>>(cb, q, Hq, Hkv, prep);
  return cudaGetLastError();
}

cudaError_t launch_logits(const Dev& cb, const uint8_t* kc, int B, int Hq, int Hkv, int64_t capacity,
                          int64_t rows, const int32_t* seq_lens, const uint8_t* prep, float* logits, int nchunks,
                          int tpc, cudaStream_t s) {
  const dim3 grid(nchunks, Hkv, B);
  switch (cb.b1) {
    case 1: k_logits<1, 2><<<grid, 128, 0, s>>>(cb, kc, Hq, Hkv, capacity, rows, seq_lens, prep, logits, tpc); break;
    case 2: k_logits<2, 3><<<grid, 128, 0, s>>>(cb, kc, Hq, Hkv, capacity, rows, seq_lens, prep, logits, tpc); break;
    default: k_logits<4, 4><<<grid, 128, 0, s>>>(cb, kc, Hq, Hkv, capacity, rows, seq_lens, prep, logits, tpc); break;
  }
  return cudaGetLastError();
}

template <int NV, int P>
static cudaError_t logits_tma_t(const Dev& cb, const uint8_t* kc, int B, int Hq, int Hkv, int64_t capacity, int64_t rows,
                                const int32_t* seq_lens, const uint8_t* prep, float* logits, int nchunks, int tpc,
                                int* status, cudaStream_t s) {
  const size_t smem = (size_t)tpc * 16 * (16 * P + 4);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_logits_tma<NV, P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)((size_t)logits_tma_max_tiles() * 16 * (16 * 4 + 4)));
    if (e != cudaSuccess) return e;
    configured = true;
  }
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
  return cudaLaunchKernelEx(&cfg, k_logits_tma<NV, P>, cb, kc, Hq, Hkv, capacity, rows, seq_lens, prep, logits, tpc,
                            status);
}

cudaError_t launch_logits_tma(const Dev& cb, const uint8_t* kc, int B, int Hq, int Hkv, int64_t capacity, int64_t rows,
                              const int32_t* seq_lens, const uint8_t* prep, float* logits, int nchunks, int tpc,
                              int* status, cudaStream_t s) {
  switch (cb.b1) {
    case 1: return logits_tma_t<1, 2>(cb, kc, B, Hq, Hkv, capacity, rows, seq_lens, prep, logits, nchunks, tpc, status, s);
    case 2: return logits_tma_t<2, 3>(cb, kc, B, Hq, Hkv, capacity, rows, seq_lens, prep, logits, nchunks, tpc, status, s);
    default: return logits_tma_t<4, 4>(cb, kc, B, Hq, Hkv, capacity, rows, seq_lens, prep, logits, nchunks, tpc, status, s);
  }
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

cudaError_t launch_attn_merge(const Dev& vcb, const float* partials, int B, int Hq, int Hkv, int nparts, float* out,
                              cudaStream_t s) {
  k_attn_merge<<<dim3(Hq, B), 128, 0, s>>>(vcb, partials, Hq, Hkv, nparts, out);
  return cudaGetLastError();
}

}  // namespace tq
