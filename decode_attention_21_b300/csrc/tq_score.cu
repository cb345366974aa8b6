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
// XOR-products of its code planes, yhat = sum_v coef_v * s_v with
// s_v = (-1)^(xor of the planes in subset v) (a Walsh-Hadamard expansion of
// the centroid table).  Each +-1 pattern is expanded from a packed word into
// fp16 tensor-core operands with one shift and one logic op per two
// coordinates, and the query side (fp32 split into fp16 hi + lo, scaled by a
// power of two) is the other operand, so the contraction runs on the tensor
// cores with fp32 accumulation.  The G <= 4 query heads of a GQA group fill
// the 8 columns of one m16n8k16 tile as (head, hi/lo) pairs.
#include <cuda_fp16.h>

#include "tq_internal.cuh"

namespace tq {

namespace {

constexpr unsigned kFull = 0xffffffffu;

// Odd subsets of the code planes (bit p <-> plane p) in increasing order; the
// first 2^(b'-1) entries are exactly the odd subsets of b' planes.
__device__ constexpr uint32_t kOddMask[8] = {1u, 2u, 4u, 7u, 8u, 11u, 13u, 14u};

// +-1 fp16 pair from bits beta (low half) and beta + 16 (high half) of w:
// bit set -> -1, clear -> +1.
__device__ __forceinline__ uint32_t pm1(uint32_t w, int beta) {
  return ((w << (15 - beta)) & 0x80008000u) | 0x3C003C00u;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
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
__device__ __forceinline__ float piece(float x, int which) {
  const float hi = __half2float(__float2half_rn(x));
  return which == 0 ? hi : x - hi;
}

__device__ __forceinline__ float pow2_ceil_scale(float amax) {
  // power of two s with amax / s <= 64
  if (!(amax > 0.f)) return 1.f;
  int e;
  frexpf(amax / 64.f, &e);
  return ldexpf(1.f, e);
}

}  // namespace

// ---------------------------------------------------------------------------
// Query preparation: one CTA per (sequence b, kv head).  q' = Pi q,
// q'' = S q', then the tensor-core B fragments of every virtual plane and of
// the sign plane in register order.  MMA k-index 2c + 8h + e of k-block kb
// maps to coordinate 32 (c + 4 (kb / 8)) + 2 (kb % 8) + h + 16 e.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_prep(const Dev cb, const float* __restrict__ q, int Hq, int Hkv,
                                              uint8_t* __restrict__ prep) {
  const int d = cb.d;
  const int G = Hq / Hkv;
  const int kvh = blockIdx.x, b = blockIdx.y;
  __shared__ float sq[4][256];
  __shared__ float sq1[4][256];
  __shared__ float sq2[4][256];
  __shared__ float sscale[8];
  const int tid = threadIdx.x;
  for (int e = tid; e < 4 * d; e += blockDim.x) {
    const int h = e / d, i = e % d;
    sq[h][i] = h < G ? q[((size_t)b * Hq + kvh * G + h) * d + i] : 0.f;
  }
  __syncthreads();
  for (int e = tid; e < 4 * d; e += blockDim.x) {
    const int h = e / d, i = e % d;
    float acc = 0.f;
    for (int j = 0; j < d; ++j) acc = fmaf(cb.PiT[(size_t)j * d + i], sq[h][j], acc);
    sq1[h][i] = acc;
  }
  __syncthreads();
  for (int e = tid; e < 4 * d; e += blockDim.x) {
    const int h = e / d, j = e % d;
    float acc = 0.f;
    for (int i = 0; i < d; ++i) acc = fmaf(cb.ST[(size_t)i * d + j], sq1[h][i], acc);
    sq2[h][j] = acc;
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  float cmax = 0.f;
  for (int v = 0; v < cb.nv; ++v) cmax = fmaxf(cmax, fabsf(cb.vcoef[v]));
  if (warp < 8) {
    const int h = warp & 3;
    const float* src = warp < 4 ? sq1[h] : sq2[h];
    float m = 0.f;
    for (int i = lane; i < d; i += 32) m = fmaxf(m, fabsf(src[i]));
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    if (lane == 0) sscale[warp] = pow2_ceil_scale(warp < 4 ? m * cmax : m);
  }
  __syncthreads();
  uint8_t* blk = prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(cb.nv, d);
  float* hdr = reinterpret_cast<float*>(blk);
  if (tid < 8) hdr[tid] = sscale[tid];
  uint2* frag = reinterpret_cast<uint2*>(blk + kPrepHeader);
  const int KB = d / 16;
  const int total = (cb.nv + 1) * KB * 32;
  for (int e = tid; e < total; e += blockDim.x) {
    const int ln = e & 31, kb = (e >> 5) % KB, v = (e >> 5) / KB;
    const int g = ln >> 2, c = ln & 3;
    const int head = g >> 1, pc = g & 1;
    const int base = 32 * (c + 4 * (kb / 8)) + 2 * (kb % 8);
    float vals[4] = {0.f, 0.f, 0.f, 0.f};
    const int coords[4] = {base, base + 16, base + 1, base + 17};
    if (head < G) {
      for (int t = 0; t < 4; ++t) {
        float x;
        if (v < cb.nv)
          x = cb.vcoef[v] * sq1[head][coords[t]] / sscale[head];
        else
          x = -sq2[head][coords[t]] / sscale[4 + head];
        vals[t] = piece(x, pc);
      }
    }
    frag[e] = make_uint2(pack_half2(vals[0], vals[1]), pack_half2(vals[2], vals[3]));
  }
}

// ---------------------------------------------------------------------------
// Shared QK step for one 16-key tile: thread (g, c) returns the estimates of
// keys t0+g and t0+g+8 for head slot c.
// ---------------------------------------------------------------------------
template <int NV, int P>
struct QK {
  uint2 bq[NV][8];
  uint2 bs[8];
  float sc1, sc2;

  __device__ __forceinline__ void load(const Dev& cb, const uint8_t* blk, int lane) {
    const float* hdr = reinterpret_cast<const float*>(blk);
    const uint2* frag = reinterpret_cast<const uint2*>(blk + kPrepHeader);
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) bq[v][kb] = frag[(v * 8 + kb) * 32 + lane];
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) bs[kb] = frag[(NV * 8 + kb) * 32 + lane];
    const int c = lane & 3;
    sc1 = hdr[c];
    sc2 = hdr[4 + c];
  }

  // wa, wb: the P plane words (column c) of keys g and g+8
  __device__ __forceinline__ void score(const uint32_t (&wa)[P], const uint32_t (&wb)[P], float& s1a, float& s1b,
                                        float& s2a, float& s2b) const {
    float acc1[4] = {0.f, 0.f, 0.f, 0.f};
    float acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      uint32_t xa = 0, xb = 0;
#pragma unroll
      for (int p = 0; p < P - 1; ++p)
        if (kOddMask[v] >> p & 1u) {
          xa ^= wa[p];
          xb ^= wb[p];
        }
#pragma unroll
      for (int kb = 0; kb < 8; ++kb)
        mma16816(acc1, pm1(xa, 2 * kb), pm1(xb, 2 * kb), pm1(xa, 2 * kb + 1), pm1(xb, 2 * kb + 1), bq[v][kb].x,
                 bq[v][kb].y);
    }
#pragma unroll
    for (int kb = 0; kb < 8; ++kb)
      mma16816(acc2, pm1(wa[P - 1], 2 * kb), pm1(wb[P - 1], 2 * kb), pm1(wa[P - 1], 2 * kb + 1),
               pm1(wb[P - 1], 2 * kb + 1), bs[kb].x, bs[kb].y);
    s1a = (acc1[0] + acc1[1]) * sc1;
    s1b = (acc1[2] + acc1[3]) * sc1;
    s2a = (acc2[0] + acc2[1]) * sc2;
    s2b = (acc2[2] + acc2[3]) * sc2;
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

// ---------------------------------------------------------------------------
// Logits: grid (chunks, Hkv, B), 4 warps; each warp scores 16-key tiles.
// ---------------------------------------------------------------------------
template <int NV, int P>
__global__ void __launch_bounds__(128) k_logits(const Dev cb, const uint8_t* __restrict__ kcache, int Hq, int Hkv,
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
  if (tile0 >= ntiles) return;
  QK<NV, P> qk;
  qk.load(cb, prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(NV, 128), lane);
  const uint32_t* recs = reinterpret_cast<const uint32_t*>(kcache);
  const uint32_t* nrm = reinterpret_cast<const uint32_t*>(kcache + norm_offset(cb, cache_rows));
  const int64_t rowbase = ((int64_t)b * Hkv + kvh) * capacity;
  const float kq = cb.qjl_const;
  float* out = logits + ((size_t)b * Hq + (size_t)kvh * G + c) * capacity;
  const int64_t tend = min(tile0 + tiles_per_cta, ntiles);
  for (int64_t tile = tile0 + warp; tile < tend; tile += 4) {
    const int64_t ta = tile * 16 + g, tb = ta + 8;
    uint32_t wa[P], wb[P];
    uint32_t na = 0, nb = 0;
    if (ta < L) {
      load_words<P>(recs + (rowbase + ta) * cb.W, c, wa);
      na = __ldg(nrm + rowbase + ta);
    } else {
#pragma unroll
      for (int p = 0; p < P; ++p) wa[p] = 0;
    }
    if (tb < L) {
      load_words<P>(recs + (rowbase + tb) * cb.W, c, wb);
      nb = __ldg(nrm + rowbase + tb);
    } else {
#pragma unroll
      for (int p = 0; p < P; ++p) wb[p] = 0;
    }
    float s1a, s1b, s2a, s2b;
    qk.score(wa, wb, s1a, s1b, s2a, s2b);
    const __half2 ha = *reinterpret_cast<const __half2*>(&na);
    const __half2 hb = *reinterpret_cast<const __half2*>(&nb);
    const float la = __low2float(ha) * fmaf(__high2float(ha) * kq, s2a, s1a);
    const float lb = __low2float(hb) * fmaf(__high2float(hb) * kq, s2b, s1b);
    if (c < G) {
      if (ta < L) out[ta] = la;
      if (tb < L) out[tb] = lb;
    }
  }
}

// ---------------------------------------------------------------------------
// Fused decode attention: QK as above, online softmax per head slot, and the
// weighted value sum  acc[i] = sum_t p_t n_v,t yhat_v,t[i]  in the rotated
// domain, again on the tensor cores: A = value bit patterns (16 coordinates
// x 16 tokens, two tokens per fp16 pair), B = p_t n_v,t (hi/lo) times the
// value codebook's coefficients.  Thread (g, c) owns head slot c and
// coordinates 16g .. 16g+15 of the accumulator.
// ---------------------------------------------------------------------------
template <int NVK, int PK, int NVV, int PV>
__global__ void __launch_bounds__(128) k_attn(const Dev kcb, const Dev vcb, const uint8_t* __restrict__ kcache,
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

  float m_run = -INFINITY, l_run = 0.f;
  float acc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;

  if (tile0 < ntiles) {
    QK<NVK, PK> qk;
    qk.load(kcb, prep + ((size_t)b * Hkv + kvh) * prep_block_bytes(NVK, 128), lane);
    float vcoef[NVV];
#pragma unroll
    for (int u = 0; u < NVV; ++u) vcoef[u] = vcb.vcoef[u];
    const uint32_t* krec = reinterpret_cast<const uint32_t*>(kcache);
    const uint32_t* knrm = reinterpret_cast<const uint32_t*>(kcache + norm_offset(kcb, cache_rows));
    const uint32_t* vrec = reinterpret_cast<const uint32_t*>(vcache);
    const __half* vnrm = reinterpret_cast<const __half*>(vcache + norm_offset(vcb, cache_rows));
    const int64_t rowbase = ((int64_t)b * Hkv + kvh) * capacity;
    const float kq = kcb.qjl_const;
    // value tokens used by this thread in a tile: 2c, 2c+1, 2c+8, 2c+9; word g/2
    const int vword = g >> 1;
    const uint32_t vsel = (g & 1) ? 0x7632u : 0x5410u;
    const int hh = g >> 1, pc = g & 1;    // B-fragment column: head slot, piece
    const int src0 = (2 * c) * 4 + hh, src1 = (2 * c + 1) * 4 + hh;

    for (int64_t tile = tile0 + warp; tile < tend; tile += 4) {
      const int64_t t0 = tile * 16;
      const int64_t ta = t0 + g, tb = ta + 8;
      uint32_t wa[PK], wb[PK];
      uint32_t na = 0, nb = 0;
      if (ta < L) {
        load_words<PK>(krec + (rowbase + ta) * kcb.W, c, wa);
        na = __ldg(knrm + rowbase + ta);
      } else {
#pragma unroll
        for (int p = 0; p < PK; ++p) wa[p] = 0;
      }
      if (tb < L) {
        load_words<PK>(krec + (rowbase + tb) * kcb.W, c, wb);
        nb = __ldg(knrm + rowbase + tb);
      } else {
#pragma unroll
        for (int p = 0; p < PK; ++p) wb[p] = 0;
      }
      // value words for this thread's four tokens
      uint32_t vw[4][PV];
      float vn[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t t = t0 + 2 * c + (j & 1) + 8 * (j >> 1);
        if (t < L) {
#pragma unroll
          for (int p = 0; p < PV; ++p) vw[j][p] = __ldg(vrec + (rowbase + t) * vcb.W + vword * PV + p);
        } else {
#pragma unroll
          for (int p = 0; p < PV; ++p) vw[j][p] = 0;
        }
      }
      if (ta < L) vn[0] = __half2float(vnrm[rowbase + ta]);
      if (tb < L) vn[1] = __half2float(vnrm[rowbase + tb]);

      float s1a, s1b, s2a, s2b;
      qk.score(wa, wb, s1a, s1b, s2a, s2b);
      const __half2 ha = *reinterpret_cast<const __half2*>(&na);
      const __half2 hb = *reinterpret_cast<const __half2*>(&nb);
      // scores in log2 units
      float sa = ta < L ? __low2float(ha) * fmaf(__high2float(ha) * kq, s2a, s1a) * scale_log2 : -INFINITY;
      float sb = tb < L ? __low2float(hb) * fmaf(__high2float(hb) * kq, s2b, s1b) * scale_log2 : -INFINITY;
      float mx = fmaxf(sa, sb);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
      const float pa = sa == -INFINITY ? 0.f : exp2f(sa - m_new);
      const float pb = sb == -INFINITY ? 0.f : exp2f(sb - m_new);
      float ps = pa + pb;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) ps += __shfl_xor_sync(kFull, ps, o);
      l_run = l_run * alpha + ps;
      m_run = m_new;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] *= alpha;
      // weights of tokens g and g+8 for head slot c, gathered into B-fragment order
      const float wA = pa * vn[0], wB = pb * vn[1];
      const float w0 = __shfl_sync(kFull, wA, src0);
      const float w1 = __shfl_sync(kFull, wA, src1);
      const float w8 = __shfl_sync(kFull, wB, src0);
      const float w9 = __shfl_sync(kFull, wB, src1);
#pragma unroll
      for (int u = 0; u < NVV; ++u) {
        const float cu = vcoef[u];
        const uint32_t b0 = pack_half2(piece(cu * w0, pc), piece(cu * w1, pc));
        const uint32_t b1 = pack_half2(piece(cu * w8, pc), piece(cu * w9, pc));
        uint32_t x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r = 0;
#pragma unroll
          for (int p = 0; p < PV; ++p)
            if (kOddMask[u] >> p & 1u) r ^= vw[j][p];
          x[j] = r;
        }
        const uint32_t w01 = __byte_perm(x[0], x[1], vsel);
        const uint32_t w89 = __byte_perm(x[2], x[3], vsel);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          mma16816(acc[mt], pm1(w01, 2 * mt), pm1(w01, 2 * mt + 1), pm1(w89, 2 * mt), pm1(w89, 2 * mt + 1), b0, b1);
      }
    }
  }
  // write this warp's partial: head slot c, coordinates 16g + 2mt (+1)
  const int nchunks = gridDim.x;
  float* part = partials + ((((size_t)b * Hkv + kvh) * nchunks + blockIdx.x) * kAttnWarps + warp) * partial_floats(128);
  float* ph = part + c * (2 + 128);
  if (g == 0) {
    ph[0] = m_run;
    ph[1] = l_run;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    ph[2 + 16 * g + 2 * mt] = acc[mt][0] + acc[mt][1];
    ph[2 + 16 * g + 2 * mt + 1] = acc[mt][2] + acc[mt][3];
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
  k_prep<<<dim3(Hkv, B), 256, 0, s>>>(cb, q, Hq, Hkv, prep);
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
