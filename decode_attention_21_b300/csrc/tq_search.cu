// Top-k inner-product search over a compressed database ([xujun] note-189244,
// 常见问题 on vector search; [cnyes] hao.cnyes.com "TurboQuant"): every query
// scores every database row with the unbiased estimator
//   est(q, x) = n ( <q', yhat> + gamma sqrt(pi/2)/m <q'', sigma> )
// and keeps the k best rows (decreasing score, ties to the smaller id).
//
// Same operand scheme as the attention logits (tq_score.cu): the score is a
// per-query constant plus masked sums of the query side over the database's
// bit planes, computed on the tensor cores (fp16 m16n8k16, subnormal 0/1
// operands from the packed words, query side split into fp16 hi + lo).
//   * prep: one CTA per (group of 4 queries, query slot): q' = Pi q,
//     q'' = S q' (d = 256), per-slot constants and B fragments.
//   * scan: CTA = 4 query groups x 2 coordinate halves (8 warps).  Each warp
//     keeps the B fragments of its group and half in registers and streams
//     16-row database tiles; the two halves of a group add their partial
//     accumulators through shared memory, and the first half updates a
//     per-query top-k list in shared memory (a candidate enters only if it
//     beats the current k-th score).
//   * the database is split into chunks (a second grid dimension) so that
//     the scan fills whole waves of resident CTAs; a merge kernel combines
//     the per-chunk lists.
#include <cuda_fp16.h>

#include <algorithm>

#include "tq_internal.cuh"

namespace tq {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kD = 256;
constexpr int kMaxK = 32;
constexpr int kRound = 4;   // 16-row tiles per exchange between the two coordinate halves
constexpr int kMaxChunks = 16;
// Resident scan CTAs per SM (registers): 2 for databases of up to 3 planes.
__host__ __device__ constexpr int search_ctas_per_sm(int P) { return P <= 3 ? 2 : 1; }
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

__device__ __forceinline__ float piece16(float x, int which) {
  const float hi = __half2float(__float2half_rn(x));
  return which == 0 ? hi : x - hi;
}

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

__device__ __forceinline__ float pow2_scale(float amax, float target) {
  if (!(amax > 0.f)) return 1.f;
  int e;
  frexpf(amax / target, &e);
  return ldexpf(1.f, e);
}

__device__ __forceinline__ float dot64(const float* __restrict__ MT, const float* xs, int i, int qt) {
  const float* col = MT + (size_t)(64 * qt) * kD + i;
  float m[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) m[j] = __ldg(col + (size_t)j * kD);
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 64; ++j) acc = fmaf(m[j], xs[64 * qt + j], acc);
  return acc;
}

}  // namespace

// Bytes of one query group's prep block (header + fragments).
__host__ __device__ inline int64_t search_block_bytes(int nv) { return kPrepHeader + (int64_t)(nv + 1) * 16 * 32 * 8; }

// Fragment layout: [plane][kb (16)][lane] uint2; k-block kb covers word
// c + 4 (kb / 8) of thread c, bit positions beta = 2 (kb % 8) (+1 for b1).
// With a query map (qmap, *qcount), query slot v of the scan is query
// qmap[v] for v < *qcount, and the rest of the grid does nothing.
__global__ void __launch_bounds__(1024) k_search_prep(const Dev cb, const float* __restrict__ q, int nq, int d_in,
                                                      uint8_t* __restrict__ prep, const int32_t* __restrict__ qmap,
                                                      const unsigned* __restrict__ qcount) {
  const int grp = blockIdx.x, slot = blockIdx.y;
  const int v = grp * 4 + slot;
  const int nv_live = qmap ? (int)min(*qcount, (unsigned)nq) : nq;
  if (grp * 4 >= nv_live) return;           // no live query in this group
  const bool live = v < nv_live;
  const int qi = live && qmap ? qmap[v] : v;
  __shared__ float sq[kD], sq1[kD], sq2[kD], part[4][kD], part2[4][kD];
  __shared__ float red[4];
  const int tid = threadIdx.x;
  const int i = tid & 255, qt = tid >> 8;
  if (tid < kD) sq[tid] = (live && tid < d_in) ? q[(size_t)qi * d_in + tid] : 0.f;
  __syncthreads();
  part[qt][i] = dot64(cb.PiT, sq, i, qt);
  part2[qt][i] = dot64(cb.SPT, sq, i, qt);
  __syncthreads();
  if (tid < kD) {
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
    float v = 0.f;
    for (int k = lane; k < kD; k += 32) {
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
  const float S1 = pow2_scale(red[0] * 262144.f, 16384.f), S2 = pow2_scale(red[1] * 262144.f, 16384.f);
  uint8_t* blk = prep + (size_t)grp * search_block_bytes(nv);
  float* hdr = reinterpret_cast<float*>(blk);
  if (tid == 0) {
    hdr[slot] = live ? S1 : 0.f;
    hdr[4 + slot] = live ? S2 : 0.f;
    hdr[8 + slot] = live ? csum * red[2] : 0.f;
    hdr[12 + slot] = live ? -red[3] : 0.f;
  }
  uint2* frag = reinterpret_cast<uint2*>(blk + kPrepHeader);
  const int total = (nv + 1) * 16 * 8;
  for (int e = tid; e < total; e += blockDim.x) {
    const int sub = e & 7, kb = (e >> 3) & 15, v = e >> 7;
    const int pc = sub >> 2, c = sub & 3;
    const int g = 2 * slot + pc;
    float vals[4] = {0.f, 0.f, 0.f, 0.f};
    if (live) {
      for (int t = 0; t < 4; ++t) {
        const int beta = 2 * (kb & 7) + (t >> 1);
        const int k = 32 * (c + 4 * (kb >> 3)) + beta + 16 * (t & 1);
        const float pf = (float)(1 << (18 - (beta & 3)));
        const float x = v < nv ? -2.f * cb.vcoef[v] * sq1[k] * pf / S1 : 2.f * sq2[k] * pf / S2;
        vals[t] = piece16(x, pc);
      }
    }
    frag[(v * 16 + kb) * 32 + g * 4 + c] = make_uint2(pack_half2(vals[0], vals[1]), pack_half2(vals[2], vals[3]));
  }
}

// Scan: 8 warps = 4 query groups x 2 coordinate halves.  Warp (grp_local,
// half) holds the fragments of k-blocks 8 half .. 8 half + 7 (word c + 4 half).
//
// Grid (query CTAs, database chunks): CTA (x, y) scans tiles
// y * tiles_per_chunk .. of the database and writes its queries' top-k to
// ids / scores + (y * nq + query) * k (with one chunk: the final lists; with
// several: per-chunk lists that k_search_merge combines).
template <int NV, int P>
__global__ void __launch_bounds__(256, search_ctas_per_sm(P)) k_search(const Dev cb, const uint8_t* __restrict__ db,
                                                   int64_t n_db, const uint8_t* __restrict__ prep, int nq, int k,
                                                   int tiles_per_chunk, int32_t* __restrict__ ids,
                                                   float* __restrict__ scores, const int32_t* __restrict__ qmap,
                                                   const unsigned* __restrict__ qcount) {
  __shared__ float xch[2][4][kRound][4][32];  // [buffer][group][tile of the round][acc element][lane]
  __shared__ float top_s[2][16][kMaxK];       // [coordinate half][query slot][rank]
  __shared__ int32_t top_i[2][16][kMaxK];
  __shared__ int top_n[2][16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gl = warp >> 1, half = warp & 1;
  const int grp = blockIdx.x * 4 + gl;
  const int nv_live = qmap ? (int)min(*qcount, (unsigned)nq) : nq;
  if (blockIdx.x * 16 >= nv_live) return;   // no live query in this CTA (uniform)
  const int ngroups = (nv_live + 3) / 4;
  const int g = lane >> 2, c = lane & 3;
  const bool live = grp < ngroups;
  if (threadIdx.x < 32) top_n[threadIdx.x >> 4][threadIdx.x & 15] = 0;
  uint2 bq[NV + 1][8];
  float S1 = 0.f, S2 = 0.f, K1 = 0.f, K2 = 0.f;
  if (live) {
    const uint8_t* blk = prep + (size_t)grp * search_block_bytes(NV);
    const uint2* frag = reinterpret_cast<const uint2*>(blk + kPrepHeader);
#pragma unroll
    for (int v = 0; v <= NV; ++v)
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) bq[v][kb] = frag[(v * 16 + 8 * half + kb) * 32 + lane];
    const float* hdr = reinterpret_cast<const float*>(blk);
    S1 = hdr[c];
    S2 = hdr[4 + c];
    K1 = hdr[8 + c];
    K2 = hdr[12 + c];
  }
  __syncthreads();
  const uint32_t* recs = reinterpret_cast<const uint32_t*>(db);
  const uint32_t* nrm = reinterpret_cast<const uint32_t*>(db + norm_offset(cb, n_db));
  constexpr int W = (kD / 32) * P;            // record words (d = 256, no extra-bit words)
  const float kq = cb.qjl_const;
  const int word = c + 4 * half;
  const int qslot = gl * 4 + c;               // this thread's query (shared-memory list index)
  const int64_t c0 = (int64_t)blockIdx.y * tiles_per_chunk;
  const int64_t ntiles = min((n_db + 15) / 16, c0 + tiles_per_chunk);   // end of this chunk
  // words and norms of one tile, loaded one tile ahead of use
  uint32_t nwa[P], nwb[P], nna = 0u, nnb = 0u;
  auto fetch = [&](int64_t tile) {
    const int64_t ta = tile * 16 + g, tb = ta + 8;
#pragma unroll
    for (int p = 0; p < P; ++p) {
      nwa[p] = (live && ta < n_db) ? __ldg(recs + ta * W + word * P + p) : 0u;
      nwb[p] = (live && tb < n_db) ? __ldg(recs + tb * W + word * P + p) : 0u;
    }
    nna = (live && ta < n_db) ? __ldg(nrm + ta) : 0u;
    nnb = (live && tb < n_db) ? __ldg(nrm + tb) : 0u;
  };
  // score a row must beat to enter this lane's query list (its k-th score
  // once the list is full), kept in a register and refreshed after insertions
  float thr = -INFINITY;
  if (c0 < ntiles) fetch(c0);
  // rounds of kRound tiles: each half scores its coordinates of the round's
  // tiles, the two halves of a group meet once per round
  for (int64_t t0 = c0; t0 < ntiles; t0 += kRound) {
    float part[kRound][4];
    uint32_t nra[kRound], nrb[kRound];
#pragma unroll
    for (int u = 0; u < kRound; ++u) {
      const int64_t tile = t0 + u;
      uint32_t wa[P], wb[P];
#pragma unroll
      for (int p = 0; p < P; ++p) {
        wa[p] = nwa[p];
        wb[p] = nwb[p];
      }
      nra[u] = nna;
      nrb[u] = nnb;
      if (tile + 1 < ntiles) fetch(tile + 1);
      float acc1[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
      if (live && tile < ntiles) {
#pragma unroll
        for (int v = 0; v <= NV; ++v) {
          uint32_t xa = 0, xb = 0;
          if (v < NV) {
#pragma unroll
            for (int p = 0; p < P - 1; ++p)
              if (kOddMask[v] >> p & 1u) {
                xa ^= wa[p];
                xb ^= wb[p];
              }
          } else {
            xa = wa[P - 1];
            xb = wb[P - 1];
          }
          uint32_t ra[16], rb[16];
          expand16(xa, ra);
          expand16(xb, rb);
          float(&acc)[4] = v < NV ? acc1 : acc2;
#pragma unroll
          for (int kb = 0; kb < 8; ++kb)
            mma_f16(acc, ra[2 * kb], rb[2 * kb], ra[2 * kb + 1], rb[2 * kb + 1], bq[v][kb].x, bq[v][kb].y);
        }
      }
      part[u][0] = acc1[0] + acc1[1];
      part[u][1] = acc1[2] + acc1[3];
      part[u][2] = acc2[0] + acc2[1];
      part[u][3] = acc2[2] + acc2[3];
    }
    // combine the two coordinate halves of the group: half h finishes tiles
    // u with u / (kRound / 2) == h of the round, using the other half's
    // partials from the exchange buffer (double-buffered: one barrier per round)
    const int buf = (int)(((t0 - c0) / kRound) & 1);
#pragma unroll
    for (int u = 0; u < kRound; ++u)
      if (u / (kRound / 2) != half)
#pragma unroll
        for (int e = 0; e < 4; ++e) xch[buf][gl][u][e][lane] = part[u][e];
    asm volatile("bar.sync %0, 64;" ::"r"(1 + gl));
    if (live) {
      const bool qok = grp * 4 + c < nv_live;
#pragma unroll
      for (int u = 0; u < kRound; ++u) {
        if (u / (kRound / 2) != half) continue;
        const int64_t ta = (t0 + u) * 16 + g, tb = ta + 8;
        const float m1a = part[u][0] + xch[buf][gl][u][0][lane];
        const float m1b = part[u][1] + xch[buf][gl][u][1][lane];
        const float m2a = part[u][2] + xch[buf][gl][u][2][lane];
        const float m2b = part[u][3] + xch[buf][gl][u][3][lane];
        const __half2 ha = *reinterpret_cast<const __half2*>(&nra[u]);
        const __half2 hb = *reinterpret_cast<const __half2*>(&nrb[u]);
        const float sa = __low2float(ha) * fmaf(__high2float(ha) * kq, fmaf(S2, m2a, K2), fmaf(S1, m1a, K1));
        const float sb = __low2float(hb) * fmaf(__high2float(hb) * kq, fmaf(S2, m2b, K2), fmaf(S1, m1b, K1));
        float* ls = top_s[half][0];
        int32_t* li = top_i[half][0];
        int* ln = top_n[half];
        // candidates: beat the current k-th score of their query in this half's list
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float sc = h == 0 ? sa : sb;
          const int64_t id = h == 0 ? ta : tb;
          const bool cand = qok && id < n_db && sc > thr;
          unsigned mask = __ballot_sync(kFull, cand);
          const bool any = mask != 0u;
          while (mask) {
            const int src = __ffs(mask) - 1;
            mask &= mask - 1;
            const float s_new = __shfl_sync(kFull, sc, src);
            const int id_new = (int)__shfl_sync(kFull, (int)id, src);
            const int qs = __shfl_sync(kFull, qslot, src);
            if (lane == 0) {
              // insert into the sorted list of query qs (decreasing score; the
              // list receives increasing ids, so ties keep the earlier id first)
              float* sq = ls + qs * kMaxK;
              int32_t* iq = li + qs * kMaxK;
              int n0 = ln[qs];
              if (n0 < k || s_new > sq[k - 1]) {
                int pos = n0 < k ? n0 : k - 1;
                while (pos > 0 && sq[pos - 1] < s_new) {
                  sq[pos] = sq[pos - 1];
                  iq[pos] = iq[pos - 1];
                  --pos;
                }
                sq[pos] = s_new;
                iq[pos] = id_new;
                if (n0 < k) ln[qs] = n0 + 1;
              }
            }
            __syncwarp();
          }
          // a list changed: refresh this lane's entry threshold
          if (any) thr = ln[qslot] < k ? -INFINITY : ls[qslot * kMaxK + k - 1];
        }
      }
    }
  }
  __syncthreads();
  // merge the two halves' lists of each query (decreasing score, ties to the smaller id)
  if (half == 0 && live && lane < 4) {
    const int qi = grp * 4 + lane;            // query slot
    // final lists (one chunk) go to the query's own row; per-chunk lists stay in slot order
    const int qo = (gridDim.y == 1 && qmap) ? (qi < nv_live ? qmap[qi] : 0) : qi;
    if (qi < nv_live) {
      const int qs = gl * 4 + lane;
      const int na = top_n[0][qs], nb = top_n[1][qs];
      int ia = 0, ib = 0;
      for (int j = 0; j < k; ++j) {
        bool take_a;
        if (ia < na && ib < nb) {
          const float sa = top_s[0][qs][ia], sb = top_s[1][qs][ib];
          take_a = sa > sb || (sa == sb && top_i[0][qs][ia] < top_i[1][qs][ib]);
        } else {
          take_a = ia < na;
        }
        const bool have = ia < na || ib < nb;
        const float sc = !have ? -INFINITY : take_a ? top_s[0][qs][ia] : top_s[1][qs][ib];
        const int32_t id = !have ? -1 : take_a ? top_i[0][qs][ia] : top_i[1][qs][ib];
        if (have) {
          if (take_a) ++ia;
          else ++ib;
        }
        ids[((size_t)blockIdx.y * nq + qo) * k + j] = id;
        scores[((size_t)blockIdx.y * nq + qo) * k + j] = sc;
      }
    }
  }
}


// Merge of the per-chunk top-k lists: one warp per query takes the k best of
// its chunks * k candidates (decreasing score, ties to the smaller id; a
// missing entry is id -1 with score -inf and ranks last).
__global__ void __launch_bounds__(128) k_search_merge(const int32_t* __restrict__ pid, const float* __restrict__ psc,
                                                      int chunks, int nq, int k, int32_t* __restrict__ ids,
                                                      float* __restrict__ scores, const int32_t* __restrict__ qmap,
                                                      const unsigned* __restrict__ qcount) {
  constexpr int kPer = kMaxChunks * kMaxK / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qi = blockIdx.x * 4 + warp;     // query slot
  const int nv_live = qmap ? (int)min(*qcount, (unsigned)nq) : nq;
  if (qi >= nv_live) return;
  const int qo = qmap ? qmap[qi] : qi;      // output row
  const int n = chunks * k;
  float s[kPer];
  int32_t id[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = lane + 32 * j;
    const int ch = e / k, r = e - ch * k;
    const bool v = e < n;
    id[j] = v ? pid[((size_t)ch * nq + qi) * k + r] : -1;
    s[j] = (v && id[j] >= 0) ? psc[((size_t)ch * nq + qi) * k + r] : -INFINITY;
    if (s[j] == -INFINITY) id[j] = -1;
  }
  // (score, id) order: higher score first, then the smaller valid id
  auto better = [](float sa, int32_t ia, float sb, int32_t ib) {
    if (ia < 0) return false;
    if (ib < 0) return true;
    return sa > sb || (sa == sb && ia < ib);
  };
  for (int out = 0; out < k; ++out) {
    float bs = -INFINITY;
    int32_t bi = -1;
    int bj = -1;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (better(s[j], id[j], bs, bi)) {
        bs = s[j];
        bi = id[j];
        bj = j;
      }
    float ws = bs;
    int32_t wi = bi;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float os = __shfl_xor_sync(kFull, ws, o);
      const int32_t oi = __shfl_xor_sync(kFull, wi, o);
      if (better(os, oi, ws, wi)) {
        ws = os;
        wi = oi;
      }
    }
    // the lane holding the winner drops it (ids are distinct across chunks)
    if (wi >= 0 && bi == wi) {
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (j == bj) {
          s[j] = -INFINITY;
          id[j] = -1;
        }
    }
    if (lane == 0) {
      ids[(size_t)qo * k + out] = wi;
      scores[(size_t)qo * k + out] = wi >= 0 ? ws : -INFINITY;
    }
  }
}

// Database chunks of the scan: enough that the grid fills its last wave of
// resident CTAs (>= 95% of the slots busy, else the best count up to 16),
// with at least 256 tiles per chunk.
int search_chunks(const Dev& cb, int64_t n_db, int nq, int sms) {
  const int64_t base = ((nq + 3) / 4 + 3) / 4;
  const int64_t per_wave = (int64_t)sms * search_ctas_per_sm(cb.P);
  const int64_t ntiles = (n_db + 15) / 16;
  const int max_s = (int)std::max<int64_t>(1, std::min<int64_t>(kMaxChunks, ntiles / 256));
  int best = 1;
  double best_eff = 0.0;
  for (int sch = 1; sch <= max_s; ++sch) {
    const int64_t units = base * sch;
    const double eff = (double)units / (double)(((units + per_wave - 1) / per_wave) * per_wave);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = sch;
    }
    if (eff >= 0.95) break;
  }
  return best;
}

int64_t search_workspace_bytes(const Dev& cb, int64_t n_db, int nq, int k, int sms) {
  const int64_t prep = align256((int64_t)((nq + 3) / 4) * search_block_bytes(cb.nv));
  const int chunks = search_chunks(cb, n_db, nq, sms);
  return chunks > 1 ? prep + align256((int64_t)chunks * nq * k * 8) : prep;
}

// The exact scan over all queries (qmap == nullptr) or over the queries
// qmap[0 .. *qcount - 1] (grids sized for nq; slots past *qcount exit).
cudaError_t launch_search_subset(const Dev& cb, const uint8_t* db, int64_t n_db, const float* q, int nq, int d_in,
                                 int k, int32_t* ids, float* scores, uint8_t* prep, int sms, const int32_t* qmap,
                                 const unsigned* qcount, cudaStream_t s) {
  const int ngroups = (nq + 3) / 4;
  k_search_prep<<<dim3(ngroups, 4), 1024, 0, s>>>(cb, q, nq, d_in, prep, qmap, qcount);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int chunks = search_chunks(cb, n_db, nq, sms);
  const int64_t ntiles = (n_db + 15) / 16;
  int64_t tpc = (ntiles + chunks - 1) / chunks;
  tpc = (tpc + kRound - 1) / kRound * kRound;
  int32_t* oid = ids;
  float* osc = scores;
  if (chunks > 1) {
    uint8_t* part = prep + align256((int64_t)ngroups * search_block_bytes(cb.nv));
    oid = reinterpret_cast<int32_t*>(part);
    osc = reinterpret_cast<float*>(part + (size_t)chunks * nq * k * 4);
  }
  const dim3 grid((ngroups + 3) / 4, chunks);
  switch (cb.b1) {
    case 1: k_search<1, 2><<<grid, 256, 0, s>>>(cb, db, n_db, prep, nq, k, (int)tpc, oid, osc, qmap, qcount); break;
    case 2: k_search<2, 3><<<grid, 256, 0, s>>>(cb, db, n_db, prep, nq, k, (int)tpc, oid, osc, qmap, qcount); break;
    default: k_search<4, 4><<<grid, 256, 0, s>>>(cb, db, n_db, prep, nq, k, (int)tpc, oid, osc, qmap, qcount); break;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || chunks == 1) return e;
  k_search_merge<<<(nq + 3) / 4, 128, 0, s>>>(oid, osc, chunks, nq, k, ids, scores, qmap, qcount);
  return cudaGetLastError();
}

cudaError_t launch_search(const Dev& cb, const uint8_t* db, int64_t n_db, const float* q, int nq, int d_in, int k,
                          int32_t* ids, float* scores, uint8_t* prep, int sms, cudaStream_t s) {
  return launch_search_subset(cb, db, n_db, q, nq, d_in, k, ids, scores, prep, sms, nullptr, nullptr, s);
}

}  // namespace tq
