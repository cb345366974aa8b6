// Top-k inner-product search on the 5th-generation tensor cores: candidate
// generation with tcgen05 (queries resident in tensor memory, database tiles
// decoded once into shared memory), then exact re-ranking of the candidates.
//
// [xujun] note-189244, 常见问题 (vector search over a compressed database);
// [cnyes] hao.cnyes.com "TurboQuant", 1 bit 掃尾 (the full-precision query
// side carries the estimate):
//   est(q, x) = n ( <q', yhat> + gamma sqrt(pi/2)/m <q'', sigma> ),
//   q' = Pi q, q'' = S Pi q, sigma in {-1, +1}.
//
// Scoring every (query, row) pair is the one dense contraction of the search:
// D[q][r] = sum_k A[q][k] B[r][k] over K = 512 (256 rotated coordinates, then
// 256 sketch rows) with
//   A = fp16(q' 2^e_q), fp16(q'' 2^e_q)            (per query, in TMEM)
//   B = fp16(c[idx]), fp16(gamma_r kq) * sigma       (per database row, SMEM)
// so that n_r D[q][r] 2^-e_q approximates est(q, r) to within a bound eps(q)
// that follows from fp16 rounding (half an ulp, 2^-11 relative, per operand)
// and fp32 accumulation:
//   eps(q) = 1.5 [ (2^-10 + 2^-12) (n_max c_max |q'|_1 + (n gamma)_max kq |q''|_1)
//                  + n_max |q''|_1 2^-24 ]
// with n_max and (n gamma)_max taken over the database.
//
// Pipeline (one persistent CTA per SM, the (query block, database tile)
// units split evenly over the CTAs):
//   * k_stc_prep: q' and q'' in fp32 (kept for the re-ranking), the fp16
//     operand words of each 128-query block, |q'|_1, |q''|_1, the scale 2^e_q;
//   * k_stc_dbmax: n_max and (n gamma)_max of the database;
//   * k_stc_scan: 4 decoder warps turn the packed records of each 128-row tile
//     into the B operand (one 16 KB K-block per ring slot, 128-byte swizzled,
//     K-major), one thread issues tcgen05.mma M128 N128 K16 into one of two
//     TMEM accumulators, and 4 epilogue warps (one query per thread) read the
//     accumulator back with tcgen05.ld and keep, per query and per part of the
//     database a CTA scans, the kCand best approximate scores;
//   * k_stc_refine: one warp per query scores every candidate exactly in fp32
//     (the stored fp32 centroids, fp32 q' and q''), keeps the k best
//     (decreasing score, ties to the smaller id), and checks the certificate:
//     for every part whose list is full, its kCand-th approximate score plus
//     eps(q) lies below the k-th exact score, so no row outside the lists can
//     enter the top k.  A query that fails it is queued for the exact scan of
//     tq_search.cu, which then overwrites its result.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "tq_internal.cuh"

namespace tq {

namespace stc {

constexpr int kD = 256;              // vector dimension (= sketch rows)
constexpr int kQ = 128;              // queries per block (TMEM lanes, MMA M)
constexpr int kR = 128;              // database rows per tile (MMA N)
constexpr int kCand = 32;            // candidates kept per (query, part)
constexpr int kMaxKTc = 16;          // largest k served by this path
constexpr int kStg = 2;              // staging slots of packed records (bulk copies)
// Per stage-1 width b': record bytes, staging slot bytes (records + norm
// entries) and B ring slots (as many 16 KB K-blocks as shared memory holds).
__host__ __device__ constexpr int rec_bytes(int b1) { return 32 * (b1 + 1); }
__host__ __device__ constexpr int stg_bytes(int b1) { return kR * rec_bytes(b1) + kR * 4; }
__host__ __device__ constexpr int ring_slots(int b1) { return b1 == 3 ? 9 : 10; }
constexpr int kSlotBytes = kR * 128; // 128 rows x 64 fp16 (one K-block)
constexpr int kDecWarps = 4;         // decoder warps (4: both word columns of a round per thread)
constexpr int kThreads = 256 + 32 * kDecWarps;   // warps: 0 MMA, 1 loader, 2-3 idle, 4-7 epilogue, 8.. decoders
constexpr int kPrepQ = 32;           // queries per prep CTA
constexpr long long kSpin = 1ll << 26;
constexpr uint32_t kTmemCols = 512;  // A: 0..255, D0: 256..383, D1: 384..511
// D = F32, A = B = F16, both K-major, N = 128, M = 128
constexpr uint32_t kIdesc = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
// shared memory map (offsets from a 1024-aligned base): B ring, staging,
// candidate lists (float / int [kCand][kQ]), tile norms [2][kR], mbarriers,
// then the TMEM base address and the abort flag
template <int B1>
struct Smem {
  static constexpr int kSlots = ring_slots(B1);
  static constexpr uint32_t kOffRing = 0;
  static constexpr uint32_t kOffStg = kOffRing + kSlots * kSlotBytes;
  static constexpr uint32_t kOffLsc = kOffStg + kStg * stg_bytes(B1);
  static constexpr uint32_t kOffLid = kOffLsc + kCand * kQ * 4;
  static constexpr uint32_t kOffNrm = kOffLid + kCand * kQ * 4;
  static constexpr uint32_t kOffBar = kOffNrm + 2 * kR * 4;
  static constexpr int kNumBars = 2 * kSlots + 8 + 2 * kStg;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kOffMisc + 16 + 1024;         // + alignment slack
  static_assert(kBytes <= 232448, "shared memory of the scan exceeds 227 KB");
};
// misc words of the workspace: [0] n_max bits, [1] (n gamma)_max bits, [2] fallback count
constexpr int kMiscWords = 64;

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// Coordinate (or sketch row) of element h (0 = low half, 1 = high half) of
// register e of 16-byte chunk ch of K-block kb (within a 256-wide slab).  The
// register pairs coordinates j and j + 16 of one 32-coordinate word column, so
// the decoder builds it from bits j and j + 16 of a packed word with one shift.
__host__ __device__ __forceinline__ int slab_coord(int kb, int ch, int e, int h) {
  return 32 * (2 * kb + (ch >> 2)) + 4 * (ch & 3) + e + 16 * h;
}

__device__ __forceinline__ uint32_t f16_bits(float x) { return (uint32_t)__half_as_ushort(__float2half_rn(x)); }

// 0xffff in each 16-bit half whose top bit (15 or 31) is set, else 0: a
// byte permute that replicates the sign of bytes 1 and 3.
__device__ __forceinline__ uint32_t half_masks(uint32_t x) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, 0xBB99;" : "=r"(r) : "r"(x), "r"(0u));
  return r;
}

// r[j] for a run-time j without dynamic register indexing (a select tree).
__device__ __forceinline__ uint32_t pick32(const uint32_t (&r)[32], int j) {
  uint32_t a[16], b[8], c[4], d[2];
#pragma unroll
  for (int k = 0; k < 16; ++k) a[k] = (j & 16) ? r[k + 16] : r[k];
#pragma unroll
  for (int k = 0; k < 8; ++k) b[k] = (j & 8) ? a[k + 8] : a[k];
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = (j & 4) ? b[k + 4] : b[k];
#pragma unroll
  for (int k = 0; k < 2; ++k) d[k] = (j & 2) ? c[k + 2] : c[k];
  return (j & 1) ? d[1] : d[0];
}

// Bounded wait on an mbarrier phase; gives up early once another role of the
// CTA has given up (abort flag).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  for (long long i = 0; i < kSpin; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 1023) == 1023 && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// The same for a whole warp: every lane gets the same answer.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag));
}

__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Min-heap of kCand (score, id) entries in the column layout [e * kQ + ql]:
// place (v, id) at slot e and sink it below any smaller child.
__device__ __forceinline__ void heap_sift(float* Lsc, int32_t* Lid, int ql, int e, float v, int32_t id) {
  while (true) {
    const int l = 2 * e + 1;
    if (l >= kCand) break;
    int m = l;
    float vm = Lsc[l * kQ + ql];
    if (l + 1 < kCand) {
      const float vr = Lsc[(l + 1) * kQ + ql];
      if (vr < vm) {
        m = l + 1;
        vm = vr;
      }
    }
    if (!(vm < v)) break;
    Lsc[e * kQ + ql] = vm;
    Lid[e * kQ + ql] = Lid[m * kQ + ql];
    e = m;
  }
  Lsc[e * kQ + ql] = v;
  Lid[e * kQ + ql] = id;
}

// CTA c of G covers units [U c / G, U (c + 1) / G); the CTA holding unit x.
__host__ __device__ __forceinline__ int64_t unit_cta(int64_t x, int64_t U, int64_t G) { return (G * (x + 1) - 1) / U; }

}  // namespace stc

using namespace stc;

// ---------------------------------------------------------------------------
// Query preparation: 32 queries per CTA.  q' = Pi q and q'' = (S Pi) q in fp32
// (256 threads, thread t computes output coordinate t of both for all 32
// queries), then per query: the scale 2^e_q that puts max(|q'|, |q''|) in
// [2^13, 2^14), the fp16 operand words (word w of a query = K elements 2w and
// 2w + 1 in the tensor-memory order of the scan), |q'|_1 and |q''|_1.
//   Aw    [NQB][256 words][128 queries] (queries past nq are zero)
//   qf    [nq][512]  fp32 q' then q''
//   qinfo [nq][4]    2^-e_q, |q'|_1, |q''|_1, 0
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_stc_prep(const Dev cb, const float* __restrict__ q, int nq, int d_in,
                                                  uint32_t* __restrict__ Aw, float* __restrict__ qf,
                                                  float* __restrict__ qinfo, unsigned* __restrict__ misc) {
  extern __shared__ __align__(16) float sp[];
  float* sq = sp;                       // [kPrepQ][kD]
  float* so = sp + kPrepQ * kD;         // [kPrepQ][2 kD]
  const int tid = threadIdx.x;
  const int q0 = blockIdx.x * kPrepQ;
  if (blockIdx.x == 0 && tid < kMiscWords) misc[tid] = 0u;
  for (int e = tid; e < kPrepQ * kD; e += 256) {
    const int qi = e / kD, k = e - qi * kD;
    sq[e] = (q0 + qi < nq && k < d_in) ? q[(size_t)(q0 + qi) * d_in + k] : 0.f;
  }
  __syncthreads();
  float a1[kPrepQ], a2[kPrepQ];
#pragma unroll
  for (int i = 0; i < kPrepQ; ++i) a1[i] = a2[i] = 0.f;
  for (int k = 0; k < kD; k += 4) {
    float m1[4], m2[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      m1[u] = __ldg(cb.PiT + (size_t)(k + u) * kD + tid);
      m2[u] = __ldg(cb.SPT + (size_t)(k + u) * kD + tid);
    }
#pragma unroll
    for (int i = 0; i < kPrepQ; ++i) {
      const float4 x = *reinterpret_cast<const float4*>(sq + i * kD + k);
      a1[i] = fmaf(m1[0], x.x, fmaf(m1[1], x.y, fmaf(m1[2], x.z, fmaf(m1[3], x.w, a1[i]))));
      a2[i] = fmaf(m2[0], x.x, fmaf(m2[1], x.y, fmaf(m2[2], x.z, fmaf(m2[3], x.w, a2[i]))));
    }
  }
#pragma unroll
  for (int i = 0; i < kPrepQ; ++i) {
    so[i * 2 * kD + tid] = a1[i];
    so[i * 2 * kD + kD + tid] = a2[i];
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int i = warp; i < kPrepQ; i += 8) {
    const int qi = q0 + i;
    const float* v = so + i * 2 * kD;
    float mx = 0.f, l1 = 0.f, l2 = 0.f;
    for (int k = lane; k < kD; k += 32) {
      mx = fmaxf(mx, fmaxf(fabsf(v[k]), fabsf(v[kD + k])));
      l1 += fabsf(v[k]);
      l2 += fabsf(v[kD + k]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
      l2 += __shfl_xor_sync(0xffffffffu, l2, o);
    }
    int ex = 0;
    if (mx > 0.f) {
      frexpf(mx, &ex);          // mx in [2^(ex-1), 2^ex)
      ex = 14 - ex;             // mx 2^ex in [2^13, 2^14)
    }
    const float sc = ldexpf(1.f, ex);
    const bool live = qi < nq;
    if (live) {
      for (int k = lane; k < 2 * kD; k += 32) qf[(size_t)qi * 2 * kD + k] = v[k];
      if (lane == 0)
        *reinterpret_cast<float4*>(qinfo + (size_t)qi * 4) = make_float4(ldexpf(1.f, -ex), l1, l2, 0.f);
    }
    const int qb = qi / kQ, ql = qi - qb * kQ;
    for (int w = lane; w < 256; w += 32) {
      const int slab = w >> 7, kb = (w >> 5) & 3, ks = (w >> 3) & 3, wi = w & 7;
      const int ch = 2 * ks + (wi >> 2), e = wi & 3;
      const float x0 = live ? v[slab * kD + slab_coord(kb, ch, e, 0)] * sc : 0.f;
      const float x1 = live ? v[slab * kD + slab_coord(kb, ch, e, 1)] * sc : 0.f;
      Aw[((size_t)qb * 256 + w) * kQ + ql] = f16_bits(x0) | (f16_bits(x1) << 16);
    }
  }
}

// n_max and (n gamma)_max over the database (non-negative floats compare as
// their bit patterns).
__global__ void __launch_bounds__(256) k_stc_dbmax(const Dev cb, const uint8_t* __restrict__ db, int64_t n_db,
                                                   unsigned* __restrict__ misc) {
  const uint32_t* nrm = reinterpret_cast<const uint32_t*>(db + norm_offset(cb, n_db));
  float mn = 0.f, mg = 0.f;
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < n_db; r += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t e = __ldg(nrm + r);
    const __half2 h = *reinterpret_cast<const __half2*>(&e);
    const float n = fabsf(__low2float(h)), g = fabsf(__high2float(h));
    mn = fmaxf(mn, n);
    mg = fmaxf(mg, n * g);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    mn = fmaxf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, o));
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMax(misc + 0, __float_as_uint(mn));
    atomicMax(misc + 1, __float_as_uint(mg));
  }
}

// ---------------------------------------------------------------------------
// The tensor-core scan.  Warp roles: warp 0 issues the MMAs (one thread) and
// owns the TMEM allocation; warps 4..7 are the epilogue (warp w reads TMEM
// lanes 32 (w % 4) .., one query per thread); warps 8..15 decode.
// Lists: lsc / lid [NQB][Pmax][kCand][kQ], decreasing approximate score.
// ---------------------------------------------------------------------------
template <int B1>
__global__ void __launch_bounds__(kThreads, 1)
    k_stc_scan(const Dev cb, const uint8_t* __restrict__ db, int64_t n_db, int nq, const uint32_t* __restrict__ Aw,
               const float* __restrict__ qinfo, float* __restrict__ lsc, int32_t* __restrict__ lid, int Pmax,
               int* __restrict__ status) {
  constexpr int P = B1 + 1;               // planes per word column (stage 1 + signs)
  using SM = Smem<B1>;
  constexpr int kSlots = SM::kSlots;
  constexpr uint32_t kOffRing = SM::kOffRing, kOffStg = SM::kOffStg, kOffLsc = SM::kOffLsc, kOffLid = SM::kOffLid,
                     kOffNrm = SM::kOffNrm, kOffBar = SM::kOffBar, kOffMisc = SM::kOffMisc;
  constexpr int kStgBytes = stg_bytes(B1);
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so the
  // compiler keeps every access through smem in the shared space
  uint8_t* smem = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = su32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t NT = (n_db + kR - 1) / kR, NQB = (nq + kQ - 1) / kQ, U = NQB * NT, G = gridDim.x;
  const int64_t u0 = U * blockIdx.x / G, u1 = U * (blockIdx.x + 1) / G;
  if (u0 >= u1) return;                   // uniform over the CTA
  const int ntile = (int)(u1 - u0);
  const uint32_t bar0 = sbase + kOffBar;
  auto blk_full = [&](int s) { return bar0 + 8u * s; };
  auto blk_empty = [&](int s) { return bar0 + 8u * (kSlots + s); };
  const uint32_t d_full0 = bar0 + 8u * (2 * kSlots), d_empty0 = d_full0 + 16, a_full = d_full0 + 32,
                 drain = d_full0 + 40, nrm_rdy0 = d_full0 + 48, stg_full0 = d_full0 + 64,
                 stg_empty0 = stg_full0 + 8 * kStg;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tslot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(blk_full(s)), "r"(kDecWarps));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(blk_empty(s)));     // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(d_full0 + 8u * b));  // MMA commit
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(d_empty0 + 8u * b)); // 4 epilogue warps
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(a_full));              // 4 epilogue warps
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(drain));               // final MMA commit
    for (int b = 0; b < 2; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(nrm_rdy0 + 8u * b)); // 4 epilogue warps
    for (int b = 0; b < kStg; ++b) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;" ::"r"(stg_full0 + 8u * b));  // loader: bytes + norms
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(stg_empty0 + 8u * b), "r"(kDecWarps));
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      int seg = 0;
      bool ok = true;
      bool issued = false;
      // tile index within the query block (u0 + i) % NT, and the ring
      // position of K-block g = 8 i + blk: slot g % kSlots, phase
      // (g / kSlots) & 1, all kept as running counters
      int64_t t = u0 % NT;
      int slot = 0;
      uint32_t sphase = 0u;
      for (int i = 0; i < ntile && ok; ++i) {
        if (i == 0 || t == 0) {
          ok = wait_bar(a_full, seg & 1, abort_flag);
          ++seg;
          if (!ok) break;
        }
        if (i >= 2 && !(ok = wait_bar(d_empty0 + 8u * (i & 1), ((i >> 1) - 1) & 1, abort_flag))) break;
        fence_after();
        const uint32_t dcol = tmem + 256 + 128 * (i & 1);
        for (int blk = 0; blk < 8 && ok; ++blk) {
          if (!(ok = wait_bar(blk_full(slot), sphase, abort_flag))) break;
          fence_after();
          const uint32_t acol = tmem + (blk & 1) * 128 + (blk >> 1) * 32;
          const uint32_t bsm = sbase + kOffRing + slot * kSlotBytes;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t acc = (blk | ks) != 0;
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, "
                "p;\n}\n" ::"r"(dcol),
                "r"(acol + 8 * ks), "l"(sw128_desc(bsm + 32 * ks)), "r"(kIdesc), "r"(acc));
          }
          issued = true;
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                           blk_empty(slot))
                       : "memory");
          if (++slot == kSlots) {
            slot = 0;
            sphase ^= 1u;
          }
        }
        if (!ok) break;
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         d_full0 + 8u * (i & 1))
                     : "memory");
        if (++t == NT) t = 0;
      }
      if (!ok) {
        atomicOr(status, 4);
        *abort_flag = 1;
      }
      if (issued) {
        // every MMA of this thread completes before TMEM is released
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(drain)
                     : "memory");
        for (long long k = 0; k < kSpin; ++k) {
          uint32_t done;
          asm volatile(
              "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}\n"
              : "=r"(done)
              : "r"(drain)
              : "memory");
          if (done) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ loader
    // packed records of each tile by bulk copy (async proxy: the decoders'
    // proxy fences do not wait for it), norm entries by the warp's loads
    constexpr int RB = 32 * (B1 + 1);            // record bytes
    const uint32_t* nrm = reinterpret_cast<const uint32_t*>(db + norm_offset(cb, n_db));
    bool ok = true;
    int64_t t = u0 % NT;                         // (u0 + i) % NT, as a running counter
    for (int i = 0; i < ntile && ok; ++i, t = t + 1 == NT ? 0 : t + 1) {
      const int sidx = i % kStg, use = i / kStg;
      if (use > 0 && !(ok = wait_bar_warp(stg_empty0 + 8u * sidx, (uint32_t)((use - 1) & 1), abort_flag))) break;
      const int64_t row0 = t * kR;
      const int valid = (int)min((int64_t)kR, n_db - row0);
      uint8_t* stg = smem + kOffStg + sidx * kStgBytes;
      if (lane == 0) {
        const uint32_t bar = stg_full0 + 8u * sidx;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"((uint32_t)(valid * RB))
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(stg)),
            "l"(db + row0 * RB), "r"((uint32_t)(valid * RB)), "r"(bar)
            : "memory");
      }
      uint32_t* sn = reinterpret_cast<uint32_t*>(stg + kR * RB);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rr = 4 * lane + e;
        sn[rr] = rr < valid ? __ldg(nrm + row0 + rr) : 0u;
      }
      __syncwarp();
      if (lane == 0) bar_arrive(stg_full0 + 8u * sidx);
    }
    if (!ok) {
      atomicOr(status, 4);
      *abort_flag = 1;
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ epilogue
    const int ql = tid - 128;                    // query lane = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    float* Lsc = reinterpret_cast<float*>(smem + kOffLsc);
    int32_t* Lid = reinterpret_cast<int32_t*>(smem + kOffLid);
    float* nrm_s = reinterpret_cast<float*>(smem + kOffNrm);
    const uint32_t* nrm = reinterpret_cast<const uint32_t*>(db + norm_offset(cb, n_db));
    // thr: the list's entry threshold (scaled scores); thr_s = thr 2^e_q, the
    // same threshold for the unscaled products (2^-e_q is a power of two, so
    // p 2^-e_q > thr exactly when p > thr 2^e_q)
    float thr = -INFINITY, inv_scale = 0.f, scale_q = INFINITY, thr_s = -INFINITY;
    int filled = 0;                              // entries in the list (a min-heap once full)
    bool ok = true;
    int seg = 0;
    // norm entry of this thread's row of tile i, whose index within its
    // query block is tt (prefetched one tile ahead)
    auto norm_of = [&](int i, int64_t tt) -> uint32_t {
      const int64_t row = tt * kR + ql;
      return (i < ntile && row < n_db) ? __ldg(nrm + row) : 0u;
    };
    // query block and tile of u0 + i as running counters
    int64_t qb = u0 / NT, t = u0 % NT;
    uint32_t nnext = norm_of(0, t);
    for (int i = 0; i < ntile && ok; ++i) {
      if (i == 0 || t == 0) {
        // new segment: reset the lists and load this query block's operand
        for (int j = 0; j < kCand; ++j) {
          Lsc[j * kQ + ql] = -INFINITY;
          Lid[j * kQ + ql] = -1;
        }
        thr = -INFINITY;
        filled = 0;
        const int qi = (int)(qb * kQ + ql);
        inv_scale = qi < nq ? __ldg(qinfo + (size_t)qi * 4) : 0.f;
        scale_q = inv_scale > 0.f ? 1.f / inv_scale : INFINITY;
        thr_s = thr * scale_q;
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __ldg(Aw + ((size_t)qb * 256 + 32 * c + j) * kQ + ql);
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
              "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(tmem + lane_off + 32 * c),
              "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
              "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
              "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
              "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        fence_before();
        __syncwarp();
        if (lane == 0) bar_arrive(a_full);
        ++seg;
      }
      const uint32_t ncur = nnext;
      nnext = norm_of(i + 1, t + 1 == NT ? 0 : t + 1);
      if (!(ok = wait_bar_warp(d_full0 + 8u * (i & 1), (uint32_t)((i >> 1) & 1), abort_flag))) break;
      fence_after();
      // n_r of every column of the tile, shared by the 128 queries (each
      // thread applies its own query's 2^-e_q); the four warps meet on an
      // mbarrier (bounded wait) rather than a named barrier
      float* nb = nrm_s + (i & 1) * kR;
      nb[ql] = __low2float(*reinterpret_cast<const __half2*>(&ncur));
      __syncwarp();
      if (lane == 0) bar_arrive(nrm_rdy0 + 8u * (i & 1));
      if (!(ok = wait_bar_warp(nrm_rdy0 + 8u * (i & 1), (uint32_t)((i >> 1) & 1), abort_flag))) break;
      const int valid = (int)min((int64_t)kR, n_db - t * kR);
      const uint32_t dcol = tmem + 256 + 128 * (i & 1);
      const int64_t row0 = t * kR;
#pragma unroll 1
      for (int cbk = 0; cbk < 4; ++cbk) {
        uint32_t r[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
            "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
              "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
              "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
              "=r"(r[30]), "=r"(r[31])
            : "r"(dcol + lane_off + 32 * cbk));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        // unscaled scores of the chunk and the mask of those above the
        // threshold (branch-free); rows past the database end masked once
        // (thr_s - p < 0 exactly when p > thr_s: the sign bit is funnel-shifted
        // into the mask, j = 31 first so that row j lands on bit j)
        uint32_t cand = 0u;
#pragma unroll
        for (int j = 31; j >= 0; --j) {
          const float pj = __uint_as_float(r[j]) * nb[32 * cbk + j];
          r[j] = __float_as_uint(pj);
          cand = __funnelshift_l(__float_as_uint(thr_s - pj), cand, 1);
        }
        const int nvalid = valid - 32 * cbk;
        cand &= nvalid >= 32 ? 0xffffffffu : (nvalid <= 0 ? 0u : (1u << nvalid) - 1u);
        if (__any_sync(0xffffffffu, cand != 0u)) {
          // take the candidates one by one (a compact loop: the score is
          // picked from the registers by a select tree, the unsorted list's
          // minimum is replaced and found again)
          while (cand) {
            const int j = __ffs(cand) - 1;
            cand &= cand - 1;
            const float sj = __uint_as_float(pick32(r, j)) * inv_scale;
            if (!(sj > thr)) continue;
            const int32_t id = (int32_t)(row0 + 32 * cbk + j);
            if (filled < kCand) {
              // filling: append; once full, order the list as a min-heap
              Lsc[filled * kQ + ql] = sj;
              Lid[filled * kQ + ql] = id;
              if (++filled == kCand) {
                for (int e = kCand / 2 - 1; e >= 0; --e) heap_sift(Lsc, Lid, ql, e, Lsc[e * kQ + ql], Lid[e * kQ + ql]);
                thr = Lsc[ql];
                thr_s = thr * scale_q;
              }
            } else {
              // full: the new entry replaces the minimum (the root) and sinks
              heap_sift(Lsc, Lid, ql, 0, sj, id);
              thr = Lsc[ql];
              thr_s = thr * scale_q;
            }
          }
          __syncwarp();
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) bar_arrive(d_empty0 + 8u * (i & 1));
      if (i == ntile - 1 || t + 1 == NT) {
        // segment end: this CTA's lists for query block qb, part = CTA - first CTA of qb
        const int part = (int)(blockIdx.x - unit_cta(qb * NT, U, G));
        const size_t base = ((size_t)qb * Pmax + part) * kCand;
        // sort the list (decreasing score; unused slots hold -inf and id -1)
        for (int a1 = 1; a1 < kCand; ++a1) {
          const float sv = Lsc[a1 * kQ + ql];
          const int32_t iv = Lid[a1 * kQ + ql];
          int b1 = a1;
          while (b1 > 0 && Lsc[(b1 - 1) * kQ + ql] < sv) {
            Lsc[b1 * kQ + ql] = Lsc[(b1 - 1) * kQ + ql];
            Lid[b1 * kQ + ql] = Lid[(b1 - 1) * kQ + ql];
            --b1;
          }
          Lsc[b1 * kQ + ql] = sv;
          Lid[b1 * kQ + ql] = iv;
        }
        for (int j = 0; j < kCand; ++j) {
          lsc[(base + j) * kQ + ql] = Lsc[j * kQ + ql];
          lid[(base + j) * kQ + ql] = Lid[j * kQ + ql];
        }
      }
      if (++t == NT) {
        t = 0;
        ++qb;
      }
    }
    if (!ok) {
      atomicOr(status, 4);
      *abort_flag = 1;
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ decoders
    // thread (r, h): row r of the tile, word column 2 kb + h in round kb (8
    // decoder warps), or both word columns (4 decoder warps)
    constexpr int kHalves = kDecWarps == 8 ? 1 : 2;
    const int r = (tid - 256) & 127, h0 = kDecWarps == 8 ? (tid - 256) >> 7 : 0;
    constexpr int L = 1 << B1;
    constexpr int RB = 32 * P;                   // record bytes
    // fp16 magnitudes of the upper half of the (symmetric) centroid table, in both halves
    uint32_t mag[L / 2];
#pragma unroll
    for (int k = 0; k < L / 2; ++k) {
      const uint32_t h = f16_bits(cb.cent[L / 2 + k]);
      mag[k] = h | (h << 16);
    }
    const float kq = cb.qjl_const;
    bool ok = true;
    // ring position of K-block g = 8 i + 2 kb + sl: slot g % kSlots and use
    // g / kSlots, as running counters
    int dslot = 0;
    int64_t duse = 0;
    for (int i = 0; i < ntile && ok; ++i) {
      const int sidx = i % kStg;
      if (!(ok = wait_bar_warp(stg_full0 + 8u * sidx, (uint32_t)((i / kStg) & 1), abort_flag))) break;
      const uint8_t* stg = smem + kOffStg + sidx * kStgBytes;
      const uint8_t* rec = stg + r * RB;
      // sigma slab value of this row: fp16(gamma kq), negative pattern in both halves
      const uint32_t ne = reinterpret_cast<const uint32_t*>(stg + kR * RB)[r];
      const float gam = __high2float(*reinterpret_cast<const __half2*>(&ne));
      const uint32_t gk = f16_bits(gam * kq) | 0x8000u;
      const uint32_t neg_g = gk | (gk << 16);
#pragma unroll 1
      for (int kb = 0; kb < 4 && ok; ++kb) {
        // ring slots of this round's two K-blocks (yhat, then sigma)
        int slot[2];
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
          slot[sl] = dslot;
          const int64_t use = duse;
          if (++dslot == kSlots) {
            dslot = 0;
            ++duse;
          }
          if (use > 0 && !(ok = wait_bar_warp(blk_empty(slot[sl]), (uint32_t)((use - 1) & 1), abort_flag))) break;
        }
        if (!ok) break;
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh) {
          const int half = h0 + hh;
          uint32_t w[P];
          const uint8_t* pw = rec + (2 * kb + half) * P * 4;
          if constexpr (P == 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(pw);
            w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
          } else if constexpr (P == 2) {
            const uint2 v = *reinterpret_cast<const uint2*>(pw);
            w[0] = v.x; w[1] = v.y;
          } else {
#pragma unroll
            for (int pp = 0; pp < P; ++pp) w[pp] = reinterpret_cast<const uint32_t*>(pw)[pp];
          }
#pragma unroll
          for (int sl = 0; sl < 2; ++sl) {
            uint8_t* dst = smem + kOffRing + slot[sl] * kSlotBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              uint32_t out[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int sh = 15 - (4 * e4 + e);
                if (sl == 1) {
                  const uint32_t xs = w[P - 1] << sh;
                  out[e] = (xs & 0x80008000u) ^ neg_g;            // sigma = 1 -> +gamma kq
                } else {
                  const uint32_t x0 = w[0] << sh;
                  uint32_t m;
                  if constexpr (B1 == 1) {
                    m = mag[0];
                  } else if constexpr (B1 == 2) {
                    const uint32_t x1 = w[1] << sh;
                    const uint32_t M = half_masks(x0 ^ x1);       // 0xffff where p0 != p1
                    m = (M & mag[0]) | (~M & mag[1]);
                  } else {
                    const uint32_t x1 = w[1] << sh, x2 = w[2] << sh;
                    const uint32_t M1 = half_masks(x0 ^ x1);
                    const uint32_t M2 = half_masks(x0 ^ x2);
                    const uint32_t lo = (M2 & mag[0]) | (~M2 & mag[1]);    // p1 == not p0 side
                    const uint32_t hi = (M2 & mag[2]) | (~M2 & mag[3]);
                    m = (M1 & lo) | (~M1 & hi);
                  }
                  out[e] = m | (~x0 & 0x80008000u);                // p0 = 0 -> negative
                }
              }
              const int ch = 4 * half + e4;
              *reinterpret_cast<uint4*>(dst + ((ch ^ (r & 7)) * 16)) = make_uint4(out[0], out[1], out[2], out[3]);
            }
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          bar_arrive(blk_full(slot[0]));
          bar_arrive(blk_full(slot[1]));
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) bar_arrive(stg_empty0 + 8u * sidx);
    }
    if (!ok) {
      atomicOr(status, 4);
      *abort_flag = 1;
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

// ---------------------------------------------------------------------------
// Exact re-ranking and the certificate: one warp per query.
//   T_a = the largest k-th entry of any one part's list (a lower bound of the
//   k-th best approximate score over all candidates), and only candidates with
//   approximate score >= T_a - 2 eps are scored exactly: at least k candidates
//   score >= T_a - eps exactly, and every skipped one scores below that.
//   The k best exact scores (ties to the smaller id) are written out unless a
//   part with a full list has its last approximate score + eps >= the k-th
//   exact score; then the query is queued for the exact scan.
// ---------------------------------------------------------------------------
template <int B1>
__global__ void __launch_bounds__(256) k_stc_refine(const Dev cb, const uint8_t* __restrict__ db, int64_t n_db, int nq,
                                                    int k, const float* __restrict__ qf,
                                                    const float* __restrict__ qinfo, const float* __restrict__ lsc,
                                                    const int32_t* __restrict__ lid, int Pmax, int64_t G,
                                                    unsigned* __restrict__ misc, int32_t* __restrict__ fq,
                                                    int32_t* __restrict__ ids, float* __restrict__ scores) {
  constexpr int P = B1 + 1, W = 8 * P, L = 1 << B1;
  __shared__ float s_q[8][2 * kD];
  __shared__ float s_sc[8][kCand];
  __shared__ int32_t s_id[8][kCand];
  __shared__ float s_cent[16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < 16) s_cent[threadIdx.x] = threadIdx.x < L ? cb.cent[threadIdx.x] : 0.f;
  __syncthreads();
  const int qi = blockIdx.x * 8 + warp;
  if (qi >= nq) return;
  const int64_t NT = (n_db + kR - 1) / kR, NQB = (nq + kQ - 1) / kQ, U = NQB * NT;
  const int qb = qi / kQ, ql = qi - qb * kQ;
  const int p_first = (int)unit_cta((int64_t)qb * NT, U, G);
  const int np = (int)unit_cta((int64_t)qb * NT + NT - 1, U, G) - p_first + 1;
  for (int e = lane; e < 2 * kD; e += 32) s_q[warp][e] = qf[(size_t)qi * 2 * kD + e];
  const float4 info = *reinterpret_cast<const float4*>(qinfo + (size_t)qi * 4);
  const float n_max = __uint_as_float(misc[0]), ng_max = __uint_as_float(misc[1]);
  const float kq = cb.qjl_const, cmax = fabsf(cb.cent[L - 1]);
  const float mass = n_max * cmax * info.y + ng_max * kq * info.z;
  const float eps = 1.5f * ((0.0009765625f + 0.000244140625f) * mass + n_max * info.z * 5.9604645e-8f) +
                    mass * 1.52587890625e-5f;
  auto at = [&](int p, int j) { return (((size_t)qb * Pmax + p) * kCand + j) * kQ + ql; };
  // T_a: the largest k-th entry of one part's list
  float Ta = -INFINITY;
  for (int p = lane; p < np; p += 32)
    if (lid[at(p, k - 1)] >= 0) Ta = fmaxf(Ta, lsc[at(p, k - 1)]);
#pragma unroll
  for (int o = 16; o; o >>= 1) Ta = fmaxf(Ta, __shfl_xor_sync(0xffffffffu, Ta, o));
  const float cut = Ta - 2.f * eps;
  __syncwarp();
  const uint32_t* recs = reinterpret_cast<const uint32_t*>(db);
  const uint32_t* nrm = reinterpret_cast<const uint32_t*>(db + norm_offset(cb, n_db));
  const float* qp = s_q[warp];
  float* ls = s_sc[warp];
  int32_t* li = s_id[warp];
  int cnt = 0;                                  // entries in the running top-k (warp-uniform)
  auto better = [](float sa, int32_t ia, float sb, int32_t ib) { return sa > sb || (sa == sb && ia < ib); };
  for (int p = 0; p < np; ++p) {
    const int32_t id = lid[at(p, lane)];
    const float ap = lsc[at(p, lane)];
    float ex = -INFINITY;
    const bool cand = id >= 0 && ap >= cut;
    if (cand) {
      // exact estimator of row id in fp32
      float a1 = 0.f, a2 = 0.f;
      const uint32_t* rec = recs + (size_t)id * W;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t w[P];
#pragma unroll
        for (int pp = 0; pp < P; ++pp) w[pp] = __ldg(rec + c * P + pp);
#pragma unroll 4
        for (int bt = 0; bt < 32; ++bt) {
          int idx = 0;
#pragma unroll
          for (int pp = 0; pp < B1; ++pp) idx |= (int)((w[pp] >> bt) & 1u) << (B1 - 1 - pp);
          a1 = fmaf(qp[32 * c + bt], s_cent[idx], a1);
          const float q2 = qp[kD + 32 * c + bt];
          a2 += ((w[P - 1] >> bt) & 1u) ? q2 : -q2;
        }
      }
      const uint32_t ne = __ldg(nrm + id);
      const __half2 h = *reinterpret_cast<const __half2*>(&ne);
      ex = __low2float(h) * fmaf(__high2float(h) * kq, a2, a1);
    }
    // insert this part's scored candidates into the running top-k
    const float kth = cnt < k ? -INFINITY : ls[k - 1];
    const int32_t kid = cnt < k ? INT32_MAX : li[k - 1];
    unsigned mask = __ballot_sync(0xffffffffu, cand && (cnt < k || better(ex, id, kth, kid)));
    while (mask) {
      const int src = __ffs(mask) - 1;
      mask &= mask - 1;
      const float s_new = __shfl_sync(0xffffffffu, ex, src);
      const int32_t id_new = __shfl_sync(0xffffffffu, id, src);
      if (lane == 0) {
        if (cnt < k || better(s_new, id_new, ls[k - 1], li[k - 1])) {
          int pos = cnt < k ? cnt : k - 1;
          while (pos > 0 && better(s_new, id_new, ls[pos - 1], li[pos - 1])) {
            ls[pos] = ls[pos - 1];
            li[pos] = li[pos - 1];
            --pos;
          }
          ls[pos] = s_new;
          li[pos] = id_new;
        }
      }
      cnt = min(cnt + 1, k);
      __syncwarp();
    }
  }
  // certificate
  bool certified = true;
  if (cnt >= k) {
    const float Sk = ls[k - 1];
    for (int p = lane; p < np; p += 32)
      if (lid[at(p, kCand - 1)] >= 0 && !(lsc[at(p, kCand - 1)] + eps < Sk)) certified = false;
  }
  certified = __all_sync(0xffffffffu, certified);
  for (int j = lane; j < k; j += 32) {
    ids[(size_t)qi * k + j] = j < cnt ? li[j] : -1;
    scores[(size_t)qi * k + j] = j < cnt ? ls[j] : -INFINITY;
  }
  if (!certified && lane == 0) fq[atomicAdd(misc + 2, 1u)] = qi;
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
namespace {
struct TcPlan {
  int64_t NT, NQB, U, G;
  int Pmax;
  int64_t off_aw, off_qf, off_qinfo, off_lsc, off_lid, off_fq, off_legacy, total;
};

TcPlan tc_plan(const Dev& cb, int64_t n_db, int nq, int k, int sms) {
  TcPlan p;
  p.NT = (n_db + kR - 1) / kR;
  p.NQB = (nq + kQ - 1) / kQ;
  p.U = p.NT * p.NQB;
  p.G = std::min<int64_t>(sms, p.U);
  p.Pmax = 1;
  for (int64_t qb = 0; qb < p.NQB; ++qb)
    p.Pmax = std::max<int>(p.Pmax, (int)(unit_cta(qb * p.NT + p.NT - 1, p.U, p.G) - unit_cta(qb * p.NT, p.U, p.G) + 1));
  int64_t off = align256(kMiscWords * 4);
  p.off_aw = off;
  off += align256(p.NQB * 256 * kQ * 4);
  p.off_qf = off;
  off += align256((int64_t)nq * 2 * kD * 4);
  p.off_qinfo = off;
  off += align256((int64_t)nq * 16);
  p.off_lsc = off;
  off += align256(p.NQB * p.Pmax * kCand * kQ * 4);
  p.off_lid = off;
  off += align256(p.NQB * p.Pmax * kCand * kQ * 4);
  p.off_fq = off;
  off += align256((int64_t)nq * 4);
  p.off_legacy = off;
  off += search_workspace_bytes(cb, n_db, nq, k, sms);
  p.total = off;
  return p;
}
}  // namespace

bool search_tc_applies(const Dev& cb, int k) { return cb.d == kD && cb.kind == 0 && cb.mode == 0 && cb.extra == 0 && k <= kMaxKTc; }

int64_t search_tc_workspace_bytes(const Dev& cb, int64_t n_db, int nq, int k, int sms) {
  return tc_plan(cb, n_db, nq, k, sms).total;
}

template <int B1>
static cudaError_t scan_t(const TcPlan& pl, const Dev& cb, const uint8_t* db, int64_t n_db, int nq, uint8_t* ws,
                          int* status, cudaStream_t s) {
  constexpr uint32_t kSmemBytes = Smem<B1>::kBytes;
  static cudaError_t configured = cudaFuncSetAttribute(k_stc_scan<B1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       (int)kSmemBytes);
  if (configured != cudaSuccess) return configured;
  k_stc_scan<B1><<<(int)pl.G, kThreads, kSmemBytes, s>>>(
      cb, db, n_db, nq, reinterpret_cast<const uint32_t*>(ws + pl.off_aw),
      reinterpret_cast<const float*>(ws + pl.off_qinfo), reinterpret_cast<float*>(ws + pl.off_lsc),
      reinterpret_cast<int32_t*>(ws + pl.off_lid), pl.Pmax, status);
  return cudaGetLastError();
}

template <int B1>
static void refine_t(const TcPlan& pl, const Dev& cb, const uint8_t* db, int64_t n_db, int nq, int k, uint8_t* ws,
                     int32_t* ids, float* scores, cudaStream_t s) {
  k_stc_refine<B1><<<(nq + 7) / 8, 256, 0, s>>>(
      cb, db, n_db, nq, k, reinterpret_cast<const float*>(ws + pl.off_qf),
      reinterpret_cast<const float*>(ws + pl.off_qinfo), reinterpret_cast<const float*>(ws + pl.off_lsc),
      reinterpret_cast<const int32_t*>(ws + pl.off_lid), pl.Pmax, pl.G, reinterpret_cast<unsigned*>(ws),
      reinterpret_cast<int32_t*>(ws + pl.off_fq), ids, scores);
}

cudaError_t launch_search_tc(const Dev& cb, const uint8_t* db, int64_t n_db, const float* q, int nq, int d_in, int k,
                             int32_t* ids, float* scores, uint8_t* ws, int sms, int* status, cudaStream_t s) {
  const TcPlan pl = tc_plan(cb, n_db, nq, k, sms);
  unsigned* misc = reinterpret_cast<unsigned*>(ws);
  static cudaError_t configured = cudaFuncSetAttribute(k_stc_prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       kPrepQ * kD * 4 * 3);
  if (configured != cudaSuccess) return configured;
  k_stc_prep<<<(int)(pl.NQB * (kQ / kPrepQ)), 256, kPrepQ * kD * 4 * 3, s>>>(
      cb, q, nq, d_in, reinterpret_cast<uint32_t*>(ws + pl.off_aw), reinterpret_cast<float*>(ws + pl.off_qf),
      reinterpret_cast<float*>(ws + pl.off_qinfo), misc);
  k_stc_dbmax<<<sms * 2, 256, 0, s>>>(cb, db, n_db, misc);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  switch (cb.b1) {
    case 1: e = scan_t<1>(pl, cb, db, n_db, nq, ws, status, s); break;
    case 2: e = scan_t<2>(pl, cb, db, n_db, nq, ws, status, s); break;
    default: e = scan_t<3>(pl, cb, db, n_db, nq, ws, status, s); break;
  }
  if (e != cudaSuccess) return e;
  switch (cb.b1) {
    case 1: refine_t<1>(pl, cb, db, n_db, nq, k, ws, ids, scores, s); break;
    case 2: refine_t<2>(pl, cb, db, n_db, nq, k, ws, ids, scores, s); break;
    default: refine_t<3>(pl, cb, db, n_db, nq, k, ws, ids, scores, s); break;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // queries that failed the certificate: the exact scan, over those queries only
  return launch_search_subset(cb, db, n_db, q, nq, d_in, k, ids, scores, ws + pl.off_legacy, sms,
                              reinterpret_cast<const int32_t*>(ws + pl.off_fq), misc + 2, s);
}


}  // namespace tq
