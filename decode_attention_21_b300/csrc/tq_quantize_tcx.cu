// Batch compression on the 5th-generation tensor cores with the A operands
// (X, then the residual) in tensor memory: d = 256 vectors (the search
// database: rows of 200 coordinates zero-padded to 256, fp32 or bf16), and
// d = 128 fp32 vectors (bf16 ones take the two-group kernel of
// tq_quantize_tc.cu), and polar-mode batches of either width and input type.
//
// [xujun] note-189244, 常见问题 (vector search over a compressed database),
//   第一步：PolarQuant (recursive radius / angle pairing);
// [suzuke] "TurboQuant: compressing AI consciousness", 技術上怎麼做到的:
//   第一步 multiply by the random orthogonal matrix, 第二步 Max-Lloyd code per
//   coordinate, 第三步 1-bit sign of the projected residual.
//
// One CTA per SM (16 warps) walks 128-row tiles.  Per tile:
//   * the warps load their rows of X straight from global memory (thread:
//     row 32 (w % 4) + lane, coordinates d/4 (w / 4) .. + d/4 - 1; the CTA's next
//     tile is prefetched into L2 by one bulk prefetch), split each value
//     into bf16 hi + lo and store the pairs to tensor memory: the A operand;
//   * thread 0 issues the rotation Y = X_hi Pi_hi^T + X_hi Pi_lo^T (+ X_lo
//     Pi_hi^T for fp32 input) as M128 N(d) K16 MMAs.  Pi_hi, Pi_lo (and S for
//     the sketch) stream through a ring of four shared-memory slots, one
//     64-wide K block of one matrix per slot (d x 64 bf16: TMA, 128-byte
//     swizzle), in a fixed order the loads and the MMAs both follow;
//   * epilogue 1: norms, stage-1 cells (bisection), residual r = y/n - yhat
//     as bf16 hi + lo into the tensor-memory columns X used.  Polar mode: each
//     thread codes the angles of levels 1..5 inside its 32-coordinate blocks
//     (slots 0..30 of the word column), the squared block radii meet in
//     shared memory and every thread of the row takes the top levels'
//     decisions (slot 31 of the word columns, heap order); the reproduction
//     walks back down from root radius 1 for the residual;
//   * thread 0 issues the sketch Z = R_hi S^T + R_lo S^T into the columns of Y;
//   * epilogue 2: sign words of Z, gamma = ||r||, record and fp16 norms.
// TMEM: Y / Z in columns 0..d-1, X and then R (bf16 pairs, coordinate k in
// column k / 2) from column 256 (hi) and 384 (lo).
// Every wait is bounded; on a timeout the kernel records an error, waits
// (bounded) for its own copies and MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tq_internal.cuh"
#include "tq_polar.cuh"
#include "tq_tc.cuh"

namespace tq {

namespace {

using namespace tc;

constexpr int kRows = 128;
constexpr int kThreads = 512;
constexpr int kSlots = 4;                                // ring of B-operand K blocks
// shared memory map per width: ring of d x 64 bf16 slots, then float
// red1[d/32][128], red2[4][128], red3[d/32][128] (polar block radii), the
// mbarriers full[kSlots], empty[kSlots], y, z, and the TMEM base
template <int D>
struct Map {
  static constexpr uint32_t kSlotBytes = D * 128;
  static constexpr uint32_t kOffRing = 0;
  static constexpr uint32_t kOffRed = kSlots * kSlotBytes;
  static constexpr uint32_t kOffBar = kOffRed + (2 * (D / 32) + 4) * kRows * 4;
  static constexpr uint32_t kOffTmem = kOffBar + 8 * (2 * kSlots + 2);
  static constexpr uint32_t kSmemBytes = kOffTmem + 16 + 1024;    // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory");
};
constexpr uint32_t kTmemCols = 512;

// Loads of one tile, in ring order: Pi_hi and Pi_lo of the d/64 K blocks
// (interleaved), then S of the K blocks (PROD only).
template <int D, bool PROD>
__host__ __device__ constexpr int loads_per_tile() { return (PROD ? 3 : 2) * (D / 64); }

}  // namespace

// POLAR: the polar stage 1 (B1 bits per angle) instead of the scalar one.
template <int D, int B1, bool PROD, bool F32, bool POLAR>
__global__ void __launch_bounds__(kThreads, 1)
    k_quantize_tcx(const __grid_constant__ CUtensorMap tm_pihi, const __grid_constant__ CUtensorMap tm_pilo,
                     const __grid_constant__ CUtensorMap tm_s, const Dev cb, uint8_t* __restrict__ cache,
                     int64_t cache_rows, const void* __restrict__ x, int64_t n, int d_in,
                     const int64_t* __restrict__ dst_rows, int* __restrict__ status) {
  // a programmatic dependent may start now: it reads none of the rows written
  // here and waits for this grid before it completes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so the
  // compiler keeps every access through smem in the shared space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp & 3;                            // TMEM lane quarter
  const int cq = warp >> 2;                          // coordinates (d/4) cq .. (d/4) cq + d/4 - 1
  const int m = 32 * q + lane;                       // tile row = TMEM lane
  using M = Map<D>;
  constexpr int QC = D / 4;                          // coordinates per thread
  constexpr int NCH = QC / 32;                       // 32-coordinate word columns per thread
  constexpr int KB = D / 64;                         // K blocks
  constexpr uint32_t kIdesc = idesc_bf16(D);
  float* red1 = reinterpret_cast<float*>(smem + M::kOffRed);
  float* red2 = red1 + (D / 32) * kRows;
  float* red3 = red2 + 4 * kRows;
  const uint32_t bar0 = sbase + M::kOffBar;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (kSlots + s); };
  const uint32_t bar_y = bar0 + 8u * (2 * kSlots), bar_z = bar_y + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + M::kOffTmem);
  constexpr int P = B1 + (PROD ? 1 : 0);
  constexpr int NL = loads_per_tile<D, PROD>();
  const int W = cb.W;
  const int64_t ntiles = (n + kRows - 1) / kRows;
  __shared__ float s_cent[16], s_bnd[16];
  __shared__ polar::Tables tpol;                   // polar mode only
  float lt[7];
  if constexpr (!POLAR) heap_levels<B1>(cb.bound, lt);
  float cr[4];                                       // centroids in registers (b' <= 2)
#pragma unroll
  for (int k = 0; k < 4; ++k) cr[k] = cb.cent[k];
  if (tid < 16) {
    s_cent[tid] = cb.cent[tid];
    s_bnd[tid] = cb.bound[tid];
  }
  if constexpr (POLAR) polar::load_tables(cb, tpol, tid, kThreads);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int k = 0; k < 2 * kSlots + 2; ++k) mbar_init(bar0 + 8u * k, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_hi = tmem + 256, t_lo = tmem + 384;   // X, then R
  const uint32_t lane_off = (uint32_t)(32 * q) << 16;

  // Ring bookkeeping (thread 0): load g of the CTA (g = tile_local * NL + c)
  // goes to slot g % kSlots; its data is there at phase (g / kSlots) & 1 of
  // the slot's full barrier, and the slot is free again once the MMAs that
  // read it commit to its empty barrier.
  const int64_t first = blockIdx.x, step = gridDim.x;
  const int64_t my_tiles = first < ntiles ? (ntiles - 1 - first) / step + 1 : 0;
  const int64_t total_loads = my_tiles * NL;
  int64_t g_issued = 0, g_done = 0;                    // loads issued; loads whose MMAs committed
  auto issue_load = [&](int64_t g) {                   // thread 0
    const int s = (int)(g % kSlots);
    if (g >= kSlots && !mbar_wait(bar_empty(s), (uint32_t)(((g / kSlots) - 1) & 1))) return false;
    const int c = (int)(g % NL);
    const CUtensorMap* map = c < 2 * KB ? ((c & 1) ? &tm_pilo : &tm_pihi) : &tm_s;
    const int kb = c < 2 * KB ? (c >> 1) : c - 2 * KB;
    mbar_expect_tx(bar_full(s), M::kSlotBytes);
    tma_load_2d(sbase + M::kOffRing + s * M::kSlotBytes, map, 64 * kb, 0, bar_full(s));
    return true;
  };
  bool ok = true;
  if (tid == 0)
    for (; g_issued < total_loads && g_issued < kSlots; ++g_issued) ok = ok && issue_load(g_issued);
  // MMAs of load g (thread 0): wait for its data, issue, commit the slot;
  // then refill the slot of load g - 1 (whose MMAs are queued ahead of
  // these) with load g - 1 + kSlots
  bool first_wait = true;
  auto consume = [&](int64_t g, auto&& issue_mmas) {
    const int s = (int)(g % kSlots);
    if (!mbar_wait(bar_full(s), (uint32_t)((g / kSlots) & 1), first_wait ? cb.first_wait : kSpinLimit)) return false;
    first_wait = false;
    fence_after();
    issue_mmas(sbase + M::kOffRing + s * M::kSlotBytes);
    mma_commit(bar_empty(s));
    g_done = g + 1;
    if (g >= 1 && g_issued < total_loads && g_issued == g - 1 + kSlots) {
      if (!issue_load(g_issued)) return false;
      ++g_issued;
    }
    return true;
  };

  bool pend_y = false, pend_z = false;
  int it = 0;
  for (int64_t tile = first; tile < ntiles; tile += step, ++it) {
    const int64_t g0 = (int64_t)it * NL;
    // the next tile's rows into L2 while this one is worked on
    if (tid == 0 && tile + step < ntiles) {
      const int64_t r0 = (tile + step) * kRows, nr = min((int64_t)kRows, n - r0);
      const size_t rb = (size_t)d_in * (F32 ? 4 : 2);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const uint8_t*>(x) + r0 * rb),
                   "r"((uint32_t)(nr * rb))
                   : "memory");
    }
    // ---- X rows into tensor memory as bf16 hi + lo pairs
    {
      const int64_t row = tile * kRows + m;
#pragma unroll
      for (int piece = 0; piece < QC / 16; ++piece) {
        const int k0 = QC * cq + 16 * piece;             // first coordinate of the piece
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0.f;
        if (row < n) {
          if constexpr (F32) {
            const float* src = static_cast<const float*>(x) + row * d_in;
#pragma unroll
            for (int e = 0; e < 16; e += 4)
              if (k0 + e < d_in) {
                const float4 f = __ldg(reinterpret_cast<const float4*>(src + k0 + e));
                v[e] = f.x;
                v[e + 1] = f.y;
                v[e + 2] = f.z;
                v[e + 3] = f.w;
              }
          } else {
            const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(x) + row * d_in;
#pragma unroll
            for (int e = 0; e < 16; e += 8)
              if (k0 + e < d_in) {
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(src + k0 + e));
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  v[e + 2 * t] = __uint_as_float(w4[t] << 16);
                  v[e + 2 * t + 1] = __uint_as_float(w4[t] & 0xFFFF0000u);
                }
              }
          }
        }
        uint32_t xh[8], xl[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const uint32_t hb = bf16x2(v[e], v[e + 1]);
          xh[e >> 1] = hb;
          xl[e >> 1] = F32 ? bf16x2(v[e] - __uint_as_float(hb << 16), v[e + 1] - __uint_as_float(hb & 0xFFFF0000u))
                           : 0u;
        }
        tmem_st8(t_hi + lane_off + (uint32_t)(k0 >> 1), xh);
        if (F32) tmem_st8(t_lo + lane_off + (uint32_t)(k0 >> 1), xl);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    // ---- rotation: loads g0 .. g0 + 2 KB - 1 (Pi_hi, Pi_lo of the K blocks)
    bool good = true;
    if (tid == 0) {
      fence_after();
      for (int c = 0; c < 2 * KB && good; ++c) {
        const int kb = c >> 1;
        good = consume(g0 + c, [&](uint32_t slot) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bd = sw128_desc(slot + 32 * ks);
            const uint32_t acol = (uint32_t)(32 * kb + 8 * ks);
            mma_bf16_ta(tmem, t_hi + acol, bd, kIdesc, (c | ks) != 0);
            if (F32 && !(c & 1)) mma_bf16_ta(tmem, t_lo + acol, bd, kIdesc, 1);
          }
        });
      }
      if (good) mma_commit(bar_y);
    }
    if (!__syncthreads_and(good)) {
      ok = false;
      break;
    }
    pend_y = true;
    if (!__syncthreads_and(mbar_wait(bar_y, it & 1))) {
      ok = false;
      break;
    }
    pend_y = false;
    fence_after();

    // ---- epilogue 1: norms (pass 1), codes and the residual operand (pass 2)
#pragma unroll
    for (int h = 0; h < NCH; ++h) {
      float v[32];
      tmem_ld32(tmem + lane_off + QC * cq + 32 * h, v);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) ss = fmaf(v[e], v[e], ss);
      red1[(NCH * cq + h) * kRows + m] = ss;
    }
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) tot += red1[k * kRows + m];
    const float nrm = sqrtf(tot);
    const float inv = nrm > 0.f ? 1.f / nrm : 0.f;
    uint32_t words[NCH][P];
    float gs = 0.f;
    if constexpr (POLAR) {
      polar::epilogue<D, NCH, B1, PROD>(tpol, tmem + lane_off, t_hi + lane_off, t_lo + lane_off, NCH * cq, inv,
                                         red3, m, words, gs, [] { __syncthreads(); });
    } else {
#pragma unroll
    for (int h = 0; h < NCH; ++h) {
#pragma unroll
      for (int p = 0; p < P; ++p) words[h][p] = 0u;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[16];
        tmem_ld16(tmem + lane_off + QC * cq + 32 * h + 16 * half, v);
        uint32_t rh[8], rl[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          float r2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float y = v[e + u] * inv;
            float r;
            if constexpr (B1 <= 2) {
              r = y - cell_cent<B1>(y, lt, cr, words[h], 16 * half + e + u);
            } else {
              const int idx = cell_heap<B1>(y, lt, s_bnd, words[h], 16 * half + e + u);
              r = y - s_cent[idx];
            }
            gs = fmaf(r, r, gs);
            r2[u] = r;
          }
          const uint32_t hb = bf16x2(r2[0], r2[1]);
          rh[e >> 1] = hb;
          rl[e >> 1] = bf16x2(r2[0] - __uint_as_float(hb << 16), r2[1] - __uint_as_float(hb & 0xFFFF0000u));
        }
        if (PROD) {
          const uint32_t col = (uint32_t)(QC / 2 * cq + 16 * h + 8 * half);
          tmem_st8(t_hi + lane_off + col, rh);
          tmem_st8(t_lo + lane_off + col, rl);
        }
      }
    }
    }
    red2[cq * kRows + m] = gs;
    if (PROD) asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    fence_before();
    __syncthreads();
    // ---- sketch: loads g0 + 2 KB .. g0 + 3 KB - 1 (S of the K blocks)
    uint32_t sword[NCH];
#pragma unroll
    for (int h = 0; h < NCH; ++h) sword[h] = 0u;
    float gamma = 0.f;
    if (PROD) {
      good = true;
      if (tid == 0) {
        fence_after();
        for (int c = 2 * KB; c < 3 * KB && good; ++c) {
          const int kb = c - 2 * KB;
          good = consume(g0 + c, [&](uint32_t slot) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t bd = sw128_desc(slot + 32 * ks);
              const uint32_t acol = (uint32_t)(32 * kb + 8 * ks);
              mma_bf16_ta(tmem, t_hi + acol, bd, kIdesc, (kb | ks) != 0);
              mma_bf16_ta(tmem, t_lo + acol, bd, kIdesc, 1);
            }
          });
        }
        if (good) mma_commit(bar_z);
      }
      if (!__syncthreads_and(good)) {
        ok = false;
        break;
      }
      pend_z = true;
      if (!__syncthreads_and(mbar_wait(bar_z, it & 1))) {
        ok = false;
        break;
      }
      pend_z = false;
      fence_after();
#pragma unroll
      for (int h = 0; h < NCH; ++h) {
        float v[32];
        tmem_ld32(tmem + lane_off + QC * cq + 32 * h, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) sword[h] |= (v[e] >= 0.f ? 1u : 0u) << e;
      }
      float g2 = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) g2 += red2[k * kRows + m];
      gamma = sqrtf(g2);
    }
    // ---- store
    const int64_t row = tile * kRows + m;
    const int64_t dst = row < n ? (dst_rows ? dst_rows[row] : row) : -1;
    if (row < n && (dst < 0 || dst >= cache_rows) && cq == 0) atomicOr(status, kBadRow);  // skipped
    if (dst >= 0 && dst < cache_rows) {
      uint32_t* rec = reinterpret_cast<uint32_t*>(cache) + dst * W;
#pragma unroll
      for (int h = 0; h < NCH; ++h) {
        const int wc = NCH * cq + h;
        if constexpr (PROD) words[h][B1] = sword[h];
        if constexpr (P == 4) {
          *reinterpret_cast<uint4*>(rec + wc * P) = make_uint4(words[h][0], words[h][1], words[h][2], words[h][3]);
        } else if constexpr (P == 2) {
          *reinterpret_cast<uint2*>(rec + wc * P) = make_uint2(words[h][0], words[h][1]);
        } else {
#pragma unroll
          for (int p = 0; p < P; ++p) rec[wc * P + p] = words[h][p];
        }
      }
      if (cq == 0) {
        uint8_t* norms = cache + norm_offset(cb, cache_rows);
        if (PROD)
          reinterpret_cast<__half2*>(norms)[dst] = __floats2half2_rn(nrm, gamma);
        else
          reinterpret_cast<__half*>(norms)[dst] = __float2half_rn(nrm);
      }
    }
    // every thread has read Z and the reduction entries before the next
    // tile's X overwrites tensor memory and its rotation the Z columns
    fence_before();
    __syncthreads();
    fence_after();
  }
  if (!ok) {
    if (tid == 0) {
      atomicOr(status, 1);
      // our own MMAs and copies in flight finish (bounded waits)
      if (pend_y) mbar_wait(bar_y, it & 1);
      if (pend_z) mbar_wait(bar_z, it & 1);
      for (int64_t g = g_done; g < g_issued; ++g) mbar_wait(bar_full((int)(g % kSlots)), (uint32_t)((g / kSlots) & 1));
      if (g_done > 0) {
        const int64_t g = g_done - 1;
        mbar_wait(bar_empty((int)(g % kSlots)), (uint32_t)((g / kSlots) & 1));
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

template <int D, int B1, bool PROD, bool F32, bool POLAR>
static cudaError_t launch_tcx_t(const CUtensorMap& tm_pihi, const CUtensorMap& tm_pilo, const CUtensorMap& tm_s,
                                const Dev& cb, uint8_t* cache, int64_t cache_rows, const void* x, int64_t n, int d_in,
                                const int64_t* dst_rows, int* status, int sms, cudaStream_t s) {
  constexpr uint32_t smem = Map<D>::kSmemBytes;
  static cudaError_t configured =
      cudaFuncSetAttribute(k_quantize_tcx<D, B1, PROD, F32, POLAR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (configured != cudaSuccess) return configured;
  const int64_t ntiles = (n + kRows - 1) / kRows;
  const int grid = (int)(ntiles < sms ? ntiles : sms);
  k_quantize_tcx<D, B1, PROD, F32, POLAR><<<grid, kThreads, smem, s>>>(tm_pihi, tm_pilo, tm_s, cb, cache, cache_rows,
                                                                       x, n, d_in, dst_rows, status);
  return cudaGetLastError();
}

// Scalar mode: d = 256 in either input type; d = 128 for fp32 input (no
// extra-bit words).  Polar mode: d = 128 or 256, either input type.
cudaError_t launch_quantize_tcx(const CUtensorMap& tm_pihi, const CUtensorMap& tm_pilo, const CUtensorMap& tm_s,
                                const Dev& cb, uint8_t* cache, int64_t cache_rows, const void* x, bool f32, int64_t n,
                                int d_in, const int64_t* dst_rows, int* status, int sms, cudaStream_t s) {
#define TQ_TC(DD, B, PR, F, PO)                                                                                  \
  return launch_tcx_t<DD, B, PR, F, PO>(tm_pihi, tm_pilo, tm_s, cb, cache, cache_rows, x, n, d_in, dst_rows, status, \
                                        sms, s)
#define TQ_TC_F(B, PR)                             \
  if (cb.d == 128) TQ_TC(128, B, PR, true, false); \
  if (f32) TQ_TC(256, B, PR, true, false);         \
  TQ_TC(256, B, PR, false, false)
#define TQ_TC_P(B, PR)                      \
  if (cb.d == 128) {                        \
    if (f32) TQ_TC(128, B, PR, true, true); \
    TQ_TC(128, B, PR, false, true);         \
  }                                         \
  if (f32) TQ_TC(256, B, PR, true, true);   \
  TQ_TC(256, B, PR, false, true)
  if (cb.mode != 0) {
    if (cb.kind == 0) {
      switch (cb.b1) {
        case 1: TQ_TC_P(1, true);
        case 2: TQ_TC_P(2, true);
        default: TQ_TC_P(3, true);
      }
    }
    switch (cb.b1) {
      case 1: TQ_TC_P(1, false);
      case 2: TQ_TC_P(2, false);
      case 3: TQ_TC_P(3, false);
      default: TQ_TC_P(4, false);
    }
  }
  if (cb.kind == 0) {
    switch (cb.b1) {
      case 1: TQ_TC_F(1, true);
      case 2: TQ_TC_F(2, true);
      default: TQ_TC_F(3, true);
    }
  }
  switch (cb.b1) {
    case 1: TQ_TC_F(1, false);
    case 2: TQ_TC_F(2, false);
    case 3: TQ_TC_F(3, false);
    default: TQ_TC_F(4, false);
  }
#undef TQ_TC_P
#undef TQ_TC_F
#undef TQ_TC
}

}  // namespace tq
