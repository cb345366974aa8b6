// Batch compression on the 5th-generation tensor cores (tcgen05 + TMEM, fed
// by TMA): the two dense contractions of the method, the rotation
// Y = X Pi^T and the QJL projection Z = R S^T, for 128-row tiles of bf16
// input vectors (d = 128, scalar stage 1).
//
// [suzuke] "TurboQuant: compressing AI consciousness", 技術上怎麼做到的:
//   第一步 multiply by the random orthogonal matrix, 第二步 Max-Lloyd code per
//   coordinate, 第三步 1-bit sign of the projected residual.
//
// Per tile (persistent CTAs, 16 warps):
//   TMA: X tile (128 x 128 bf16, 128B-swizzled, two 64-column blocks); Pi and
//        S once per CTA.
//   MMA (one thread): Y = X Pi_hi^T + X Pi_lo^T into TMEM columns 0..127
//        (Pi = Pi_hi + Pi_lo, both bf16: fp32-accurate rotation of bf16 x).
//   epilogue 1 (warp w: TMEM lanes 32 (w%4).., columns 32 (w/4)..): n = ||y||
//        (an outlier-channel split: each group's own norm), codes by
//        bisection over the boundaries (each level one comparison, setting
//        that level's code-plane bit), residual r = y/n - yhat written to
//        shared memory as bf16 hi + lo in the MMA's swizzled K-major layout.
//   MMA: Z = R_hi S^T + R_lo S^T into TMEM columns 128..255.
//   epilogue 2: sign words of Z, gamma = ||r||, record and fp16 norms.
// Every wait on an mbarrier is bounded; on a timeout the kernel records an
// error code, waits (bounded) for its own copies and MMAs, frees its TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "tq_internal.cuh"
#include "tq_polar.cuh"
#include "tq_tc.cuh"

namespace tq {

namespace {

constexpr int kRows = 128;
constexpr int kThreads = 512;                          // two groups of 8 warps
constexpr int kStages = 3;                             // X tiles in flight
constexpr uint32_t kBlockBytes = kRows * 128;          // 64 bf16 columns x 128 rows
constexpr uint32_t kTileBytes = 2 * kBlockBytes;       // 128 columns
// shared memory map (offsets from a 1024-aligned base)
constexpr uint32_t kOffX = 0;                          // kStages x kTileBytes
constexpr uint32_t kOffPiHi = kStages * kTileBytes;
constexpr uint32_t kOffPiLo = kOffPiHi + kTileBytes;
constexpr uint32_t kOffS = kOffPiLo + kTileBytes;
constexpr uint32_t kOffRed = kOffS + kTileBytes;       // float red1[2][4][128], red2[2][4][128], red3[2][4][128]
constexpr uint32_t kOffBar = kOffRed + 3 * 2 * 4 * kRows * 4;
// mbarriers: full[kStages], const, y[2], z[2]; then the TMEM base and the
// per-stage counts of issued and consumed loads
constexpr uint32_t kOffTmem = kOffBar + 8 * (kStages + 5);
constexpr uint32_t kOffCnt = kOffTmem + 8;
constexpr uint32_t kSmemBytes = kOffCnt + 8 * kStages + 1024;   // + alignment slack
constexpr uint32_t kTmemCols = 512;                    // per group: Y / Z 128, R_hi 64, R_lo 64
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr uint32_t kIdesc = tc::idesc_bf16(128);
using namespace tc;

}  // namespace

// POLAR: the recursive-polar stage 1 (B1 bits per angle) instead of the
// scalar one (no extra-bit words).
template <int B1, bool PROD, bool EXT, bool POLAR>
__global__ void __launch_bounds__(kThreads, 1)
    k_quantize_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_pihi,
                  const __grid_constant__ CUtensorMap tm_pilo, const __grid_constant__ CUtensorMap tm_s, const Dev cb,
                  uint8_t* __restrict__ cache, int64_t cache_rows, int64_t n, const int64_t* __restrict__ dst_rows,
                  int* __restrict__ status) {
  // a programmatic dependent (the query prep) may start now: it reads none of
  // the rows written here and waits for this grid before it completes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = warp >> 3;                           // tile group: local tiles g, g + 2, ...
  const bool leader = (tid & 255) == 0;              // the group's MMA and TMA issuer
  const int q = warp & 3;                            // TMEM lane quarter
  const int wh = (warp >> 2) & 1;                    // column groups 2 wh, 2 wh + 1
  const int m = 32 * q + lane;                       // tile row = TMEM lane
  float* red1 = reinterpret_cast<float*>(smem + kOffRed) + g * 4 * kRows;
  float* red2 = reinterpret_cast<float*>(smem + kOffRed) + (2 + g) * 4 * kRows;
  float* red3 = reinterpret_cast<float*>(smem + kOffRed) + (4 + g) * 4 * kRows;   // polar block radii
  const uint32_t bar0 = sbase + kOffBar;
  auto bar_full = [&](int st) { return bar0 + 8u * st; };
  const uint32_t bar_const = bar0 + 8u * kStages;
  const uint32_t bar_y = bar0 + 8u * (kStages + 1 + g), bar_z = bar0 + 8u * (kStages + 3 + g);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  int* n_issued = reinterpret_cast<int*>(smem + kOffCnt);        // loads issued into each stage
  int* n_taken = n_issued + kStages;                              // loads waited for
  const int64_t ntiles = (n + kRows - 1) / kRows;
  constexpr int b1 = B1, P = B1 + (PROD ? 1 : 0);
  constexpr bool prod = PROD;
  const int W = cb.W;
  // stage-1 tables in shared memory (the middle boundaries also in registers)
  __shared__ float s_cent[16], s_centx[32], s_bnd[16], s_bndx[32];
  float lt[7], ltx[7];
  heap_levels<B1>(cb.bound, lt);
  float cr[4];                                       // centroids in registers (b' <= 2)
#pragma unroll
  for (int k = 0; k < 4; ++k) cr[k] = cb.cent[k];
  heap_levels<EXT ? B1 + 1 : 1>(cb.bound_x, ltx);
  if (tid < 16) {
    s_cent[tid] = cb.cent[tid];
    s_bnd[tid] = cb.bound[tid];
  }
  if (tid < 32) {
    s_centx[tid] = cb.cent_x[tid];
    s_bndx[tid] = cb.bound_x[tid];
  }
  // outlier-channel split: word columns cg < kx are group A, with its own norms
  const int kx = cb.split ? cb.extra / 32 : 0;
  __shared__ polar::Tables tpol;                     // polar mode only
  if constexpr (POLAR) polar::load_tables(cb, tpol, tid, kThreads);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int k = 0; k < kStages + 5; ++k) mbar_init(bar0 + 8u * k, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < 2 * kStages) n_issued[tid] = 0;
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tg = tmem + 256u * g;               // Y, then Z: columns +0..127
  const uint32_t t_rhi = tg + 128, t_rlo = tg + 192; // residual operand (bf16 pairs)
  const uint32_t lane_off = (uint32_t)(32 * q) << 16;

  // local tile it of this CTA is tile blockIdx.x + it * gridDim.x, staged in
  // X stage it % kStages; its load is issued by the prologue (it < kStages)
  // or by the group that ran tile it - kStages, once that tile's rotation
  // has consumed the stage
  const int64_t first = blockIdx.x, step = gridDim.x;
  auto load_x = [&](int64_t it) {
    const int st = (int)(it % kStages);
    const uint32_t dst = sbase + kOffX + st * kTileBytes;
    mbar_expect_tx(bar_full(st), kTileBytes);
    for (int kb = 0; kb < 2; ++kb)
      tma_load_2d(dst + kb * kBlockBytes, &tm_x, 64 * kb, (int)((first + it * step) * kRows), bar_full(st));
    atomicAdd(&n_issued[st], 1);
  };
  if (tid == 0 && first < ntiles) {
    mbar_expect_tx(bar_const, (prod ? 3 : 2) * kTileBytes);
    for (int kb = 0; kb < 2; ++kb) {
      tma_load_2d(sbase + kOffPiHi + kb * kBlockBytes, &tm_pihi, 64 * kb, 0, bar_const);
      tma_load_2d(sbase + kOffPiLo + kb * kBlockBytes, &tm_pilo, 64 * kb, 0, bar_const);
      if (prod) tma_load_2d(sbase + kOffS + kb * kBlockBytes, &tm_s, 64 * kb, 0, bar_const);
    }
    for (int it = 0; it < kStages && first + it * step < ntiles; ++it) load_x(it);
  }
  bool ok = true;
  bool const_pending = first < ntiles;   // Pi / S loads not yet waited for
  if (first < ntiles) ok = __syncthreads_and(mbar_wait(bar_const, 0, cb.first_wait)) != 0;
  if (ok) const_pending = false;
  // this group's MMA commits not yet waited for (drained on a timeout)
  bool pend_y = false, pend_z = false;
  int j = 0;                              // this group's tile count (mbarrier phases)

  for (int64_t it = g; ok && first + it * step < ntiles; it += 2, ++j) {
    const int64_t tile = first + it * step;
    const int st = (int)(it % kStages);
    const uint32_t xs = sbase + kOffX + st * kTileBytes;
    // ---- rotation on the tensor cores: Y = X Pi_hi^T + X Pi_lo^T
    bool good = true;
    if (leader) {
      good = mbar_wait(bar_full(st), (uint32_t)((it / kStages) & 1));
      if (good) {
        atomicAdd(&n_taken[st], 1);
        fence_after();
        for (int kb = 0; kb < 2; ++kb)
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tg, sw128_desc(xs + kb * kBlockBytes + 32 * ks),
                     sw128_desc(sbase + kOffPiHi + kb * kBlockBytes + 32 * ks), kIdesc, (kb | ks) != 0);
        for (int kb = 0; kb < 2; ++kb)
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tg, sw128_desc(xs + kb * kBlockBytes + 32 * ks),
                     sw128_desc(sbase + kOffPiLo + kb * kBlockBytes + 32 * ks), kIdesc, 1);
        mma_commit(bar_y);
      }
    }
    if (!group_and(g, good)) {
      ok = false;
      break;
    }
    pend_y = true;
    if (!group_and(g, mbar_wait(bar_y, j & 1))) {
      ok = false;
      break;
    }
    pend_y = false;
    fence_after();
    // the stage is consumed: fetch local tile it + kStages into it
    if (leader && first + (it + kStages) * step < ntiles) load_x(it + kStages);

    // ---- epilogue 1: norms (pass 1), codes and the residual operand (pass 2)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int cg = 2 * wh + h;
      float v[32];
      tmem_ld32(tg + lane_off + 32 * cg, v);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) ss = fmaf(v[e], v[e], ss);
      red1[cg * kRows + m] = ss;
    }
    group_sync(g);
    uint32_t words[2][P + 1];   // per column group: code planes, then the extra low bit (EXT columns)
    float nrm0 = 0.f;           // column group 2 wh's norm (the norm entry's writer uses it)
    if constexpr (POLAR) {
      float tot = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) tot += red1[k * kRows + m];
      nrm0 = sqrtf(tot);
      const float inv = nrm0 > 0.f ? 1.f / nrm0 : 0.f;
      float gs = 0.f;
      polar::epilogue<128, 2, B1, PROD>(tpol, tg + lane_off, t_rhi + lane_off, t_rlo + lane_off, 2 * wh, inv, red3, m,
                                        words, gs, [&] { group_sync(g); });
      red2[(2 * wh) * kRows + m] = gs;
      red2[(2 * wh + 1) * kRows + m] = 0.f;
    } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int cg = 2 * wh + h;
      float tot = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) tot += ((k < kx) == (cg < kx)) ? red1[k * kRows + m] : 0.f;
      const float nrm = sqrtf(tot);
      if (h == 0) nrm0 = nrm;
      const float inv = nrm > 0.f ? 1.f / nrm : 0.f;
      const bool ext = EXT && (32 * cg < cb.extra);   // the same for the whole warp
      uint32_t* word = words[h];
#pragma unroll
      for (int p = 0; p <= P; ++p) word[p] = 0u;
      float gs = 0.f;
      // the column group's 32 coordinates in two halves of 16 (fewer live
      // registers); XC: the extended (b' + 1)-bit codebook of extra-bit
      // columns.  The choice is made once per column group, outside the
      // element loops.
      auto column_group = [&](auto xc) {
        constexpr bool XC = decltype(xc)::value;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[16];
          tmem_ld16(tg + lane_off + 32 * cg + 16 * half, v);
          uint32_t rh[8], rl[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float r2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const float y = v[e + u] * inv;
              const int jb = 16 * half + e + u;       // bit of the column group's words
              float r;
              if constexpr (XC) {
                const int idx = cell_heap<B1 + 1>(y, ltx, s_bndx, word, jb);
                r = y - s_centx[idx];
              } else if constexpr (B1 <= 2) {
                r = y - cell_cent<B1>(y, lt, cr, word, jb);
              } else {
                const int idx = cell_heap<B1>(y, lt, s_bnd, word, jb);
                r = y - s_cent[idx];
              }
              gs = fmaf(r, r, gs);
              r2[u] = r;
            }
            // bf16 hi + lo pieces of the residual pair
            const uint32_t hb = bf16x2(r2[0], r2[1]);
            rh[e >> 1] = hb;
            rl[e >> 1] = bf16x2(r2[0] - __uint_as_float(hb << 16), r2[1] - __uint_as_float(hb & 0xFFFF0000u));
          }
          if (prod) {
            // A operand of the sketch in tensor memory: lane = row, column
            // 16 cg + i holds coordinates 32 cg + 2i (low half) and 2i + 1
            tmem_st8(t_rhi + lane_off + 16 * cg + 8 * half, rh);
            tmem_st8(t_rlo + lane_off + 16 * cg + 8 * half, rl);
          }
        }
      };
      if (EXT && ext)
        column_group(std::integral_constant<bool, EXT>{});
      else
        column_group(std::integral_constant<bool, false>{});
      red2[cg * kRows + m] = gs;
    }
    }
    if (prod) asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    fence_before();
    group_sync(g);
    // ---- QJL projection on the tensor cores: Z = R_hi S^T + R_lo S^T (into
    // the columns of Y, which every thread of the group has read)
    uint32_t sword[2] = {0u, 0u};
    float gam[2] = {0.f, 0.f};
    if (prod) {
      if (leader) {
        fence_after();
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16_ta(tg, t_rhi + 8 * ks, sw128_desc(sbase + kOffS + (ks >> 2) * kBlockBytes + 32 * (ks & 3)), kIdesc,
                      ks != 0);
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16_ta(tg, t_rlo + 8 * ks, sw128_desc(sbase + kOffS + (ks >> 2) * kBlockBytes + 32 * (ks & 3)), kIdesc,
                      1);
        mma_commit(bar_z);
      }
      pend_z = true;
      if (!group_and(g, mbar_wait(bar_z, j & 1))) {
        ok = false;
        break;
      }
      pend_z = false;
      fence_after();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int cg = 2 * wh + h;
        float v[32];
        tmem_ld32(tg + lane_off + 32 * cg, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) sword[h] |= (v[e] >= 0.f ? 1u : 0u) << e;
        float g2 = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) g2 += ((k < kx) == (cg < kx)) ? red2[k * kRows + m] : 0.f;
        gam[h] = sqrtf(g2);
      }
    }
    // ---- store
    const int64_t row = tile * kRows + m;
    const int64_t dst = row < n ? (dst_rows ? dst_rows[row] : row) : -1;
    if (row < n && (dst < 0 || dst >= cache_rows) && wh == 0) atomicOr(status, kBadRow);  // skipped
    if (dst >= 0 && dst < cache_rows) {
      uint32_t* rec = reinterpret_cast<uint32_t*>(cache) + dst * W;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int cg = 2 * wh + h;
        const bool ext = EXT && (32 * cg < cb.extra);
        const uint32_t xword = ext ? words[h][b1] : 0u;
        if constexpr (PROD) words[h][b1] = sword[h];
        if constexpr (P == 4 && !EXT) {
          *reinterpret_cast<uint4*>(rec + cg * P) = make_uint4(words[h][0], words[h][1], words[h][2], words[h][3]);
        } else if constexpr (P == 2 && !EXT) {
          *reinterpret_cast<uint2*>(rec + cg * P) = make_uint2(words[h][0], words[h][1]);
        } else {
#pragma unroll
          for (int p = 0; p < P; ++p) rec[cg * P + p] = words[h][p];
        }
        if (EXT && ext) rec[(128 / 32) * P + cg] = xword;
      }
      if (wh == 0) {
        uint8_t* norms = cache + norm_offset(cb, cache_rows);
        if (kx) {
          // group A's (column group 0) and group B's norms
          float t1 = 0.f, t2 = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (k >= kx) {
              t1 += red1[k * kRows + m];
              t2 += red2[k * kRows + m];
            }
          __half2* e = reinterpret_cast<__half2*>(norms) + 2 * dst;
          e[0] = __floats2half2_rn(nrm0, gam[0]);
          e[1] = __floats2half2_rn(sqrtf(t1), sqrtf(t2));
        } else if (prod) {
          reinterpret_cast<__half2*>(norms)[dst] = __floats2half2_rn(nrm0, gam[0]);
        } else {
          reinterpret_cast<__half*>(norms)[dst] = __float2half_rn(nrm0);
        }
      }
    }
    // every thread of the group has read Z (and its red entries) before the
    // group's next rotation overwrites them
    fence_before();
    group_sync(g);
  }
  if (!ok) {
    if (tid == 0) atomicOr(status, 1);
    // this group's own MMAs in flight finish (bounded waits)
    if (leader && pend_y) mbar_wait(bar_y, j & 1);
    if (leader && pend_z) mbar_wait(bar_z, j & 1);
  }
  // every load issued lands (bounded) before the shared memory is released
  fence_before();
  __syncthreads();
  if (tid == 0) {
    if (const_pending) mbar_wait(bar_const, 0);
    for (int st = 0; st < kStages; ++st)
      for (int k = n_taken[st]; k < n_issued[st]; ++k) mbar_wait(bar_full(st), (uint32_t)(k & 1));
  }
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

template <int B1, bool PROD, bool EXT, bool POLAR>
static cudaError_t launch_tc_t(const CUtensorMap& tm_x, const CUtensorMap& tm_pihi, const CUtensorMap& tm_pilo,
                               const CUtensorMap& tm_s, const Dev& cb, uint8_t* cache, int64_t cache_rows, int64_t n,
                               const int64_t* dst_rows, int* status, int sms, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_quantize_tc<B1, PROD, EXT, POLAR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t ntiles = (n + kRows - 1) / kRows;
  const int grid = (int)(ntiles < sms ? ntiles : sms);
  k_quantize_tc<B1, PROD, EXT, POLAR><<<grid, kThreads, kSmemBytes, s>>>(tm_x, tm_pihi, tm_pilo, tm_s, cb, cache,
                                                                         cache_rows, n, dst_rows, status);
  return cudaGetLastError();
}

cudaError_t launch_quantize_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_pihi, const CUtensorMap& tm_pilo,
                               const CUtensorMap& tm_s, const Dev& cb, uint8_t* cache, int64_t cache_rows, int64_t n,
                               const int64_t* dst_rows, int* status, int sms, cudaStream_t s) {
#define TQ_TC(B, PR, EX) \
  return launch_tc_t<B, PR, EX, false>(tm_x, tm_pihi, tm_pilo, tm_s, cb, cache, cache_rows, n, dst_rows, status, sms, s)
#define TQ_TCP(B, PR) \
  return launch_tc_t<B, PR, false, true>(tm_x, tm_pihi, tm_pilo, tm_s, cb, cache, cache_rows, n, dst_rows, status, sms, s)
  if (cb.mode != 0) {   // polar mode (no extra-bit words)
    if (cb.kind == 0) {
      switch (cb.b1) {
        case 1: TQ_TCP(1, true);
        case 2: TQ_TCP(2, true);
        default: TQ_TCP(3, true);
      }
    }
    switch (cb.b1) {
      case 1: TQ_TCP(1, false);
      case 2: TQ_TCP(2, false);
      case 3: TQ_TCP(3, false);
      default: TQ_TCP(4, false);
    }
  }
  const bool ext = cb.extra != 0;
  if (cb.kind == 0) {
    switch (cb.b1 * 2 + (ext ? 1 : 0)) {
      case 2: TQ_TC(1, true, false);
      case 3: TQ_TC(1, true, true);
      case 4: TQ_TC(2, true, false);
      case 5: TQ_TC(2, true, true);
      case 6: TQ_TC(3, true, false);
      default: TQ_TC(3, true, true);
    }
  }
  switch (cb.b1 * 2 + (ext ? 1 : 0)) {
    case 2: TQ_TC(1, false, false);
    case 3: TQ_TC(1, false, true);
    case 4: TQ_TC(2, false, false);
    case 5: TQ_TC(2, false, true);
    case 6: TQ_TC(3, false, false);
    case 7: TQ_TC(3, false, true);
    default: TQ_TC(4, false, false);
  }
#undef TQ_TCP
#undef TQ_TC
}

}  // namespace tq
