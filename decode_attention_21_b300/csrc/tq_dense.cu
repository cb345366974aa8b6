// Unquantized attention logits: the comparator that the pages' speed-up of
// 4-bit TurboQuant keys is quoted against ([xujun] 常见问题: the 8x figure is
// attention logits against 32-bit unquantized keys on H100).  Plain dot
// products of the G query heads of a kv head with fp32 or bf16 keys, on the
// tensor cores for bf16 keys (bf16 mma.sync m16n8k16, fp32 accumulation) and
// on the FMA pipe for fp32 keys; one pass over the keys, HBM-bound by design.
//
// Tile = 16 keys; thread (g, c) of a warp supplies keys g and g+8 and, of
// each row, the 16-byte chunks c, c+4, c+8, c+12 (so the four threads of a
// row read 64 contiguous bytes per load).  Word w = 4i + j of that slice
// (chunk c + 4i, pair j) holds dimensions dim(w) = 8c + 32i + 2j, +1.  MMA
// k-index 16 kb + 2c + (0, 1) takes word 2kb and 16 kb + 2c + 8 + (0, 1)
// word 2kb + 1; the query side (B) follows the same map.  B columns: 4 heads
// x (bf16 hi, lo) of q.
#include <cuda_bf16.h>

#include <algorithm>

#include "tq.h"
#include "tq_internal.cuh"

namespace tq {

namespace {

constexpr int kD = 128;

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint4 ld_stream16(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// This thread's 32 bf16 elements of one key row as 16 words (bf16 pairs).
struct Slice {
  uint32_t w[16];
  __device__ __forceinline__ void load(const uint8_t* row, int c, uint64_t pol, bool valid) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = valid ? ld_stream16(row + 16 * (c + 4 * i), pol) : make_uint4(0, 0, 0, 0);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  }
};

}  // namespace

// Tensor-core variant (used for bf16 keys, whose words are the operands as
// stored).  Grid (chunks, Hkv, B), 128 threads; each warp scores 16-key
// tiles warp, warp + 4, ... of its CTA's chunk, two tiles in flight.
__global__ void __launch_bounds__(128) k_logits_dense_tc(const uint8_t* __restrict__ keys, int Hq, int Hkv,
                                                      int64_t capacity, const int32_t* __restrict__ seq_lens,
                                                      const float* __restrict__ q, float* __restrict__ logits,
                                                      int64_t tiles_per_cta) {
  constexpr int EB = 2;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int G = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t L = seq_lens[b];
  const int64_t ntiles = (L + 15) / 16;
  const int64_t t0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t t1 = min(t0 + tiles_per_cta, ntiles);
  if (t0 >= t1) return;
  // B fragments: column g = head g/2, piece g%2 (bf16 hi, lo of q)
  uint32_t bq[8][2];
  {
    const int h = g >> 1, pc = g & 1;
    const float* qh = q + ((size_t)b * Hq + (size_t)kvh * G + h) * kD;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int w = 2 * kb + r, dim = 8 * c + 32 * (w >> 2) + 2 * (w & 3);
        float v0 = 0.f, v1 = 0.f;
        if (h < G) {
          v0 = qh[dim];
          v1 = qh[dim + 1];
        }
        const uint32_t hi = pack_bf16(v0, v1);
        if (pc == 0) {
          bq[kb][r] = hi;
        } else {
          const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
          bq[kb][r] = pack_bf16(v0 - h0, v1 - h1);
        }
      }
  }
  const uint8_t* base = keys + ((size_t)b * Hkv + kvh) * capacity * (kD * EB);
  float* out = logits + ((size_t)b * Hq + (size_t)kvh * G + c) * capacity;
  const uint64_t pol = l2_policy_evict_first();
  for (int64_t tile = t0 + warp; tile < t1; tile += 8) {
    const int64_t tile2 = tile + 4;
    const bool two = tile2 < t1;
    Slice ka, kb8, kc, kd8;
    const int64_t ta = tile * 16 + g, tc = tile2 * 16 + g;
    ka.load(base + (size_t)ta * (kD * EB), c, pol, ta < L);
    kb8.load(base + (size_t)(ta + 8) * (kD * EB), c, pol, ta + 8 < L);
    kc.load(base + (size_t)tc * (kD * EB), c, pol, two && tc < L);
    kd8.load(base + (size_t)(tc + 8) * (kD * EB), c, pol, two && tc + 8 < L);
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      mma_bf16(acc[0], ka.w[2 * kb], kb8.w[2 * kb], ka.w[2 * kb + 1], kb8.w[2 * kb + 1], bq[kb][0], bq[kb][1]);
      mma_bf16(acc[1], kc.w[2 * kb], kd8.w[2 * kb], kc.w[2 * kb + 1], kd8.w[2 * kb + 1], bq[kb][0], bq[kb][1]);
    }
    if (c < G) {
      if (ta < L) out[ta] = acc[0][0] + acc[0][1];
      if (ta + 8 < L) out[ta + 8] = acc[0][2] + acc[0][3];
      if (two && tc < L) out[tc] = acc[1][0] + acc[1][1];
      if (two && tc + 8 < L) out[tc + 8] = acc[1][2] + acc[1][3];
    }
  }
}


// SIMT variant (used for fp32 keys, where splitting every element into bf16
// hi + lo for the tensor cores costs more than the dot products): one warp
// scores two keys per step; lane l holds elements 8 (l % 16) .. +7 of key
// 2s + l / 16 and the matching slices of the G query heads; each partial dot
// is reduced over the 16 lanes of its half-warp.  Four key pairs in flight.
constexpr int kPairsInFlight = 4;

__global__ void __launch_bounds__(256) k_logits_dense_simt(const uint8_t* __restrict__ keys, int Hq, int Hkv,
                                                           int64_t capacity, const int32_t* __restrict__ seq_lens,
                                                           const float* __restrict__ q, float* __restrict__ logits,
                                                           int64_t pairs_per_cta) {
  constexpr int EB = 4;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int G = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, part = lane & 15;
  const int64_t L = seq_lens[b];
  const int64_t npairs = (L + 1) / 2;
  const int64_t p0 = (int64_t)blockIdx.x * pairs_per_cta;
  const int64_t p1 = min(p0 + pairs_per_cta, npairs);
  if (p0 >= p1) return;
  float qs[4][8];
#pragma unroll
  for (int h = 0; h < 4; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) qs[h][i] = h < G ? q[((size_t)b * Hq + kvh * G + h) * kD + 8 * part + i] : 0.f;
  const uint8_t* base = keys + ((size_t)b * Hkv + kvh) * capacity * (kD * EB);
  float* out = logits + ((size_t)b * Hq + (size_t)kvh * G) * capacity;
  const uint64_t pol = l2_policy_evict_first();
  for (int64_t p = p0 + warp; p < p1; p += 8 * kPairsInFlight) {
    float x[kPairsInFlight][8];
    int64_t t[kPairsInFlight];
#pragma unroll
    for (int k = 0; k < kPairsInFlight; ++k) {
      t[k] = 2 * (p + 8 * k) + half;
      if (p + 8 * k < p1 && t[k] < L) {
        const uint8_t* row = base + (size_t)t[k] * (kD * EB) + part * 32;
        const uint4 a = ld_stream16(row, pol), c2 = ld_stream16(row + 16, pol);
        x[k][0] = __uint_as_float(a.x); x[k][1] = __uint_as_float(a.y);
        x[k][2] = __uint_as_float(a.z); x[k][3] = __uint_as_float(a.w);
        x[k][4] = __uint_as_float(c2.x); x[k][5] = __uint_as_float(c2.y);
        x[k][6] = __uint_as_float(c2.z); x[k][7] = __uint_as_float(c2.w);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[k][i] = 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < kPairsInFlight; ++k) {
      float sdot[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaf(qs[h][i], x[k][i], a);
        sdot[h] = a;
      }
#pragma unroll
      for (int o = 8; o; o >>= 1)
#pragma unroll
        for (int h = 0; h < 4; ++h) sdot[h] += __shfl_xor_sync(0xffffffffu, sdot[h], o);
      if (part < G && p + 8 * k < p1 && t[k] < L) {
        const float v = part == 0 ? sdot[0] : part == 1 ? sdot[1] : part == 2 ? sdot[2] : sdot[3];
        out[(size_t)part * capacity + t[k]] = v;
      }
    }
  }
}

// Resident CTAs of a kernel on this device (one wave of its grid).
int resident_ctas(const void* fn, int threads) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, 0);
  return std::max(1, sms) * std::max(1, per_sm);
}

}  // namespace tq

namespace tq {
tq_status report_error(tq_status st, const char* msg);
}

extern "C" tq_status tq_logits_dense(const void* keys, int32_t key_dtype, int32_t d, int32_t B, int32_t Hq,
                                     int32_t Hkv, int64_t capacity, const int32_t* seq_lens, const float* q,
                                     float* logits, void* stream) {
  const tq::NvtxRange nvtx_range("tq_logits_dense");
  if (key_dtype != TQ_F32 && key_dtype != TQ_BF16)
    return tq::report_error(TQ_EINVAL, "tq_logits_dense: key_dtype must be TQ_F32 or TQ_BF16");
  if (d != 128) return tq::report_error(TQ_EUNSUPPORTED, "tq_logits_dense: only d = 128 is implemented");
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || capacity < 0 || Hq % Hkv || B > 65535 || Hkv > 65535)
    return tq::report_error(TQ_EINVAL, "tq_logits_dense: bad sizes");
  if (Hq / Hkv > 4) return tq::report_error(TQ_EUNSUPPORTED, "tq_logits_dense: GQA groups larger than 4");
  if (capacity == 0) return TQ_OK;
  if (!keys || !seq_lens || !q || !logits) return tq::report_error(TQ_EINVAL, "tq_logits_dense: NULL device pointer");
  if ((reinterpret_cast<uintptr_t>(keys) | reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(logits)) & 15)
    return tq::report_error(TQ_EINVAL, "tq_logits_dense: device pointers must be 16-byte aligned");
  // chunks sized so that the grid is one wave of resident CTAs
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t units = (int64_t)B * Hkv;
  if (key_dtype == TQ_BF16) {
    static const int ctas = tq::resident_ctas(reinterpret_cast<const void*>(tq::k_logits_dense_tc), 128);
    const int64_t tiles = (capacity + 15) / 16;
    const int64_t want = std::max<int64_t>(1, ctas / units);
    const int64_t tpc = std::max<int64_t>(4, (tiles + want - 1) / want);
    const dim3 grid((unsigned)((tiles + tpc - 1) / tpc), (unsigned)Hkv, (unsigned)B);
    tq::k_logits_dense_tc<<<grid, 128, 0, s>>>(static_cast<const uint8_t*>(keys), Hq, Hkv, capacity,
                                                        seq_lens, q, logits, tpc);
  } else {
    static const int ctas = tq::resident_ctas(reinterpret_cast<const void*>(tq::k_logits_dense_simt), 256);
    const int64_t pairs = (capacity + 1) / 2;
    const int64_t want = std::max<int64_t>(1, ctas / units);
    const int64_t ppc = std::max<int64_t>(32, (pairs + want - 1) / want);
    const dim3 grid((unsigned)((pairs + ppc - 1) / ppc), (unsigned)Hkv, (unsigned)B);
    tq::k_logits_dense_simt<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(keys), Hq, Hkv, capacity, seq_lens, q,
                                                 logits, ppc);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return tq::report_error(TQ_ECUDA, cudaGetErrorString(e));
  return TQ_OK;
}
