// Device helpers of the tcgen05 kernels that compress token batches: TMA and
// bulk copies completed on mbarriers (bounded waits), tcgen05.mma with bf16
// operands (A from shared memory or from tensor memory), tensor-memory loads
// and stores, and the stage-1 cell search of the epilogues.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

namespace tq {
namespace tc {

constexpr long long kSpinLimit = 1ll << 26;

// kind::f16 instruction descriptor: D = F32, A = B = BF16, both K-major,
// M = 128, N = n (a multiple of 16 up to 256).
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Bounded wait for the phase with parity `parity` to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit = kSpinLimit) {
  for (long long i = 0; i < limit; ++i) {
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

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// A from tensor memory (lane = row, two bf16 per 32-bit column along K).
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// Named barrier of one 8-warp tile group (ids 1, 2; id 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int g) { asm volatile("bar.sync %0, 256;" ::"r"(1 + g) : "memory"); }

// The same barrier, returning whether v holds in every thread of the group.
__device__ __forceinline__ bool group_and(int g, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.and.pred q, %2, 256, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(1 + g)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Two fp32 values rounded to bf16 in one instruction: a in the low half.
__device__ __forceinline__ uint32_t bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// Stage-1 cell of y among the 2^L - 1 sorted boundaries b: bisection, each
// level one comparison y >= t (so the cell equals #{k : y >= b_k}); level l
// sets bit j of w[l] (most significant bit first).  lt holds the boundaries
// of the first levels in heap order (lt[0] = b[2^(L-1) - 1], then each
// level's candidates left to right).
template <int L>
__device__ __forceinline__ int cell_heap(float y, const float (&lt)[7], const float* s_bnd, uint32_t* w, int j) {
  if constexpr (L <= 2) {
    // one or two levels: the boundaries from registers
    const bool p0 = y >= lt[0];
    if (p0) w[0] |= 1u << j;
    if constexpr (L == 1) return p0 ? 1 : 0;
    const bool p1 = y >= (p0 ? lt[2] : lt[1]);
    if (p1) w[1] |= 1u << j;
    return (p0 ? 2 : 0) | (p1 ? 1 : 0);
  } else {
    // deeper tables: the first level from a register, the others from shared
    // memory (a register select tree was measured slower here)
    int idx = 0;
#pragma unroll
    for (int l = 0; l < L; ++l) {
      const int half = 1 << (L - 1 - l);
      const float t = l == 0 ? lt[0] : s_bnd[idx + half - 1];
      if (y >= t) {
        idx += half;
        w[l] |= 1u << j;
      }
    }
    return idx;
  }
}

// As cell_heap for L <= 2, returning the centroid of the cell from the
// registers cr[0 .. 2^L - 1] (selects instead of an index and a table load).
template <int L>
__device__ __forceinline__ float cell_cent(float y, const float (&lt)[7], const float (&cr)[4], uint32_t* w, int j) {
  static_assert(L <= 2, "register centroids for one or two levels");
  const bool p0 = y >= lt[0];
  if (p0) w[0] |= 1u << j;
  if constexpr (L == 1) {
    return p0 ? cr[1] : cr[0];
  } else {
    const bool p1 = y >= (p0 ? lt[2] : lt[1]);
    if (p1) w[1] |= 1u << j;
    const float lo = p1 ? cr[1] : cr[0], hi = p1 ? cr[3] : cr[2];
    return p0 ? hi : lo;
  }
}

// Heap-ordered boundaries of the first three bisection levels of a 2^L-cell
// table (node n at level l, position k: boundary (2k + 1) 2^(L-1-l) - 1).
template <int L>
__device__ __forceinline__ void heap_levels(const float* bnd, float (&lt)[7]) {
#pragma unroll
  for (int nd = 0; nd < 7; ++nd) {
    const int l = nd == 0 ? 0 : nd < 3 ? 1 : 2, k = nd - ((1 << l) - 1);
    lt[nd] = l < L ? bnd[(2 * k + 1) * (1 << (L - 1 - l)) - 1] : 0.f;
  }
}

}  // namespace tc
}  // namespace tq
