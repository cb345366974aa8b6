// Bulk-copy staging shared by the scoring kernels: cp.async.bulk copies of
// cache bytes into shared memory, completed on mbarriers, waited on with
// bounded spins, and L2 prefetches.
#pragma once
#include <cstdint>

#include "tq_internal.cuh"

namespace tq {
namespace stage {
constexpr int kStageTiles = 8;
constexpr int kRing = 4;
constexpr int kPrefetchStages = 1;    // stages per CTA prefetched into L2 before the prep completes
constexpr long long kWaitLimit = 1ll << 26;

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// Bulk copy of streamed cache bytes (L2 evict-first: read once per call).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(l2_policy_evict_first())
      : "memory");
}

// Prefetch into L2 (no shared-memory copy): safe before the wait for the
// cache's writer, since L2 is where the writer's stores land; the bulk copies
// after the wait then hit L2 instead of HBM.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Run r (r = 0, 1, ..) of the tokens t0 .. t0 + n - 1 of (b, kvh) in a paged
// cache, i.e. the part of them in their (r+1)-th page: false if there is no
// such run; else its first token k (relative to t0), its token count and its
// first cache row.  Runs are independent, so the lanes of a warp can each
// look up and copy one.
__device__ __forceinline__ bool page_run(const RowMap& map, int b, int kvh, int Hkv, int64_t t0, int n, int r,
                                         int* status, int& k, int& cnt, int64_t& row) {
  uint32_t p0, o0;
  split_token(map, (uint32_t)t0, p0, o0);
  const int first = min(n, map.page - (int)o0);
  k = r == 0 ? 0 : first + (r - 1) * map.page;
  if (k >= n) return false;
  cnt = r == 0 ? first : min(n - k, map.page);
  int32_t pg = __ldg(map.table + (int64_t)b * map.max_pages + p0 + r);
  if (pg < 0 || pg >= map.num_pages) {
    atomicOr(status, kBadRow);
    pg = 0;
  }
  row = ((int64_t)pg * Hkv + kvh) * map.page + (r == 0 ? o0 : 0);
  return true;
}

// First cache row of the 16-token tile starting at token t0 of (b, kvh):
// contiguous, or through the block table (an entry outside the cache sets
// kBadRow in *status and yields page 0's row).
__device__ __forceinline__ int64_t tile_row(const RowMap& map, int b, int kvh, int Hkv, int64_t capacity, int64_t t0,
                                            int* status) {
  if (!map.table) return ((int64_t)b * Hkv + kvh) * capacity + t0;
  uint32_t pi, off;
  split_token(map, (uint32_t)t0, pi, off);
  int32_t pg = __ldg(map.table + (int64_t)b * map.max_pages + pi);
  if (pg < 0 || pg >= map.num_pages) {
    atomicOr(status, kBadRow);
    pg = 0;
  }
  return ((int64_t)pg * Hkv + kvh) * map.page + off;
}

__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, long long limit = kWaitLimit) {
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
}  // namespace stage
}  // namespace tq
