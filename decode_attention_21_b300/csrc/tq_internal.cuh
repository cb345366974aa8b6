// Internal definitions shared by the CUDA kernels and the C-ABI layer.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tq {

constexpr int kMaxL = 16;        // largest stage-1 cell count (4 bits)
constexpr int kMaxLevels = 9;    // polar levels for d <= 256

// Codebook as the kernels see it; passed by value as a kernel parameter.
struct Dev {
  int d, m, b1, kind, mode, extra;
  int P;            // stored planes per 32-coordinate word column
  int W;            // 32-bit words per record
  int nb;           // norm bytes per row (4 prod, 2 mse, 8 split)
  int nv;           // stage-1 virtual planes (odd subsets of the code planes)
  uint32_t vmask[kMaxL];  // plane p in subset <=> bit p set
  float vcoef[kMaxL];     // yhat = sum_v vcoef[v] * (-1)^(xor of the subset's bits)
  float cent[kMaxL], bound[kMaxL];
  float cent_x[2 * kMaxL], bound_x[2 * kMaxL];
  // extended (b' + 1)-bit codebook of the first `extra` coordinates: the
  // Walsh-Hadamard coefficients of cent_x over the odd subsets of its b' + 1
  // planes (plane b' = the extra bit), nvx = 2 nv of them
  int nvx;
  float vcoef_x[kMaxL];
  float qjl_const;        // sqrt(pi/2) / m (split: group B's, m = d - extra)
  // outlier-channel split: rotated coordinates 0..extra-1 are group A (the
  // extended codebook, own norms, QJL constant sqrt(pi/2) / extra)
  int split;
  float qjl_const_x;
  // polls of the first bounded wait of every launch (the others use the
  // full limit); lowered only by tq_set_first_wait_limit, for tests
  long long first_wait;
  // polar mode, per level l = 1..D (index l): boundary and centroid (cos, sin)
  float pb_cos[kMaxLevels][kMaxL], pb_sin[kMaxLevels][kMaxL];
  float pc_cos[kMaxLevels][kMaxL], pc_sin[kMaxLevels][kMaxL];
  // device tables
  const float* Pi;        // [d][d] row-major, y = Pi x
  const float* PiT;       // [d][d], PiT[j*d + i] = Pi[i][j]
  const float* ST;        // [d][m], ST[i*m + j] = S[j][i]
  const float* SPT;       // [d][m], SPT[i*m + j] = (S Pi)[j][i]: q'' = (S Pi) q in one pass
  const uint16_t* Pi_hi;  // bf16 split of Pi (row-major): Pi ~ hi + lo
  const uint16_t* Pi_lo;
  const uint16_t* S_bf;   // bf16 S (exact), row-major [m][d]
};

inline __host__ __device__ int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// One NVTX range per C-ABI call, named after the call (shows in profiler
// timelines; a few nanoseconds when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name);
  ~NvtxRange();
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// L2 residency hints.  The packed caches are streamed once per call
// (evict-first); the small codebook tables (Pi, S Pi, S) are read by every
// query prep and cache append and should stay in L2 (evict-last).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Read-only load of a table entry with an L2 cache policy.
__device__ __forceinline__ float ld_table(const float* p, uint64_t policy) {
  float v;
  asm volatile("ld.global.nc.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(policy));
  return v;
}

// Polar angle decisions.  "angle(ra, rb) >= t" is the exact sign of
// rb cos t - ra sin t >= 0 for fp32 inputs (a zero determinant goes to the
// upper cell).  The fp32 value v = fma(rb, c, -round(ra s)) is off the exact
// determinant by at most half an ulp of round(ra s) plus the rounding of v,
// so whenever |v| > max(2^-21 |round(ra s)|, 2^-100) its sign is the exact
// sign; otherwise (near-ties, tiny products) both products are formed exactly
// in fp64.  Valid for products below 2^127 in magnitude (unit rows).
// The fp64 products sit in a function of their own so that they run only on
// that rare branch (B300's fp64 rate is a small fraction of its fp32 rate).
static __device__ __noinline__ int ge_exact_f64(float rb, float ra, float c, float s) {
  return (double)rb * (double)c - (double)ra * (double)s >= 0.0 ? 1 : 0;
}
__device__ __forceinline__ int ge_exact(float rb, float ra, float c, float s) {
  const float ps = ra * s;
  const float v = fmaf(rb, c, -ps);
  if (__builtin_expect(fabsf(v) > fmaxf(fabsf(ps) * 0x1p-21f, 0x1p-100f), 1)) return v > 0.f ? 1 : 0;
  return ge_exact_f64(rb, ra, c, s);
}

// fp32 radius with separately rounded products, sum and square root.
__device__ __forceinline__ float radius_rn(float a, float b) {
  return __fsqrt_rn(__fadd_rn(__fmul_rn(a, a), __fmul_rn(b, b)));
}

// Byte offset of the norm region of a cache holding `rows` rows.
inline __host__ __device__ int64_t norm_offset(const Dev& cb, int64_t rows) {
  return align256(rows * cb.W * 4);
}

// Per-(sequence, kv head) block of query data prepared once per step.
//   header: float S1[4], S2[4], K1[4], K2[4], K1x[4], K2x[4], pad (per head
//           slot; K1x, K2x: the constants of a split's group A)
//   fragments: [2][d/16][32 lanes] uint2  (plane 0 = stage 1, plane 1 = QJL)
constexpr int kPrepHeader = 128;
inline __host__ __device__ int64_t prep_block_bytes(int d) { return kPrepHeader + (int64_t)2 * (d / 16) * 32 * 8; }

// Split-KV partial of one warp: per head slot (4): m, l, acc[d].
inline __host__ __device__ int64_t partial_floats(int d) { return 4 * (2 + d); }

constexpr int kAttnWarps = 4;     // warps per attention / logits CTA

// Where the cache row of token t of sequence b, kv head kvh lives.
//   contiguous (table == nullptr): row (b*Hkv + kvh)*capacity + t;
//   paged: block table entry table[b*max_pages + t/page] names a page that
//   holds `page` consecutive rows per kv head: row (entry*Hkv + kvh)*page + t%page.
// page is a multiple of 16, so a 16-token tile never straddles two pages.
struct RowMap {
  const int32_t* table;
  int32_t page;        // tokens per page
  int32_t max_pages;   // entries per table row (capacity = max_pages * page < 2^31)
  int32_t num_pages;   // pages in the cache; other entries are rejected
  int32_t page_shift;  // log2(page) for a power-of-two page, else -1
};

// Page index and offset within the page of token t.
__device__ __forceinline__ void split_token(const RowMap& m, uint32_t t, uint32_t& pi, uint32_t& off) {
  if (m.page_shift >= 0) {
    pi = t >> m.page_shift;
    off = t & (uint32_t)(m.page - 1);
  } else {
    pi = t / (uint32_t)m.page;
    off = t - pi * (uint32_t)m.page;
  }
}

// Destination rows of a cache append: rows 0..n-1, an explicit list, or for a
// paged cache the last token (seq_lens[b] - 1) of each (b, kvh) of a batch of
// B*Hkv rows in (b, kvh) order; sequences with seq_lens[b] <= 0 are skipped.
struct AppendDst {
  const int64_t* rows;      // explicit list, or nullptr
  RowMap map;               // paged when map.table != nullptr
  const int32_t* seq_lens;  // paged: lengths including the appended token
  int32_t Hkv;
};

// Status word bits set by the kernels (the codebook's device status word):
// low bits = a bounded wait gave up (1 quantize, 2 scoring); kBadRow = an
// append destination or a block-table entry lay outside the cache (the
// access was skipped, or for a scoring read redirected to page 0).
constexpr int kBadRow = 0x100;

// Destination row of append row `row`: >= 0, or -1 (skip: empty sequence),
// or -2 (skip: outside the cache).
__device__ __forceinline__ int64_t append_row(const AppendDst& a, int64_t row, int64_t cache_rows) {
  int64_t dst;
  if (a.map.table) {
    const int b = (int)(row / a.Hkv), kvh = (int)(row - (int64_t)b * a.Hkv);
    const int32_t t = a.seq_lens[b] - 1;
    if (t < 0) return -1;
    uint32_t pi, off;
    split_token(a.map, (uint32_t)t, pi, off);
    if (pi >= (uint32_t)a.map.max_pages) return -2;
    const int32_t pg = a.map.table[(int64_t)b * a.map.max_pages + pi];
    if (pg < 0 || pg >= a.map.num_pages) return -2;
    dst = ((int64_t)pg * a.Hkv + kvh) * a.map.page + off;
  } else {
    dst = a.rows ? a.rows[row] : row;
  }
  return (dst >= 0 && dst < cache_rows) ? dst : -2;
}

// Host-side launchers (one per kernel family); each returns the launch error.
cudaError_t launch_quantize_simt(const Dev& cb, uint8_t* cache, int64_t cache_rows, const void* x, int x_dtype,
                                 int64_t n, int d_in, const float* y, const float* norms, const AppendDst& dst,
                                 int* status, cudaStream_t s);
cudaError_t launch_advance_lengths(int32_t* seq_lens, int B, int32_t delta, cudaStream_t s);
cudaError_t launch_quantize_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_pihi, const CUtensorMap& tm_pilo,
                               const CUtensorMap& tm_s, const Dev& cb, uint8_t* cache, int64_t cache_rows, int64_t n,
                               const int64_t* dst_rows, int* status, int sms, cudaStream_t s);
cudaError_t launch_quantize_tcx(const CUtensorMap& tm_pihi, const CUtensorMap& tm_pilo, const CUtensorMap& tm_s,
                                const Dev& cb, uint8_t* cache, int64_t cache_rows, const void* x, bool f32, int64_t n,
                                int d_in, const int64_t* dst_rows, int* status, int sms, cudaStream_t s);
cudaError_t launch_prep(const Dev& cb, const float* q, int B, int Hq, int Hkv, uint8_t* prep, cudaStream_t s);
// The query prep with a decode step's key append (n rows of x into the
// cache at dst_rows; scalar mode, d = 128, no extra-bit words) in one grid.
cudaError_t launch_prep_append(const Dev& cb, const float* q, int B, int Hq, int Hkv, uint8_t* prep, uint8_t* cache,
                               int64_t cache_rows, const void* x, int x_dtype, int64_t n, int d_in,
                               const int64_t* dst_rows, int* status, cudaStream_t s);
cudaError_t launch_logits(const Dev& cb, const uint8_t* kcache, int B, int Hq, int Hkv, int64_t capacity,
                          int64_t cache_rows, const int32_t* seq_lens, const uint8_t* prep, float* logits,
                          int nchunks, int tiles_per_cta, cudaStream_t s);
cudaError_t launch_logits_staged(const Dev& cb, const uint8_t* kcache, int B, int Hq, int Hkv, int64_t capacity,
                                 int64_t cache_rows, const RowMap& map, const int32_t* seq_lens, const uint8_t* prep,
                                 float* logits, int nchunks, int tiles_per_cta, int* status, cudaStream_t s);
cudaError_t launch_attn(const Dev& kcb, const Dev& vcb, const uint8_t* kcache, const uint8_t* vcache, int B, int Hq,
                        int Hkv, int64_t capacity, int64_t cache_rows, const int32_t* seq_lens, const uint8_t* prep,
                        float scale_log2, float* partials, int nchunks, int tiles_per_cta, cudaStream_t s);
cudaError_t launch_attn_staged(const Dev& kcb, const Dev& vcb, const uint8_t* kcache, const uint8_t* vcache, int B,
                               int Hq, int Hkv, int64_t capacity, int64_t cache_rows, const RowMap& map,
                               const int32_t* seq_lens, const uint8_t* prep, float scale_log2, float* partials,
                               int nchunks, int tiles_per_cta, int* status, cudaStream_t s);
// Key / value codebook pairs the staged scalar attention kernel is built for.
bool attn_staged_supports(const Dev& kcb, const Dev& vcb);
cudaError_t launch_attn_polar_staged(const Dev& kcb, const Dev& vcb, const uint8_t* kcache, const uint8_t* vcache,
                                     int B, int Hq, int Hkv, int64_t capacity, int64_t cache_rows, const RowMap& map,
                                     const int32_t* seq_lens, const uint8_t* prep, float scale_log2, float* partials,
                                     int nchunks, int tiles_per_cta, int* status, cudaStream_t s);
cudaError_t launch_prep_polar(const Dev& cb, const float* q, int B, int Hq, int Hkv, uint8_t* prep, cudaStream_t s);
cudaError_t launch_logits_polar(const Dev& cb, const uint8_t* kcache, int B, int Hq, int Hkv, int64_t capacity,
                                int64_t cache_rows, const RowMap& map, const int32_t* seq_lens, const uint8_t* prep,
                                float* logits, int nchunks, int tiles_per_cta, int* status, cudaStream_t s);
cudaError_t launch_attn_polar(const Dev& kcb, const Dev& vcb, const uint8_t* kcache, const uint8_t* vcache, int B,
                              int Hq, int Hkv, int64_t capacity, int64_t cache_rows, const int32_t* seq_lens,
                              const uint8_t* prep, float scale_log2, float* partials, int nchunks, int tiles_per_cta,
                              cudaStream_t s);
int64_t search_workspace_bytes(const Dev& cb, int64_t n_db, int nq, int k, int sms);
cudaError_t launch_search(const Dev& cb, const uint8_t* db, int64_t n_db, const float* q, int nq, int d_in, int k,
                          int32_t* ids, float* scores, uint8_t* prep, int sms, cudaStream_t s);
cudaError_t launch_search_subset(const Dev& cb, const uint8_t* db, int64_t n_db, const float* q, int nq, int d_in,
                                 int k, int32_t* ids, float* scores, uint8_t* prep, int sms, const int32_t* qmap,
                                 const unsigned* qcount, cudaStream_t s);
// Tensor-core search (tcgen05 candidates + exact re-ranking), for d = 256
// scalar-mode databases without extra bits and k <= 16.  Its workspace starts
// with 64 status words; word 2 counts the queries sent to the exact scan.
bool search_tc_applies(const Dev& cb, int k);
int64_t search_tc_workspace_bytes(const Dev& cb, int64_t n_db, int nq, int k, int sms);
cudaError_t launch_search_tc(const Dev& cb, const uint8_t* db, int64_t n_db, const float* q, int nq, int d_in, int k,
                             int32_t* ids, float* scores, uint8_t* ws, int sms, int* status, cudaStream_t s);
// group_stride: floats between the partials of consecutive 4-head groups.
cudaError_t launch_attn_merge(const Dev& vcb, const float* partials, int B, int Hq, int Hkv, int nparts,
                              int64_t group_stride, float* out, cudaStream_t s);

}  // namespace tq
