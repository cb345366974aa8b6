/*
 * tq.h -- C ABI of the TurboQuant hot path on one NVIDIA B300 (sm_103a).
 *
 * TurboQuant compresses key/value-cache and search-database vectors online and
 * without data: a seeded random rotation Pi, a per-coordinate Lloyd-Max code
 * at b-1 bits (or a recursive-polar code), and a 1-bit QJL sign sketch of the
 * residual with its norm; compressed keys are scored against full-precision
 * queries with an unbiased inner-product estimator.  Sources (web pages on
 * Google Research's TurboQuant, arXiv 2504.19874):
 *   [xujun]  xujun.org note-189244, sections "第一步：PolarQuant",
 *            "第二步：QJL", "性能数据";
 *   [suzuke] suzuke.github.io "TurboQuant: compressing AI consciousness",
 *            section "技術上怎麼做到的" (第一步, 第二步, 第三步);
 *   [cnyes]  hao.cnyes.com "TurboQuant", sections "極坐標的妙用", "1 bit 掃尾".
 *
 * Conventions for every entry point below
 *   - Pointers marked "device" are CUDA device pointers on the current device;
 *     "host" pointers are ordinary CPU memory.  The caller owns all of them.
 *   - ``stream`` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Hot calls only enqueue work on it: they never allocate memory
 *     and never synchronise.
 *   - Arguments are validated on the host before any launch; a bad argument
 *     returns TQ_EINVAL (or TQ_EUNSUPPORTED for a valid but unimplemented
 *     shape) and enqueues nothing.  A failed launch returns TQ_ECUDA.
 *     Errors of work already enqueued surface on a later call or sync.
 *     tq_last_error() gives a message for the calling thread.
 *   - All device buffers must be 16-byte aligned.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_EINVAL = 1,        /* invalid argument                                  */
  TQ_ENOMEM = 2,        /* codebook allocation failed / workspace too small  */
  TQ_ECUDA = 3,         /* a CUDA runtime call or launch failed              */
  TQ_ETIMEOUT = 4,      /* a bounded device-side wait gave up                */
  TQ_EUNSUPPORTED = 5   /* valid request outside the implemented shapes     */
} tq_status;

typedef enum { TQ_MODE_SCALAR = 0, TQ_MODE_POLAR = 1 } tq_mode;

/* PROD: (b-1)-bit stage 1 + 1-bit QJL sketch; keys and database rows.
 * MSE:  b-bit stage 1 only; values.                                          */
typedef enum { TQ_KIND_PROD = 0, TQ_KIND_MSE = 1 } tq_kind;

typedef enum { TQ_F32 = 0, TQ_BF16 = 1 } tq_dtype;

/* Everything the method fixes before the first vector arrives.
 * [suzuke] 第一步 (seeded orthogonal rotation), 第二步 (Max-Lloyd codes at
 * b-1 bits), 第三步 (1-bit QJL); [xujun] 第一步 (Beta law after rotation).   */
typedef struct {
  int32_t d;          /* vector dimension after padding: 128 or 256          */
  int32_t bits;       /* total bits per coordinate: PROD 2..4, MSE 1..4       */
  int32_t m;          /* QJL sketch rows; must equal d (ignored for MSE)      */
  int32_t mode;       /* tq_mode                                             */
  int32_t kind;       /* tq_kind                                             */
  int32_t extra;      /* scalar mode: the first `extra` rotated coordinates
                         get one more stage-1 bit; 0, d/4 or d/2             */
  uint64_t seed_pi;   /* splitmix64 stream of the Gaussian matrix behind Pi  */
  uint64_t seed_s;    /* splitmix64 stream of S                               */
  const double* pi;   /* host, optional: d*d row-major Pi overriding seed_pi */
  const float* s;     /* host, optional: m*d row-major S (bf16-exact values)
                         overriding seed_s                                   */
  const int32_t* outliers;  /* host, optional: `extra` distinct input channels
                         (0 .. d-1) forming an outlier group.  Non-NULL
                         selects the outlier-channel split (below).          */
} tq_codebook_desc;

/* Outlier-channel split ([xujun] 社区验证 and [suzuke] 實際跑出來的數據
 * quote 2.5- and 3.5-bit caches; the pages do not say how a fractional width
 * arises, and this is the reading implemented): the outlier channels (group
 * A, E = `extra` of them) and the other d - E channels (group B) are each
 * compressed as their own vector by their own instance of the method, group
 * A with one more bit per coordinate:
 *   - own rotation: Pi_A (E x E, Haar, seed_pi), Pi_B ((d-E) x (d-E),
 *     seed_pi + 1); the codebook's Pi (tq_codebook_tables) is the d x d map
 *     x -> (Pi_A x_A, Pi_B x_B), so rotated coordinates 0..E-1 are group A's
 *     (in the order listed) and the rest group B's (channel order);
 *   - own Lloyd-Max tables on the law of a rotated coordinate of an E- and a
 *     (d-E)-dimensional unit vector (B: b' bits, A: b'+1 bits);
 *   - own sketch: S = diag(S_A, S_B) (seed_s, seed_s + 1; m_g = d_g rows)
 *     and own QJL constant sqrt(pi/2)/d_g;
 *   - own norms: the norm entry is four fp16 values n_A, gamma_A, n_B,
 *     gamma_B (8 bytes);
 *   - the estimate of <q, x> is the sum of the two groups' estimates.
 * The record is the mixed-bit record (E extended coordinates).  Supported:
 * d = 128, scalar mode, PROD keys, extra = 32 or 64, bits 2..4; pi and s
 * overrides must be NULL.  Bits per coordinate: (E (b+1) + (d-E) b)/d codes
 * + 0.5 for the norms (b = 2: 2.75 at E = 32, 3.0 at E = 64).               */

typedef struct tq_codebook tq_codebook;   /* opaque; immutable once built */

/* Solve the Lloyd-Max tables on the rotated-coordinate law (Beta_d, or the
 * polar angle laws), draw Pi (Householder QR of a seeded Gaussian matrix,
 * positive-diagonal R) and S (Gaussian rounded to fp32 then bf16), and upload
 * them to the current device.  Setup only: allocates device memory and
 * synchronises.  *out receives the codebook; free it with tq_free_codebook.
 * Errors: TQ_EINVAL (bad field), TQ_ENOMEM, TQ_ECUDA.                       */
tq_status tq_make_codebook(const tq_codebook_desc* desc, tq_codebook** out);
void tq_free_codebook(tq_codebook* cb);

/* Host copies of the fp32 tables the kernels use, for inspection and tests.
 * centroids: 2^b' floats, boundaries: 2^b' - 1 floats (b' = stage-1 bits;
 * scalar mode; polar mode returns the level-2 angle tables).  pi: d*d fp64
 * row-major, s: m*d fp32 (PROD only).  Any output pointer may be NULL.       */
tq_status tq_codebook_tables(const tq_codebook* cb, float* centroids, float* boundaries,
                             double* pi, float* s);

/* Host-only: the tables tq_make_codebook would build for `desc`, computed on
 * the CPU without touching a device (for inspection and cross-checks).
 * Scalar mode: centroids 2^b' floats and boundaries 2^b' - 1 floats of the
 * stage-1 quantizer (level is ignored).  Polar mode: the angle quantizer of
 * tree level `level` (1 = first pairing of coordinates, up to log2 d).
 * pi: d*d fp64 row-major; s: m*d fp32 (PROD).  Outputs may be NULL.
 * Errors: TQ_EINVAL for a bad descriptor or level.                          */
tq_status tq_host_tables(const tq_codebook_desc* desc, int32_t level, float* centroids, float* boundaries,
                         double* pi, float* s);

/* Bytes of one packed row record (code planes + sign plane + extra words). */
size_t tq_record_bytes(const tq_codebook* cb);

/* Bytes of a cache holding `rows` rows: the records, padding to 256 bytes,
 * then one norm entry per row (PROD: fp16 ||x|| and fp16 ||r||; MSE: fp16
 * ||x||; outlier-channel split: fp16 n_A, gamma_A, n_B, gamma_B).  Record layout: word (c, p) at word offset c*P + p (P planes, plane
 * 0 = most significant stage-1 bit, last plane of PROD = QJL signs), bit j of
 * word c <-> coordinate 32c + j.                                             */
size_t tq_cache_bytes(const tq_codebook* cb, int64_t rows);

/* Append / overwrite rows of a packed cache (online per-token compression:
 * [suzuke] 為什麼這個方法特別聰明, no calibration, no offline pass).
 *   cache      device, tq_cache_bytes(cb, cache_rows) bytes
 *   x          device, n x d_in row-major, dtype TQ_F32 or TQ_BF16; d_in <= d
 *              and columns d_in..d-1 are taken as zero
 *   dst_rows   device int64[n] target rows (distinct), or NULL for rows
 *              0..n-1; a row outside 0..cache_rows-1 is skipped and flagged
 *              for tq_check_device (TQ_EINVAL)
 * Each row: n = ||x||, y = Pi x / n, stage-1 codes, r = y - yhat, gamma =
 * ||r||, sign(S r); n and gamma stored as fp16 (round to nearest even).    */
tq_status tq_quantize(const tq_codebook* cb, void* cache, int64_t cache_rows,
                      const void* x, int32_t x_dtype, int64_t n, int32_t d_in,
                      const int64_t* dst_rows, void* stream);

/* As tq_quantize but from already rotated unit rows: y device fp32 [n, d],
 * norms device fp32 [n] (stored as ||x||).  For an outlier-channel split
 * codebook, y holds each group's unit vector (group A in columns 0..E-1) and
 * norms is fp32 [n, 2] (n_A, n_B).  The stage-1 codes depend only on
 * fp32 comparisons of y, so they are reproducible bit for bit.              */
tq_status tq_quantize_rotated(const tq_codebook* cb, void* cache, int64_t cache_rows,
                              const float* y, const float* norms, int64_t n,
                              const int64_t* dst_rows, void* stream);

/* Workspace bytes tq_logits / tq_decode_attention need for B sequences and Hq
 * query heads (per-step query rotation and sketch, plus split partials).    */
size_t tq_logits_workspace(const tq_codebook* kcb, int32_t B, int32_t Hq, int32_t Hkv);

/* Attention logits of full-precision queries against compressed keys
 * ([cnyes] 1 bit 掃尾; [xujun] 第二步 unbiased estimator):
 *   logits[b, h, t] = n_t ( <Pi q, yhat_t> + gamma_t sqrt(pi/2)/m <S Pi q, sigma_t> )
 * for t < seq_lens[b]; entries t >= seq_lens[b] are left untouched.
 *   kcache     device, rows (b*Hkv + kvh)*capacity + t, PROD kind
 *   seq_lens   device int32[B], each <= capacity
 *   q          device fp32 [B, Hq, d] (Hq = G*Hkv with G = 1..4, 8, 12 or
 *              16; head h uses kv head h / G; groups above 4 are scored four
 *              heads per launch)
 *   logits     device fp32 [B, Hq, capacity]
 *   workspace  device, >= tq_logits_workspace(kcb, B, Hq, Hkv) bytes        */
tq_status tq_logits(const tq_codebook* kcb, const void* kcache, int32_t B, int32_t Hq,
                    int32_t Hkv, int64_t capacity, const int32_t* seq_lens, const float* q,
                    float* logits, void* workspace, size_t ws_bytes, void* stream);

/* One decode step of the logits path: the step's new keys are compressed
 * into the cache, then every key is scored ([suzuke] 為什麼這個方法特別聰明:
 * each token is compressed online as it arrives; [cnyes] 1 bit 掃尾: the
 * query is rotated and sketched once per step).  Equivalent to
 *   tq_quantize(kcb, kcache, B*Hkv*capacity, x, x_dtype, n, d_in, dst_rows)
 *   tq_logits(kcb, kcache, B, Hq, Hkv, capacity, seq_lens, q, logits, ...)
 * on the same stream, with bit-identical cache bytes and logits (seq_lens
 * must already count the appended keys).  For scalar-mode codebooks with
 * d = 128, no extra-bit words and 1 <= n <= 4096 the append runs inside the
 * query-prep launch, which takes one kernel hand-off off the step; other
 * codebooks, and n = 0, run the two calls as such.
 *   kcache     device, rows (b*Hkv + kvh)*capacity + t (as tq_logits)
 *   x          device, n x d_in row-major, TQ_F32 or TQ_BF16 (as tq_quantize)
 *   dst_rows   device int64[n] target rows of kcache, or NULL for 0..n-1; a
 *              row outside the cache is skipped and flagged (TQ_EINVAL at
 *              tq_check_device)
 * Other arguments and errors as tq_quantize and tq_logits.                  */
tq_status tq_append_logits(const tq_codebook* kcb, void* kcache, const void* x, int32_t x_dtype,
                           int64_t n, int32_t d_in, const int64_t* dst_rows, int32_t B,
                           int32_t Hq, int32_t Hkv, int64_t capacity, const int32_t* seq_lens,
                           const float* q, float* logits, void* workspace, size_t ws_bytes,
                           void* stream);

/* Unquantized comparator of tq_logits: the same logits from uncompressed
 * keys ([xujun] 常见问题: TurboQuant's attention-logit speed-up is quoted
 * against 32-bit unquantized keys):
 *   logits[b, h, t] = <q[b, h], keys[b, h / G, t]>   for t < seq_lens[b];
 * entries t >= seq_lens[b] are left untouched.
 *   keys       device [B, Hkv, capacity, d], fp32 or bf16 (key_dtype TQ_F32 /
 *              TQ_BF16), row-major
 *   d          128 (TQ_EUNSUPPORTED otherwise)
 *   seq_lens   device int32[B], each <= capacity
 *   q          device fp32 [B, Hq, d] (G = Hq / Hkv <= 4)
 *   logits     device fp32 [B, Hq, capacity]
 * fp32 accumulation; no workspace.                                          */
tq_status tq_logits_dense(const void* keys, int32_t key_dtype, int32_t d, int32_t B, int32_t Hq,
                          int32_t Hkv, int64_t capacity, const int32_t* seq_lens, const float* q,
                          float* logits, void* stream);

/* Workspace bytes of tq_decode_attention (the query prep, and split-KV
 * partials per 4-head group of each kv head). */
size_t tq_decode_attention_workspace(const tq_codebook* kcb, int32_t B, int32_t Hq,
                                     int32_t Hkv, int64_t capacity);

/* Fused decode attention over compressed keys and values (MSE kind).
 * [xujun] 常见问题: the attention step over the compressed cache is where the
 * quoted speed-up over unquantized keys comes from (not end to end);
 * [suzuke] 為什麼這個方法特別聰明: keys and values are compressed online, one
 * token at a time, so each decode step attends over the compressed cache as
 * it stands; [cnyes] 1 bit 掃尾: the logits inside are the estimator of
 * tq_logits (full-precision query, compressed keys).
 *   s_t = scale * logits[b, h, t], p = softmax over t < seq_lens[b],
 *   out[b, h] = Pi_v^T sum_t p_t n_v,t yhat_v,t
 * (weighted sum in the rotated domain, rotated back once per head; fp32
 * throughout).  seq_lens[b] == 0 gives a zero row.  Split-KV partials live
 * in the caller's workspace and are merged by a second kernel.
 * Key / value pairs: keys with the QJL term (PROD) at any width with values
 * at 1-4 bits, in scalar or polar mode; in scalar mode and with a capacity
 * that is a multiple of 16 also MSE-only keys or 2.5 / 3.5-bit keys (extra
 * bits) with 3- or 4-bit values, and 2.5 / 3.5-bit values (extra = d/4, 2 or
 * 3 bits) with keys that have the QJL term.  Other pairs: TQ_EUNSUPPORTED.
 * Heads as for tq_logits (G = 1..4, 8, 12 or 16).                          */
tq_status tq_decode_attention(const tq_codebook* kcb, const tq_codebook* vcb,
                              const void* kcache, const void* vcache, int32_t B, int32_t Hq,
                              int32_t Hkv, int64_t capacity, const int32_t* seq_lens,
                              const float* q, float scale, float* out, void* workspace,
                              size_t ws_bytes, void* stream);

/* tq_decode_attention without a workspace argument, for callers that cannot
 * allocate device memory for this library (a plugin whose host framework owns
 * all device memory, or a loop that must not call cudaMalloc).  The pages
 * have no counterpart to this entry point.  Scratch comes from one 4 MiB
 * array built into the library (reserved on every GPU that loads it, until
 * exit); a call that would need more returns TQ_EINVAL with a message and
 * launches nothing.  Arguments and results are those of tq_decode_attention.
 * All calls share the array and it keeps the last call's contents (each call
 * writes every byte it later reads, so nothing needs clearing); calls that
 * overlap on the GPU race on it and must be serialised.  The first call on
 * each device looks up the array's device address (cudaGetSymbolAddress with
 * that device current); make that first call before any stream capture.
 * This entry point itself allocates no memory.                              */
tq_status tq_decode_attention_static(const tq_codebook* kcb, const tq_codebook* vcb,
                                     const void* kcache, const void* vcache, int32_t B, int32_t Hq,
                                     int32_t Hkv, int64_t capacity, const int32_t* seq_lens,
                                     const float* q, float scale, float* out, void* stream);

/* ---- Paged caches and the in-place decode loop --------------------------
 * The per-token, calibration-free use of the method ([suzuke] 為什麼這個方法
 * 特別聰明: each new key or value is compressed the moment it arrives) fills
 * a cache one token per step.  The pages fix no memory layout for this; the
 * entry points below add the usual one, a pool of fixed-size pages named by a
 * per-sequence block table, so sequences grow without reserving their full
 * capacity.  The arithmetic is that of the contiguous entry points, bit for
 * bit: a paged call returns exactly what the contiguous call returns on a
 * cache holding the same rows.
 *
 * Paged layout (shared by keys and values):
 *   cache        tq_cache_bytes(cb, num_pages * Hkv * page_size) bytes; page
 *                p holds, for each kv head h, page_size consecutive rows
 *                starting at row (p*Hkv + h)*page_size (records, then the
 *                norm region, as in any cache)
 *   page_size    tokens per page, a positive multiple of 16
 *   block_table  device int32 [B, max_pages]: token t of sequence b lives in
 *                page block_table[b*max_pages + t/page_size], slot
 *                t % page_size; entries for pages past seq_lens[b] are not read
 *   capacity     max_pages * page_size tokens per sequence (below 2^31)
 * The kernels read the table and seq_lens without validating them against the
 * host: a table entry outside 0..num_pages-1 is never dereferenced (a read
 * goes to page 0 instead, a write is skipped) and sets a flag that the next
 * tq_check_device reports as TQ_EINVAL.                                      */

/* Append one token per (sequence, kv head): x device [B, Hkv, d_in] (TQ_F32
 * or TQ_BF16) is compressed as by tq_quantize and written at token
 * seq_lens[b] - 1 of sequence b (seq_lens counts the appended token);
 * sequences with seq_lens[b] <= 0 are skipped, and a token past the capacity
 * is skipped and flagged.                                                    */
tq_status tq_append_paged(const tq_codebook* cb, void* cache, int32_t num_pages, int32_t page_size,
                          const int32_t* block_table, int32_t max_pages, int32_t B, int32_t Hkv,
                          const int32_t* seq_lens, const void* x, int32_t x_dtype, int32_t d_in,
                          void* stream);

/* tq_logits over a paged key cache (keys as for tq_logits: scalar or polar
 * mode with the QJL term, or MSE-only keys in scalar mode):
 *   logits  device fp32 [B, Hq, max_pages * page_size]
 *   workspace >= tq_logits_workspace(kcb, B, Hq, Hkv) bytes                  */
tq_status tq_logits_paged(const tq_codebook* kcb, const void* kcache, int32_t num_pages, int32_t page_size,
                          const int32_t* block_table, int32_t max_pages, int32_t B, int32_t Hq, int32_t Hkv,
                          const int32_t* seq_lens, const float* q, float* logits, void* workspace,
                          size_t ws_bytes, void* stream);

/* tq_decode_attention over paged key and value caches (same block table and
 * page size for both; scalar or polar mode):
 *   workspace >= tq_decode_attention_workspace(kcb, B, Hq, Hkv,
 *                max_pages * page_size) bytes                                */
tq_status tq_decode_attention_paged(const tq_codebook* kcb, const tq_codebook* vcb, const void* kcache,
                                    const void* vcache, int32_t num_pages, int32_t page_size,
                                    const int32_t* block_table, int32_t max_pages, int32_t B, int32_t Hq,
                                    int32_t Hkv, const int32_t* seq_lens, const float* q, float scale, float* out,
                                    void* workspace, size_t ws_bytes, void* stream);

/* seq_lens[b] += delta for b < B, on the stream.  With it one decode step
 * (tq_advance_lengths by 1, tq_append_paged of the new keys and values,
 * tq_decode_attention_paged) reads and updates only device state, so the step
 * can be captured once in a CUDA graph and replayed step after step.        */
tq_status tq_advance_lengths(int32_t* seq_lens, int32_t B, int32_t delta, void* stream);

/* Workspace bytes of tq_search (depends on n_db, nq, k): query operands and
 * candidate lists of the tensor-core scan, plus the exact scan's query
 * fragments and per-chunk top-k lists. */
size_t tq_search_workspace(const tq_codebook* cb, int64_t n_db, int32_t nq, int32_t k);

/* Top-k inner-product search over a compressed database ([xujun] 常见问题,
 * vector search; [cnyes]): score(q, x_i) is the estimator above; returns, per
 * query, the k best rows by decreasing score, ties to the smaller id.
 *   db_cache   device, rows 0..n_db-1, PROD kind
 *   q          device fp32 [nq, d_in], d_in <= d (zero-padded)
 *   ids        device int32 [nq, k];  scores  device fp32 [nq, k]; entries
 *              past n_db are id -1, score -inf
 *   k          1..32
 * Scores are the fp32 estimator of the returned rows.  With d = 256 (scalar
 * mode, no extra bits) and k <= 16, candidates come from fp16 tensor-core
 * scores (tcgen05, queries held in tensor memory) whose error against the
 * estimator is bounded per query; the candidates are re-scored exactly, and a
 * query whose candidate lists cannot prove its top k (the bound is too wide
 * for its score gaps, e.g. many equal rows) is re-run by the exact scan, so
 * the result is that of the exact scan either way.  Other shapes run the
 * exact scan (fp16 bit-plane products on mma.sync) directly.                */
tq_status tq_search(const tq_codebook* cb, const void* db_cache, int64_t n_db, const float* q,
                    int32_t nq, int32_t d_in, int32_t k, int32_t* ids, float* scores,
                    void* workspace, size_t ws_bytes, void* stream);

/* Test and diagnostic use (synchronises the device): *count = the number of
 * queries of the last tq_search on `workspace` that the exact scan re-ran, or
 * -1 when that call (this codebook, this k) used the exact scan only.       */
tq_status tq_search_fallbacks(const tq_codebook* cb, const void* workspace, int32_t k, int32_t* count);

/* Synchronise the device and report, since the last check, whether any
 * kernel of this codebook gave up a bounded wait on its own copies or
 * tensor-core operations (TQ_ETIMEOUT), or met an append destination or a
 * block-table entry outside the cache (TQ_EINVAL); the flag is cleared.
 * TQ_OK otherwise.  Not a hot call.                                          */
tq_status tq_check_device(const tq_codebook* cb);

/* Test hook: the nth device allocation of tq_make_codebook from now on
 * (0 = the next one) fails as if the device were out of memory, so that the
 * call returns TQ_ENOMEM after freeing what it had allocated; -1 turns the
 * hook off.  Process-wide; for tests only.  Errors: TQ_EINVAL for nth < -1. */
tq_status tq_fail_allocation(int32_t nth);

/* Test use: from the next launch on, the first bounded device-side wait of
 * every kernel that uses this codebook (the first bulk-copy stage of the
 * logits and attention kernels, the Pi / S loads of the tensor-core
 * quantize kernel) gives up after `polls` polls (0: at once; -1: back to the
 * default of 2^26).  A kernel that gives up records TQ_ETIMEOUT for
 * tq_check_device, waits (with the full limit) for the copies and tensor-core
 * operations it has already issued, frees its tensor memory and returns; its
 * outputs are then incomplete.  It lets a test drive the timeout path without
 * faulting or hanging anything.  Not thread-safe against calls running on
 * this codebook.                                                             */
tq_status tq_set_first_wait_limit(tq_codebook* cb, int64_t polls);

/* Message of the calling thread's last failed call ("" if none). */
const char* tq_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H_ */
