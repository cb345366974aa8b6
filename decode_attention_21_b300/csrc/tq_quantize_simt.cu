// Row-wise compression on the CUDA cores (fp32): rotation, stage 1 (scalar
// Lloyd-Max or recursive polar), QJL sign sketch of the residual, bit-plane
// packing and fp16 norms.  One warp per row.  Used for fp32 inputs, for
// already-rotated inputs and for the polar mode; bf16 batches in scalar mode
// take the tensor-core kernel.
//
// [suzuke] "TurboQuant: compressing AI consciousness", 技術上怎麼做到的:
//   第一步 rotate, 第二步 code at b-1 bits (polar angles, Max-Lloyd),
//   第三步 1-bit sign of the projected residual.
// [xujun] note-189244, 第一步 (recursive polar pairing), 第二步 (QJL).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tq_internal.cuh"

namespace tq {

namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Slot (32*word + bit) of angle j of level `lev` (see the polar layout in tq.h).
__device__ __forceinline__ int polar_slot(int lev, int j, int logd) {
  if (lev <= 5) {
    const int per = 32 >> lev;             // 16, 8, 4, 2, 1 angles per subtree
    const int base = 32 - (64 >> lev);     // 0, 16, 24, 28, 30
    return 32 * (j / per) + base + (j % per);
  }
  const int heap = ((1 << (logd - lev)) - 1) + j;
  return 32 * heap + 31;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(256) k_quantize_simt(const Dev cb, uint8_t* __restrict__ cache,
                                                       int64_t cache_rows, const void* __restrict__ x,
                                                       int x_dtype, int64_t n, int d_in,
                                                       const float* __restrict__ y_in,
                                                       const float* __restrict__ n_in, const AppendDst dmap,
                                                       int* __restrict__ status) {
  // a programmatic dependent (the query prep) may start now: it reads none of
  // the rows written here and waits for this grid before it completes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int K = D / 32;
  constexpr int LOGD = D == 128 ? 7 : 8;
  __shared__ float s_y[8][D];
  __shared__ float s_a[8][D];
  __shared__ float s_b[8][D];
  __shared__ unsigned char s_code[8][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* buf = s_y[warp];
  uint32_t* recs = reinterpret_cast<uint32_t*>(cache);
  unsigned char* norms = cache + norm_offset(cb, cache_rows);
  const int b1 = cb.b1, P = cb.P, W = cb.W;
  const bool prod = cb.kind == 0;
  const int64_t stride = (int64_t)gridDim.x * 8;

  // outlier-channel split: word columns k < kx (coordinates 0..extra-1) are
  // group A, with its own norms; otherwise kx = 0 and one group holds all
  const int kx = cb.split ? cb.extra / 32 : 0;
  for (int64_t row = (int64_t)blockIdx.x * 8 + warp; row < n; row += stride) {
    float y[K];
    float nrm, nrm_x = 0.f;
    if (y_in) {
#pragma unroll
      for (int k = 0; k < K; ++k) y[k] = y_in[row * D + lane + 32 * k];
      if (kx) {
        nrm_x = n_in[2 * row];
        nrm = n_in[2 * row + 1];
      } else {
        nrm = n_in[row];
      }
    } else {
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int j = lane + 32 * k;
        float v = 0.f;
        if (j < d_in) {
          if (x_dtype == 0)
            v = static_cast<const float*>(x)[row * d_in + j];
          else
            v = __bfloat162float(static_cast<const __nv_bfloat16*>(x)[row * d_in + j]);
        }
        buf[j] = v;
        y[k] = 0.f;
      }
      __syncwarp();
      for (int j = 0; j < D; ++j) {
        const float xj = buf[j];
        const float* prow = cb.PiT + (size_t)j * D + lane;
#pragma unroll
        for (int k = 0; k < K; ++k) y[k] = fmaf(__ldg(prow + 32 * k), xj, y[k]);
      }
      float ss = 0.f, ssx = 0.f;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        if (k < kx) ssx = fmaf(y[k], y[k], ssx);
        else ss = fmaf(y[k], y[k], ss);
      }
      ss = warp_sum(ss);
      nrm = sqrtf(ss);
      const float inv = nrm > 0.f ? 1.f / nrm : 0.f;
      float inv_x = 0.f;
      if (kx) {
        nrm_x = sqrtf(warp_sum(ssx));
        inv_x = nrm_x > 0.f ? 1.f / nrm_x : 0.f;
      }
#pragma unroll
      for (int k = 0; k < K; ++k) y[k] *= k < kx ? inv_x : inv;
      __syncwarp();
    }

    // ---- stage 1
    int idx[K];
    float r[K];
    if (cb.mode == 0) {
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int i = lane + 32 * k;
        const float v = y[k];
        int c = 0;
        if (i < cb.extra) {
          const int nbd = (2 << b1) - 1;
          for (int t = 0; t < nbd; ++t) c += (v >= cb.bound_x[t]) ? 1 : 0;
          r[k] = v - cb.cent_x[c];
        } else {
          const int nbd = (1 << b1) - 1;
          for (int t = 0; t < nbd; ++t) c += (v >= cb.bound[t]) ? 1 : 0;
          r[k] = v - cb.cent[c];
        }
        idx[k] = c;
      }
    } else {
      // recursive polar: level 1 pairs (y[2a], y[2a+1]), then pairs of radii
      float* ya = s_a[warp];
      float* yb = s_b[warp];
      unsigned char* code = s_code[warp];
#pragma unroll
      for (int k = 0; k < K; ++k) buf[lane + 32 * k] = y[k];
      __syncwarp();
      const int L = 1 << b1;
      for (int a = lane; a < D / 2; a += 32) {
        const float p = buf[2 * a], q = buf[2 * a + 1];
        int Q = 0;
        if (p <= 0.f && q > 0.f) Q = 1;
        else if (p < 0.f && q <= 0.f) Q = 2;
        else if (p >= 0.f && q < 0.f) Q = 3;
        const float ar = Q == 0 ? p : (Q == 1 ? q : (Q == 2 ? -p : -q));
        const float br = Q == 0 ? q : (Q == 1 ? -p : (Q == 2 ? -q : p));
        int c;
        if (L == 2) c = Q >> 1;
        else if (L == 4) c = Q;
        else {
          const int per = L / 4;
          int cnt = 0;
          for (int j = 0; j < per - 1; ++j) cnt += ge_exact(br, ar, cb.pb_cos[1][j], cb.pb_sin[1][j]);
          c = Q * per + cnt;
        }
        code[polar_slot(1, a, LOGD)] = (unsigned char)c;
        ya[a] = radius_rn(p, q);
      }
      __syncwarp();
      float* rin = ya;
      float* rout = yb;
      for (int lev = 2; lev <= LOGD; ++lev) {
        const int cnt_ang = D >> lev;
        for (int j = lane; j < cnt_ang; j += 32) {
          const float ra = rin[2 * j], rb = rin[2 * j + 1];
          int c = 0;
          for (int t = 0; t < L - 1; ++t) c += ge_exact(rb, ra, cb.pb_cos[lev][t], cb.pb_sin[lev][t]);
          code[polar_slot(lev, j, LOGD)] = (unsigned char)c;
          rout[j] = radius_rn(ra, rb);
        }
        __syncwarp();
        float* tmp = rin;
        rin = rout;
        rout = tmp;
      }
      // decode the reproduction, root radius 1
      if (lane == 0) rin[0] = 1.f;
      __syncwarp();
      for (int lev = LOGD; lev >= 2; --lev) {
        const int cnt_ang = D >> lev;
        for (int j = lane; j < cnt_ang; j += 32) {
          const int c = code[polar_slot(lev, j, LOGD)];
          const float rho = rin[j];
          rout[2 * j] = rho * cb.pc_cos[lev][c];
          rout[2 * j + 1] = rho * cb.pc_sin[lev][c];
        }
        __syncwarp();
        float* tmp = rin;
        rin = rout;
        rout = tmp;
      }
      for (int a = lane; a < D / 2; a += 32) {
        const int c = code[polar_slot(1, a, LOGD)];
        rout[2 * a] = rin[a] * cb.pc_cos[1][c];
        rout[2 * a + 1] = rin[a] * cb.pc_sin[1][c];
      }
      __syncwarp();
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int i = lane + 32 * k;
        r[k] = y[k] - rout[i];
        idx[k] = (i == D - 1) ? 0 : code[i];   // slot view; the last slot is padding
      }
      __syncwarp();
    }

    // ---- pack code planes (bit j of word c <-> coordinate / slot 32c + j)
    uint32_t mine0 = 0, mine1 = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int i = lane + 32 * k;
      const int top = (i < cb.extra) ? (idx[k] >> 1) : idx[k];
      for (int p = 0; p < b1; ++p) {
        const uint32_t w = __ballot_sync(kFull, (top >> (b1 - 1 - p)) & 1);
        const int wi = k * P + p;
        if ((wi & 31) == lane) {
          if (wi < 32) mine0 = w; else mine1 = w;
        }
      }
    }
    for (int k = 0; k < cb.extra / 32; ++k) {
      const uint32_t w = __ballot_sync(kFull, idx[k] & 1);
      const int wi = (D / 32) * P + k;
      if ((wi & 31) == lane) {
        if (wi < 32) mine0 = w; else mine1 = w;
      }
    }

    // ---- QJL: gamma = ||r|| (per group for a split), signs of S r
    float gamma = 0.f, gamma_x = 0.f;
    if (prod) {
      float ss = 0.f, ssx = 0.f;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        if (k < kx) ssx = fmaf(r[k], r[k], ssx);
        else ss = fmaf(r[k], r[k], ss);
      }
      gamma = sqrtf(warp_sum(ss));
      if (kx) gamma_x = sqrtf(warp_sum(ssx));
      __syncwarp();
#pragma unroll
      for (int k = 0; k < K; ++k) buf[lane + 32 * k] = r[k];
      __syncwarp();
      float z[K];
#pragma unroll
      for (int k = 0; k < K; ++k) z[k] = 0.f;
      for (int i = 0; i < D; ++i) {
        const float ri = buf[i];
        const float* srow = cb.ST + (size_t)i * D + lane;
#pragma unroll
        for (int k = 0; k < K; ++k) z[k] = fmaf(__ldg(srow + 32 * k), ri, z[k]);
      }
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const uint32_t w = __ballot_sync(kFull, z[k] >= 0.f);
        const int wi = k * P + b1;
        if ((wi & 31) == lane) {
          if (wi < 32) mine0 = w; else mine1 = w;
        }
      }
    }
    __syncwarp();

    // ---- store (a destination outside the cache is skipped and flagged)
    const int64_t dst = append_row(dmap, row, cache_rows);
    if (dst == -2 && lane == 0) atomicOr(status, kBadRow);
    if (dst >= 0) {
      uint32_t* rec = recs + dst * W;
      if (lane < W) rec[lane] = mine0;
      if (lane + 32 < W) rec[lane + 32] = mine1;
      if (lane == 0) {
        if (kx) {
          __half2* e = reinterpret_cast<__half2*>(norms) + 2 * dst;
          e[0] = __floats2half2_rn(nrm_x, gamma_x);
          e[1] = __floats2half2_rn(nrm, gamma);
        } else if (prod) {
          reinterpret_cast<__half2*>(norms)[dst] = __floats2half2_rn(nrm, gamma);
        } else {
          reinterpret_cast<__half*>(norms)[dst] = __float2half_rn(nrm);
        }
      }
    }
  }
}

// Latency path for short batches (a decode step appends one vector per kv
// head): one CTA per row, 4 threads per coordinate, so each row's two
// matrix-vector products are 4 x D independent 32-term dot products whose
// loads are all in flight at once.  Scalar mode only; same arithmetic and bit
// layout as k_quantize_simt.
template <int D>
struct Quarter {
  float m[D / 4];
  // column slice i, rows q*D/4 .. (q+1)*D/4 - 1 of the transposed matrix MT
  __device__ __forceinline__ void load(const float* __restrict__ MT, int i, int q) {
    const float* col = MT + (size_t)(q * (D / 4)) * D + i;
    const uint64_t keep = l2_policy_evict_last();
#pragma unroll
    for (int j = 0; j < D / 4; ++j) m[j] = ld_table(col + (size_t)j * D, keep);
  }
  __device__ __forceinline__ float dot(const float* xs, int q) const {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < D / 4; ++j) acc = fmaf(m[j], xs[q * (D / 4) + j], acc);
    return acc;
  }
};

template <int D>
__global__ void __launch_bounds__(4 * D) k_quantize_row(const Dev cb, uint8_t* __restrict__ cache, int64_t cache_rows,
                                                        const void* __restrict__ x, int x_dtype, int64_t n, int d_in,
                                                        const float* __restrict__ y_in, const float* __restrict__ n_in,
                                                        const AppendDst dmap, int* __restrict__ status) {
  // a programmatic dependent (the query prep) may start now: it reads none of
  // the rows written here and waits for this grid before it completes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int NW = D / 32;
  __shared__ float xs[D];
  __shared__ float part[4][D];
  __shared__ float red[NW];
  __shared__ uint32_t words[64];
  const int t = threadIdx.x, i = t % D, q = t / D;
  const int lane = i & 31, w = i >> 5;
  const int b1 = cb.b1, P = cb.P;
  const bool prod = cb.kind == 0;
  uint32_t* recs = reinterpret_cast<uint32_t*>(cache);
  unsigned char* norms = cache + norm_offset(cb, cache_rows);
  // at d = 128 both matrices' column slices stay in registers for every row
  // of this CTA (one round trip to L2); the 1024-thread d = 256 CTA reloads them
  constexpr bool kKeep = D == 128;
  Quarter<kKeep ? D : 4> mpi, ms;
  if (kKeep && !y_in) mpi.load(cb.PiT, i, q);
  if (kKeep && prod) ms.load(cb.ST, i, q);
  // outlier-channel split: warps w < kx (coordinates 0..extra-1) are group
  // A, with its own norms; otherwise kx = 0
  const int kx = cb.split ? cb.extra / 32 : 0;
  for (int64_t row = blockIdx.x; row < n; row += gridDim.x) {
    float y = 0.f, nrm = 0.f;
    if (y_in) {
      if (q == 0) {
        y = y_in[row * D + i];
        nrm = kx ? n_in[2 * row + (w < kx ? 0 : 1)] : n_in[row];
      }
    } else {
      if (q == 0) {
        float v = 0.f;
        if (i < d_in) {
          if (x_dtype == 0)
            v = static_cast<const float*>(x)[row * d_in + i];
          else
            v = __bfloat162float(static_cast<const __nv_bfloat16*>(x)[row * d_in + i]);
        }
        xs[i] = v;
      }
      __syncthreads();
      if constexpr (kKeep) {
        part[q][i] = mpi.dot(xs, q);
      } else {
        Quarter<D> m1;
        m1.load(cb.PiT, i, q);
        part[q][i] = m1.dot(xs, q);
      }
      __syncthreads();
      if (q == 0) {
        y = (part[0][i] + part[1][i]) + (part[2][i] + part[3][i]);
        const float ss = warp_sum(y * y);
        if (lane == 0) red[w] = ss;
      }
      __syncthreads();
      if (q == 0) {
        // this thread's group: words kx.. (group B, or all), or 0..kx-1
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < NW; ++k) ss += ((k < kx) == (w < kx)) ? red[k] : 0.f;
        nrm = sqrtf(ss);
        y *= nrm > 0.f ? 1.f / nrm : 0.f;
      }
    }
    float r = 0.f;
    int idx = 0;
    if (q == 0) {
      if (i < cb.extra) {
        const int nbd = (2 << b1) - 1;
        for (int k = 0; k < nbd; ++k) idx += (y >= cb.bound_x[k]) ? 1 : 0;
        r = y - cb.cent_x[idx];
      } else {
        const int nbd = (1 << b1) - 1;
        for (int k = 0; k < nbd; ++k) idx += (y >= cb.bound[k]) ? 1 : 0;
        r = y - cb.cent[idx];
      }
      const int top = i < cb.extra ? idx >> 1 : idx;
      for (int p = 0; p < b1; ++p) {
        const uint32_t bw = __ballot_sync(kFull, (top >> (b1 - 1 - p)) & 1);
        if (lane == 0) words[w * P + p] = bw;
      }
      if (i < cb.extra) {
        const uint32_t bw = __ballot_sync(kFull, idx & 1);
        if (lane == 0) words[NW * P + w] = bw;
      }
    }
    // every warp has read the norm partials in red before they are replaced
    // by the residual's
    __syncthreads();
    if (q == 0 && prod) {
      xs[i] = r;
      const float ss = warp_sum(r * r);
      if (lane == 0) red[w] = ss;
    }
    __syncthreads();
    float gamma = 0.f, nrm_x = 0.f, gamma_x = 0.f;
    if (prod) {
      if constexpr (kKeep) {
        part[q][i] = ms.dot(xs, q);
      } else {
        Quarter<D> m2;
        m2.load(cb.ST, i, q);
        part[q][i] = m2.dot(xs, q);
      }
      __syncthreads();
      if (q == 0) {
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < NW; ++k) ss += ((k < kx) == (w < kx)) ? red[k] : 0.f;
        gamma = sqrtf(ss);
        const float z = (part[0][i] + part[1][i]) + (part[2][i] + part[3][i]);
        const uint32_t bw = __ballot_sync(kFull, z >= 0.f);
        if (lane == 0) words[w * P + b1] = bw;
      }
    }
    __syncthreads();
    // a split's norm entry is written by thread 0 (group A) with group B's
    // values taken from thread 32 kx (the first coordinate of group B); kx
    // is the same for the whole block
    if (kx) {
      if (t == 32 * kx) {
        xs[0] = nrm;
        xs[1] = gamma;
      }
      __syncthreads();
      if (t == 0) {
        nrm_x = nrm;
        gamma_x = gamma;
        nrm = xs[0];
        gamma = xs[1];
      }
    }
    // Launched as a programmatic dependent, this CTA may have computed its
    // rows while the kernel before it (a scoring kernel reading this cache)
    // was still running: nothing is written, and no destination is looked up,
    // before that kernel has completed (a no-op after the first row, and for
    // an ordinary launch).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // a destination outside the cache is skipped and flagged
    const int64_t dst = append_row(dmap, row, cache_rows);
    if (dst == -2 && t == 0) atomicOr(status, kBadRow);
    if (dst >= 0) {
      if (t < cb.W) recs[dst * cb.W + t] = words[t];
      if (t == 0) {
        if (kx) {
          __half2* e = reinterpret_cast<__half2*>(norms) + 2 * dst;
          e[0] = __floats2half2_rn(nrm_x, gamma_x);
          e[1] = __floats2half2_rn(nrm, gamma);
        } else if (prod) {
          reinterpret_cast<__half2*>(norms)[dst] = __floats2half2_rn(nrm, gamma);
        } else {
          reinterpret_cast<__half*>(norms)[dst] = __float2half_rn(nrm);
        }
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_quantize_simt(const Dev& cb, uint8_t* cache, int64_t cache_rows, const void* x, int x_dtype,
                                 int64_t n, int d_in, const float* y, const float* norms, const AppendDst& dst,
                                 int* status, cudaStream_t s) {
  if (cb.mode == 0 && n <= 16384) {
    // short batches (a decode step's appends): launched as a programmatic
    // dependent, so the rows are rotated and coded while the previous kernel
    // finishes; the stores wait for it (griddepcontrol.wait in the kernel)
    const int blocks = (int)(n < 148 * 16 ? n : 148 * 16);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(cb.d == 128 ? 512 : 1024);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cb.d == 128)
      return cudaLaunchKernelEx(&cfg, k_quantize_row<128>, cb, cache, cache_rows, x, x_dtype, n, d_in, y, norms, dst,
                                status);
    return cudaLaunchKernelEx(&cfg, k_quantize_row<256>, cb, cache, cache_rows, x, x_dtype, n, d_in, y, norms, dst,
                              status);
  }
  const int64_t blocks64 = (n + 7) / 8;
  const int blocks = (int)(blocks64 < 148 * 16 ? (blocks64 > 0 ? blocks64 : 1) : 148 * 16);
  if (cb.d == 128)
    k_quantize_simt<128><<<blocks, 256, 0, s>>>(cb, cache, cache_rows, x, x_dtype, n, d_in, y, norms, dst, status);
  else
    k_quantize_simt<256><<<blocks, 256, 0, s>>>(cb, cache, cache_rows, x, x_dtype, n, d_in, y, norms, dst, status);
  return cudaGetLastError();
}

// Decode-loop bookkeeping on the device: seq_lens[b] += delta, so a captured
// step (advance, append, attend) can be replayed without host updates.
__global__ void k_advance_lengths(int32_t* __restrict__ seq_lens, int B, int32_t delta) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) seq_lens[b] += delta;
}

cudaError_t launch_advance_lengths(int32_t* seq_lens, int B, int32_t delta, cudaStream_t s) {
  k_advance_lengths<<<(B + 255) / 256, 256, 0, s>>>(seq_lens, B, delta);
  return cudaGetLastError();
}

}  // namespace tq
