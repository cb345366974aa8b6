// C ABI of the TurboQuant hot path: codebook setup, argument validation and
// kernel launches.  Every declaration is documented in include/tq.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "tq.h"
#include "tq_internal.cuh"
#include "tq_math.h"

namespace tq {
NvtxRange::NvtxRange(const char* name) { nvtxRangePushA(name); }
NvtxRange::~NvtxRange() { nvtxRangePop(); }
}  // namespace tq


struct tq_codebook {
  tq::Dev dev;
  tq_codebook_desc desc;
  int device;
  int sms;
  std::vector<float> cent, bound;
  std::vector<double> pi;
  std::vector<float> s;
  std::vector<void*> allocs;
  bool tc_ready;                  // tensor maps of Pi_hi, Pi_lo, S built
  CUtensorMap tm_pihi, tm_pilo, tm_s;
  int* d_status;                  // device word set by a kernel whose bounded wait gave up
};

namespace {

thread_local std::string g_err;

tq_status fail(tq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

tq_status ok() {
  g_err.clear();
  return TQ_OK;
}

tq_status launched(const char* what, cudaError_t e) {
  if (e != cudaSuccess) return fail(TQ_ECUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return ok();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 row-major [rows, cols] matrix, 128-byte swizzled boxes of 64 columns x 128 rows.
// Row-major bf16 matrix, tiles of 64 columns x box_rows rows, 128-byte swizzle.
bool encode_bf16_rows(CUtensorMap* tm, const void* base, int64_t rows, int64_t cols, uint32_t box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr uint32_t kOddMaskHost[8] = {1u, 2u, 4u, 7u, 8u, 11u, 13u, 14u};
constexpr long long kDefaultWaitPolls = 1ll << 26;   // polls of a bounded device-side wait
constexpr int kLogitsCtas = 148 * 4;   // resident CTAs of the logits kernel
// Resident CTAs of the attention kernel (one wave): 4 per SM, 3 for keys
// with four or more stage-1 virtual planes or extra-bit words (more
// registers), 3 in polar mode.
int attn_ctas(const tq_codebook* kcb, const tq_codebook* vcb = nullptr) {
  if (kcb->dev.mode == TQ_MODE_POLAR) return 148 * 3;
  const bool heavy = kcb->dev.nv >= 4 || kcb->dev.extra > 0 || (vcb && vcb->dev.extra > 0);
  return heavy ? 148 * 3 : 148 * 4;
}

// Test hook (tq_fail_allocation): device allocations of tq_make_codebook
// still to go before one fails as if the device were out of memory (-1: none).
int g_fail_after = -1;

template <class T>
tq_status upload(tq_codebook* cb, const std::vector<T>& h, const T** out) {
  void* p = nullptr;
  if (g_fail_after >= 0 && g_fail_after-- == 0)
    return fail(TQ_ENOMEM, "cudaMalloc(%zu) failed: allocation failure injected by tq_fail_allocation",
                h.size() * sizeof(T));
  cudaError_t e = cudaMalloc(&p, h.size() * sizeof(T));
  if (e != cudaSuccess) return fail(TQ_ENOMEM, "cudaMalloc(%zu) failed: %s", h.size() * sizeof(T), cudaGetErrorString(e));
  cb->allocs.push_back(p);
  e = cudaMemcpy(p, h.data(), h.size() * sizeof(T), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(TQ_ECUDA, "cudaMemcpy failed: %s", cudaGetErrorString(e));
  *out = static_cast<const T*>(p);
  return TQ_OK;
}

uint16_t bf16_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
  return (uint16_t)u;
}

float bf16_value(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

void chunking(int B, int Hkv, int64_t capacity, int target, int* nchunks, int* tiles_per_cta) {
  const int64_t tiles = (capacity + 15) / 16;
  if (tiles <= 0) {
    *nchunks = 1;
    *tiles_per_cta = 4;
    return;
  }
  // as many chunks per unit as fit in one wave of `target` resident CTAs
  // (rounding up would leave a few CTAs for a second wave)
  const int64_t units = (int64_t)B * Hkv;
  const int64_t want = std::max<int64_t>(1, target / units);
  int64_t tpc = std::max<int64_t>(4, (tiles + want - 1) / want);
  *tiles_per_cta = (int)tpc;
  *nchunks = (int)((tiles + tpc - 1) / tpc);
}

tq_status check_scoring_codebook(const tq_codebook* cb, int kind, const char* what, bool mixed_ok = false) {
  if (!cb) return fail(TQ_EINVAL, "%s: codebook is NULL", what);
  if (cb->dev.kind != kind) return fail(TQ_EINVAL, "%s: codebook has the wrong kind", what);
  if (cb->dev.d != 128) return fail(TQ_EUNSUPPORTED, "%s: only d = 128 is implemented", what);
  if (cb->dev.extra != 0 && !(mixed_ok && cb->dev.kind == TQ_KIND_PROD && cb->dev.mode == TQ_MODE_SCALAR &&
                              cb->dev.extra <= 64))
    return fail(TQ_EUNSUPPORTED, "%s: this mixed-bit cache is not scored here", what);
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != cb->device) return fail(TQ_EINVAL, "%s: codebook lives on device %d, current device is %d", what, cb->device, dev);
  return TQ_OK;
}

}  // namespace

namespace tq {
// Records an error message for tq_last_error (used by entry points in other files).
tq_status report_error(tq_status st, const char* msg) { return fail(st, "%s", msg); }
}  // namespace tq

extern "C" {

const char* tq_last_error(void) { return g_err.c_str(); }

static tq_status check_desc(const tq_codebook_desc* desc, const char* what) {
  const tq_codebook_desc& D = *desc;
  if (D.d != 128 && D.d != 256) return fail(TQ_EINVAL, "%s: d must be 128 or 256 (got %d)", what, D.d);
  if (D.kind != TQ_KIND_PROD && D.kind != TQ_KIND_MSE) return fail(TQ_EINVAL, "%s: bad kind %d", what, D.kind);
  if (D.mode != TQ_MODE_SCALAR && D.mode != TQ_MODE_POLAR) return fail(TQ_EINVAL, "%s: bad mode %d", what, D.mode);
  const int b1 = D.kind == TQ_KIND_PROD ? D.bits - 1 : D.bits;
  if (b1 < 1 || b1 > 4 || (D.kind == TQ_KIND_PROD && b1 > 3))
    return fail(TQ_EINVAL, "%s: bits %d out of range for this kind", what, D.bits);
  if (D.kind == TQ_KIND_PROD && D.m != D.d) return fail(TQ_EINVAL, "%s: m must equal d", what);
  if (D.extra != 0 && D.extra != D.d / 4 && D.extra != D.d / 2)
    return fail(TQ_EINVAL, "%s: extra must be 0, d/4 or d/2", what);
  if (D.extra != 0 && (D.mode != TQ_MODE_SCALAR || b1 + 1 > 4))
    return fail(TQ_EINVAL, "%s: extra bits need scalar mode and b' <= 3", what);
  if (D.outliers) {
    if (D.d != 128 || D.kind != TQ_KIND_PROD || D.mode != TQ_MODE_SCALAR || D.extra == 0)
      return fail(TQ_EINVAL, "%s: the outlier-channel split needs d = 128, PROD kind, scalar mode and extra = 32 or 64",
                  what);
    if (D.pi || D.s) return fail(TQ_EINVAL, "%s: the outlier-channel split takes no Pi or S override", what);
    std::vector<char> seen(D.d, 0);
    for (int e = 0; e < D.extra; ++e) {
      const int c = D.outliers[e];
      if (c < 0 || c >= D.d || seen[c]) return fail(TQ_EINVAL, "%s: outlier channels must be distinct, in 0..d-1", what);
      seen[c] = 1;
    }
  }
  return TQ_OK;
}

// Outlier-channel split: the d x d rotation x -> (Pi_A x_A, Pi_B x_B) (rows
// 0..E-1 from group A's channels in the listed order, the rest from group B's
// in channel order) and the block-diagonal sketch diag(S_A, S_B), each group
// drawn from its own seeds (A: seed_pi, seed_s; B: seed_pi + 1, seed_s + 1).
static void split_matrices(const tq_codebook_desc& D, std::vector<double>& pi, std::vector<float>& s) {
  const int d = D.d, E = D.extra, F = d - E;
  std::vector<int> B;
  std::vector<char> isA(d, 0);
  for (int e = 0; e < E; ++e) isA[D.outliers[e]] = 1;
  for (int c = 0; c < d; ++c)
    if (!isA[c]) B.push_back(c);
  const std::vector<double> pa = tqm::haar_rotation(E, D.seed_pi), pb = tqm::haar_rotation(F, D.seed_pi + 1);
  pi.assign((size_t)d * d, 0.0);
  for (int i = 0; i < E; ++i)
    for (int j = 0; j < E; ++j) pi[(size_t)i * d + D.outliers[j]] = pa[(size_t)i * E + j];
  for (int i = 0; i < F; ++i)
    for (int j = 0; j < F; ++j) pi[(size_t)(E + i) * d + B[j]] = pb[(size_t)i * F + j];
  const std::vector<double> sa = tqm::gaussians(D.seed_s, (size_t)E * E), sb = tqm::gaussians(D.seed_s + 1, (size_t)F * F);
  s.assign((size_t)d * d, 0.f);
  for (int i = 0; i < E; ++i)
    for (int j = 0; j < E; ++j) s[(size_t)i * d + j] = tqm::round_bf16(sa[(size_t)i * E + j]);
  for (int i = 0; i < F; ++i)
    for (int j = 0; j < F; ++j) s[(size_t)(E + i) * d + E + j] = tqm::round_bf16(sb[(size_t)i * F + j]);
}

tq_status tq_host_tables(const tq_codebook_desc* desc, int32_t level, float* centroids, float* boundaries,
                         double* pi, float* s) {
  if (!desc) return fail(TQ_EINVAL, "tq_host_tables: NULL descriptor");
  tq_status st = check_desc(desc, "tq_host_tables");
  if (st != TQ_OK) return st;
  const tq_codebook_desc& D = *desc;
  const int d = D.d;
  const int b1 = D.kind == TQ_KIND_PROD ? D.bits - 1 : D.bits;
  const int L = 1 << b1;
  const int logd = d == 128 ? 7 : 8;
  if (D.mode == TQ_MODE_SCALAR) {
    const tqm::Quantizer q = tqm::lloyd_max_beta(D.outliers ? d - D.extra : d, L);
    for (int k = 0; k < L && centroids; ++k) centroids[k] = (float)q.c[k];
    for (int k = 0; k < L - 1 && boundaries; ++k) boundaries[k] = (float)q.t[k];
  } else {
    if (level < 1 || level > logd) return fail(TQ_EINVAL, "tq_host_tables: level %d out of 1..%d", level, logd);
    if (level == 1) {
      for (int k = 0; k < L && centroids; ++k) centroids[k] = (float)((2.0 * k + 1.0) * M_PI / L);
      for (int k = 0; k < L - 1 && boundaries; ++k) boundaries[k] = (float)(2.0 * M_PI * (k + 1) / L);
    } else {
      const tqm::Quantizer q = tqm::lloyd_max_polar(1 << (level - 1), L);
      for (int k = 0; k < L && centroids; ++k) centroids[k] = (float)q.c[k];
      for (int k = 0; k < L - 1 && boundaries; ++k) boundaries[k] = (float)q.t[k];
    }
  }
  if (D.outliers) {
    std::vector<double> P;
    std::vector<float> S;
    split_matrices(D, P, S);
    if (pi) std::memcpy(pi, P.data(), P.size() * sizeof(double));
    if (s) std::memcpy(s, S.data(), S.size() * sizeof(float));
    return ok();
  }
  if (pi) {
    const std::vector<double> P = D.pi ? std::vector<double>(D.pi, D.pi + (size_t)d * d) : tqm::haar_rotation(d, D.seed_pi);
    std::memcpy(pi, P.data(), P.size() * sizeof(double));
  }
  if (s && D.kind == TQ_KIND_PROD) {
    const std::vector<double> g = tqm::gaussians(D.seed_s, (size_t)D.m * d);
    for (size_t e = 0; e < g.size(); ++e) s[e] = D.s ? D.s[e] : tqm::round_bf16(g[e]);
  }
  return ok();
}

tq_status tq_make_codebook(const tq_codebook_desc* desc, tq_codebook** out) {
  const tq::NvtxRange nvtx_range("tq_make_codebook");
  if (!desc || !out) return fail(TQ_EINVAL, "tq_make_codebook: NULL argument");
  *out = nullptr;
  const tq_codebook_desc& D = *desc;
  {
    tq_status st0 = check_desc(desc, "tq_make_codebook");
    if (st0 != TQ_OK) return st0;
  }
  const int b1 = D.kind == TQ_KIND_PROD ? D.bits - 1 : D.bits;

  int device = -1;
  {
    const cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return fail(TQ_ECUDA, "tq_make_codebook: no CUDA device: %s", cudaGetErrorString(e));
  }
  tq_codebook* cb = new tq_codebook();
  cb->desc = D;
  cb->desc.pi = nullptr;
  cb->desc.s = nullptr;
  cb->desc.outliers = nullptr;
  cb->device = device;
  tq::Dev& dv = cb->dev;
  std::memset(&dv, 0, sizeof(dv));
  const int d = D.d;
  dv.d = d;
  dv.m = D.kind == TQ_KIND_PROD ? D.m : 0;
  dv.b1 = b1;
  dv.kind = D.kind;
  dv.mode = D.mode;
  dv.extra = D.extra;
  dv.P = b1 + (D.kind == TQ_KIND_PROD ? 1 : 0);
  dv.W = (d / 32) * dv.P + D.extra / 32;
  dv.split = D.outliers != nullptr;
  dv.nb = dv.split ? 8 : (D.kind == TQ_KIND_PROD ? 4 : 2);
  // group B (the main codebook) and group A (the extended one) of a split
  // are E- and (d - E)-dimensional instances: own laws and QJL constants
  const int d_main = dv.split ? d - D.extra : d, d_ext = dv.split ? D.extra : d;
  dv.qjl_const = (float)(std::sqrt(M_PI / 2.0) / d_main);
  dv.qjl_const_x = (float)(std::sqrt(M_PI / 2.0) / d_ext);
  dv.first_wait = kDefaultWaitPolls;
  const int L = 1 << b1;

  if (D.mode == TQ_MODE_SCALAR) {
    const tqm::Quantizer q = tqm::lloyd_max_beta(d_main, L);
    cb->cent.resize(L);
    cb->bound.resize(L - 1);
    for (int k = 0; k < L; ++k) cb->cent[k] = dv.cent[k] = (float)q.c[k];
    for (int k = 0; k < L - 1; ++k) cb->bound[k] = dv.bound[k] = (float)q.t[k];
    if (D.extra) {
      const tqm::Quantizer qx = tqm::lloyd_max_beta(d_ext, 2 * L);
      for (int k = 0; k < 2 * L; ++k) dv.cent_x[k] = (float)qx.c[k];
      for (int k = 0; k < 2 * L - 1; ++k) dv.bound_x[k] = (float)qx.t[k];
    }
    // Walsh-Hadamard expansion of the centroid table over the +-1 planes
    // s'_p = (-1)^(bit p of idx), plane 0 = most significant bit.
    dv.nv = L / 2;
    for (int v = 0; v < dv.nv; ++v) {
      const uint32_t mask = kOddMaskHost[v];
      double a = 0.0;
      for (int idx = 0; idx < L; ++idx) {
        int par = 0;
        for (int p = 0; p < b1; ++p)
          if (mask >> p & 1u) par ^= (idx >> (b1 - 1 - p)) & 1;
        a += (par ? -1.0 : 1.0) * (double)dv.cent[idx];
      }
      dv.vmask[v] = mask;
      dv.vcoef[v] = (float)(a / L);
    }
    // extended codebook: idx_x = (top << 1) | extra bit, plane p (p <= b1) is
    // bit b1 - p of idx_x
    dv.nvx = D.extra ? L : 0;
    for (int v = 0; v < dv.nvx; ++v) {
      const uint32_t mask = kOddMaskHost[v];
      double a = 0.0;
      for (int idx = 0; idx < 2 * L; ++idx) {
        int par = 0;
        for (int p = 0; p <= b1; ++p)
          if (mask >> p & 1u) par ^= (idx >> (b1 - p)) & 1;
        a += (par ? -1.0 : 1.0) * (double)dv.cent_x[idx];
      }
      dv.vcoef_x[v] = (float)(a / (2 * L));
    }
    for (int idx = 0; idx < (D.extra ? 2 * L : 0); ++idx) {
      double r = 0.0;
      for (int v = 0; v < dv.nvx; ++v) {
        int par = 0;
        for (int p = 0; p <= b1; ++p)
          if (kOddMaskHost[v] >> p & 1u) par ^= (idx >> (b1 - p)) & 1;
        r += (par ? -1.0 : 1.0) * dv.vcoef_x[v];
      }
      if (std::fabs(r - dv.cent_x[idx]) > 1e-6 * std::fabs(dv.cent_x[2 * L - 1])) {
        delete cb;
        return fail(TQ_EINVAL, "tq_make_codebook: extended centroid table is not symmetric");
      }
    }
    // the expansion must reproduce every centroid (even subsets vanish for a
    // symmetric table)
    for (int idx = 0; idx < L; ++idx) {
      double r = 0.0;
      for (int v = 0; v < dv.nv; ++v) {
        int par = 0;
        for (int p = 0; p < b1; ++p)
          if (dv.vmask[v] >> p & 1u) par ^= (idx >> (b1 - 1 - p)) & 1;
        r += (par ? -1.0 : 1.0) * dv.vcoef[v];
      }
      if (std::fabs(r - dv.cent[idx]) > 1e-6 * std::fabs(dv.cent[L - 1])) {
        delete cb;
        return fail(TQ_EINVAL, "tq_make_codebook: centroid table is not symmetric");
      }
    }
  } else {
    const int logd = d == 128 ? 7 : 8;
    // level 1: uniform quantizer on [0, 2 pi); boundaries inside the first quadrant
    for (int j = 1; j < L / 4; ++j) {
      const double t = (double)(float)(2.0 * M_PI * j / L);
      dv.pb_cos[1][j - 1] = (float)std::cos(t);
      dv.pb_sin[1][j - 1] = (float)std::sin(t);
    }
    for (int k = 0; k < L; ++k) {
      const double c = (double)(float)((2.0 * k + 1.0) * M_PI / L);
      dv.pc_cos[1][k] = (float)std::cos(c);
      dv.pc_sin[1][k] = (float)std::sin(c);
    }
    for (int lev = 2; lev <= logd; ++lev) {
      const tqm::Quantizer q = tqm::lloyd_max_polar(1 << (lev - 1), L);
      for (int k = 0; k < L - 1; ++k) {
        const double t = (double)(float)q.t[k];
        dv.pb_cos[lev][k] = (float)std::cos(t);
        dv.pb_sin[lev][k] = (float)std::sin(t);
      }
      for (int k = 0; k < L; ++k) {
        const double c = (double)(float)q.c[k];
        dv.pc_cos[lev][k] = (float)std::cos(c);
        dv.pc_sin[lev][k] = (float)std::sin(c);
      }
      if (lev == 2) {
        cb->cent.resize(L);
        cb->bound.resize(L - 1);
        for (int k = 0; k < L; ++k) cb->cent[k] = (float)q.c[k];
        for (int k = 0; k < L - 1; ++k) cb->bound[k] = (float)q.t[k];
      }
    }
    dv.nv = 1;   // one decoded stage-1 plane for the scoring kernels
  }

  // rotation
  std::vector<float> split_s;
  if (dv.split) {
    split_matrices(D, cb->pi, split_s);
  } else if (D.pi) {
    cb->pi.assign(D.pi, D.pi + (size_t)d * d);
  } else {
    cb->pi = tqm::haar_rotation(d, D.seed_pi);
  }
  std::vector<float> pi32((size_t)d * d), piT((size_t)d * d);
  std::vector<uint16_t> pi_hi((size_t)d * d), pi_lo((size_t)d * d);
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) {
      const float v = (float)cb->pi[(size_t)i * d + j];
      pi32[(size_t)i * d + j] = v;
      piT[(size_t)j * d + i] = v;
      const uint16_t h = bf16_bits(v);
      pi_hi[(size_t)i * d + j] = h;
      pi_lo[(size_t)i * d + j] = bf16_bits(v - bf16_value(h));
    }
  tq_status st;
  if ((st = upload(cb, pi32, &dv.Pi)) != TQ_OK || (st = upload(cb, piT, &dv.PiT)) != TQ_OK ||
      (st = upload(cb, pi_hi, &dv.Pi_hi)) != TQ_OK || (st = upload(cb, pi_lo, &dv.Pi_lo)) != TQ_OK) {
    tq_free_codebook(cb);
    return st;
  }
  if (D.kind == TQ_KIND_PROD) {
    const int m = D.m;
    cb->s.resize((size_t)m * d);
    if (dv.split) {
      cb->s = split_s;
    } else if (D.s) {
      for (size_t e = 0; e < cb->s.size(); ++e) {
        if (tqm::round_bf16(D.s[e]) != D.s[e]) {
          tq_free_codebook(cb);
          return fail(TQ_EINVAL, "tq_make_codebook: S entries must be bf16-exact");
        }
        cb->s[e] = D.s[e];
      }
    } else {
      const std::vector<double> g = tqm::gaussians(D.seed_s, (size_t)m * d);
      for (size_t e = 0; e < cb->s.size(); ++e) cb->s[e] = tqm::round_bf16(g[e]);
    }
    std::vector<float> sT((size_t)d * m);
    std::vector<uint16_t> sbf((size_t)m * d);
    for (int j = 0; j < m; ++j)
      for (int i = 0; i < d; ++i) {
        sT[(size_t)i * m + j] = cb->s[(size_t)j * d + i];
        sbf[(size_t)j * d + i] = bf16_bits(cb->s[(size_t)j * d + i]);
      }
    // (S Pi), accumulated in fp64, stored transposed
    std::vector<float> spT((size_t)d * m);
    for (int j = 0; j < m; ++j)
      for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int k = 0; k < d; ++k) acc += (double)cb->s[(size_t)j * d + k] * cb->pi[(size_t)k * d + i];
        spT[(size_t)i * m + j] = (float)acc;
      }
    if ((st = upload(cb, sT, &dv.ST)) != TQ_OK || (st = upload(cb, sbf, &dv.S_bf)) != TQ_OK ||
        (st = upload(cb, spT, &dv.SPT)) != TQ_OK) {
      tq_free_codebook(cb);
      return st;
    }
  }
  {
    std::vector<int> zero(4, 0);
    const int* dst = nullptr;
    if ((st = upload(cb, zero, &dst)) != TQ_OK) {
      tq_free_codebook(cb);
      return st;
    }
    cb->d_status = const_cast<int*>(dst);
  }
  cudaDeviceGetAttribute(&cb->sms, cudaDevAttrMultiProcessorCount, cb->device);
  cb->tc_ready = false;
  // tensor maps of Pi_hi, Pi_lo and S for the tensor-core quantize kernels:
  // 64-column blocks of all d rows (d = 128: with extra-bit coordinates too;
  // d = 256: without; polar mode has none)
  if (d == 128 || D.extra == 0) {
    bool good = encode_bf16_rows(&cb->tm_pihi, dv.Pi_hi, d, d, d) && encode_bf16_rows(&cb->tm_pilo, dv.Pi_lo, d, d, d);
    if (D.kind == TQ_KIND_PROD) good = good && encode_bf16_rows(&cb->tm_s, dv.S_bf, D.m, d, d);
    else cb->tm_s = cb->tm_pihi;
    cb->tc_ready = good;
  }
  *out = cb;
  return ok();
}

tq_status tq_fail_allocation(int32_t nth) {
  if (nth < -1) return fail(TQ_EINVAL, "tq_fail_allocation: nth must be >= -1");
  g_fail_after = nth;
  return ok();
}

tq_status tq_set_first_wait_limit(tq_codebook* cb, int64_t polls) {
  if (!cb) return fail(TQ_EINVAL, "tq_set_first_wait_limit: NULL codebook");
  if (polls < -1) return fail(TQ_EINVAL, "tq_set_first_wait_limit: polls must be >= -1");
  cb->dev.first_wait = polls < 0 ? kDefaultWaitPolls : (long long)polls;
  return ok();
}

tq_status tq_check_device(const tq_codebook* cb) {
  const tq::NvtxRange nvtx_range("tq_check_device");
  if (!cb) return fail(TQ_EINVAL, "tq_check_device: NULL codebook");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(TQ_ECUDA, "tq_check_device: %s", cudaGetErrorString(e));
  int flag = 0;
  e = cudaMemcpy(&flag, cb->d_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(TQ_ECUDA, "tq_check_device: %s", cudaGetErrorString(e));
  if (flag) {
    const int zero = 0;
    cudaMemcpy(cb->d_status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (flag & ~tq::kBadRow)
      return fail(TQ_ETIMEOUT, "tq_check_device: a kernel's bounded wait on its copies or MMAs gave up");
    return fail(TQ_EINVAL, "tq_check_device: an append destination or a block-table entry lay outside the cache "
                           "(those writes were skipped; reads of such a page went to page 0)");
  }
  return ok();
}

void tq_free_codebook(tq_codebook* cb) {
  if (!cb) return;
  for (void* p : cb->allocs) cudaFree(p);
  delete cb;
}

tq_status tq_codebook_tables(const tq_codebook* cb, float* centroids, float* boundaries, double* pi, float* s) {
  if (!cb) return fail(TQ_EINVAL, "tq_codebook_tables: NULL codebook");
  if (centroids) std::memcpy(centroids, cb->cent.data(), cb->cent.size() * sizeof(float));
  if (boundaries) std::memcpy(boundaries, cb->bound.data(), cb->bound.size() * sizeof(float));
  if (pi) std::memcpy(pi, cb->pi.data(), cb->pi.size() * sizeof(double));
  if (s && !cb->s.empty()) std::memcpy(s, cb->s.data(), cb->s.size() * sizeof(float));
  return ok();
}

size_t tq_record_bytes(const tq_codebook* cb) { return cb ? (size_t)cb->dev.W * 4 : 0; }

size_t tq_cache_bytes(const tq_codebook* cb, int64_t rows) {
  if (!cb || rows < 0) return 0;
  return (size_t)(tq::norm_offset(cb->dev, rows) + rows * cb->dev.nb);
}

static tq_status quantize_common(const char* what, const tq_codebook* cb, void* cache, int64_t cache_rows,
                                 const void* x, int32_t x_dtype, int64_t n, int32_t d_in, const float* y,
                                 const float* norms, const int64_t* dst_rows, void* stream,
                                 const tq::AppendDst* paged = nullptr) {
  if (!cb) return fail(TQ_EINVAL, "%s: codebook is NULL", what);
  if (n < 0 || cache_rows < 0) return fail(TQ_EINVAL, "%s: negative size", what);
  if (n == 0) return ok();
  if (!cache || !aligned16(cache)) return fail(TQ_EINVAL, "%s: cache must be a 16-byte aligned device pointer", what);
  if (!dst_rows && !paged && n > cache_rows) return fail(TQ_EINVAL, "%s: n = %lld rows exceed cache_rows = %lld", what, (long long)n, (long long)cache_rows);
  if (!y) {
    if (!x) return fail(TQ_EINVAL, "%s: x is NULL", what);
    if (x_dtype != TQ_F32 && x_dtype != TQ_BF16) return fail(TQ_EINVAL, "%s: bad dtype %d", what, x_dtype);
    if (d_in < 1 || d_in > cb->dev.d) return fail(TQ_EINVAL, "%s: d_in = %d must be in 1..%d", what, d_in, cb->dev.d);
  } else if (!norms) {
    return fail(TQ_EINVAL, "%s: norms is NULL", what);
  }
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != cb->device) return fail(TQ_EINVAL, "%s: codebook lives on device %d, current device is %d", what, cb->device, dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // batches on the tensor cores with X in tensor memory: d = 256 (bf16 or
  // fp32) and d = 128 fp32 without extra-bit coordinates (either mode)
  const bool tcx = cb->dev.d == 256 || (x_dtype == TQ_F32 && cb->dev.extra == 0);
  if (!paged && !y && tcx && cb->tc_ready && n >= 2048 && d_in % (x_dtype == TQ_BF16 ? 8 : 4) == 0 &&
      aligned16(x) && n < (1ll << 31))
    return launched(what, tq::launch_quantize_tcx(cb->tm_pihi, cb->tm_pilo, cb->tm_s, cb->dev,
                                                  static_cast<uint8_t*>(cache), cache_rows, x, x_dtype == TQ_F32, n,
                                                  d_in, dst_rows, cb->d_status, cb->sms, s));
  // d = 128 bf16 batches (scalar or polar mode): tensor-core rotation and
  // sketch, X by TMA, two tile groups
  if (!paged && !y && cb->dev.d == 128 && x_dtype == TQ_BF16 && cb->tc_ready && n >= 2048 && d_in % 8 == 0 &&
      aligned16(x) && n < (1ll << 31)) {
    CUtensorMap tm_x;
    if (encode_bf16_rows(&tm_x, x, n, d_in))
      return launched(what, tq::launch_quantize_tc(tm_x, cb->tm_pihi, cb->tm_pilo, cb->tm_s, cb->dev,
                                                   static_cast<uint8_t*>(cache), cache_rows, n, dst_rows,
                                                   cb->d_status, cb->sms, s));
  }
  tq::AppendDst dst = {};
  dst.rows = dst_rows;
  if (paged) dst = *paged;
  return launched(what, tq::launch_quantize_simt(cb->dev, static_cast<uint8_t*>(cache), cache_rows, x, x_dtype, n,
                                                 d_in, y, norms, dst, cb->d_status, s));
}

tq_status tq_quantize(const tq_codebook* cb, void* cache, int64_t cache_rows, const void* x, int32_t x_dtype,
                      int64_t n, int32_t d_in, const int64_t* dst_rows, void* stream) {
  const tq::NvtxRange nvtx_range("tq_quantize");
  return quantize_common("tq_quantize", cb, cache, cache_rows, x, x_dtype, n, d_in, nullptr, nullptr, dst_rows,
                         stream);
}

tq_status tq_quantize_rotated(const tq_codebook* cb, void* cache, int64_t cache_rows, const float* y,
                              const float* norms, int64_t n, const int64_t* dst_rows, void* stream) {
  const tq::NvtxRange nvtx_range("tq_quantize_rotated");
  if (n > 0 && !y) return fail(TQ_EINVAL, "tq_quantize_rotated: y is NULL");
  return quantize_common("tq_quantize_rotated", cb, cache, cache_rows, nullptr, TQ_F32, n, cb ? cb->dev.d : 0, y,
                         norms, dst_rows, stream);
}

size_t tq_logits_workspace(const tq_codebook* kcb, int32_t B, int32_t Hq, int32_t Hkv) {
  (void)Hq;
  if (!kcb || B <= 0 || Hkv <= 0) return 0;
  return (size_t)tq::align256((int64_t)B * Hkv * tq::prep_block_bytes(kcb->dev.d));
}

static tq_status check_heads(const char* what, int32_t B, int32_t Hq, int32_t Hkv, int64_t capacity) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || capacity < 0) return fail(TQ_EINVAL, "%s: bad sizes", what);
  if (Hq % Hkv) return fail(TQ_EINVAL, "%s: Hq = %d is not a multiple of Hkv = %d", what, Hq, Hkv);
  const int G = Hq / Hkv;
  if (G > 4 && (G % 4 != 0 || G > 16))
    return fail(TQ_EUNSUPPORTED, "%s: a GQA group of %d query heads is not implemented (1..4, 8, 12 or 16)", what, G);
  if (B > 65535 || Hkv > 65535 || Hq > 65535) return fail(TQ_EINVAL, "%s: too many heads or sequences", what);
  return TQ_OK;
}

// A decode step's key append carried by the first query-prep launch (see
// tq_append_logits); n = 0: none.
struct FusedAppend {
  const void* x = nullptr;
  int32_t x_dtype = 0;
  int64_t n = 0;
  int32_t d_in = 0;
  const int64_t* dst_rows = nullptr;
};

static tq_status logits_common(const char* what, const tq_codebook* kcb, const void* kcache, int64_t rows,
                               const tq::RowMap& map, int32_t B, int32_t Hq, int32_t Hkv, int64_t capacity,
                               const int32_t* seq_lens, const float* q, float* logits, void* workspace,
                               size_t ws_bytes, void* stream, const FusedAppend& app = FusedAppend()) {
  tq_status st;
  // keys with the QJL term (PROD), or MSE-only keys in scalar mode
  if ((st = check_scoring_codebook(kcb, kcb && kcb->dev.kind == TQ_KIND_MSE ? TQ_KIND_MSE : TQ_KIND_PROD, what,
                                   true)) != TQ_OK)
    return st;
  if (kcb->dev.kind == TQ_KIND_MSE && kcb->dev.mode != TQ_MODE_SCALAR)
    return fail(TQ_EUNSUPPORTED, "%s: MSE-only keys are scored in scalar mode only", what);
  if ((st = check_heads(what, B, Hq, Hkv, capacity)) != TQ_OK) return st;
  if (capacity == 0) return ok();
  if (!kcache || !seq_lens || !q || !logits || !workspace) return fail(TQ_EINVAL, "%s: NULL device pointer", what);
  if (!aligned16(kcache) || !aligned16(q) || !aligned16(logits) || !aligned16(workspace))
    return fail(TQ_EINVAL, "%s: device pointers must be 16-byte aligned", what);
  if (ws_bytes < tq_logits_workspace(kcb, B, Hq, Hkv)) return fail(TQ_ENOMEM, "%s: workspace too small", what);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* prep = static_cast<uint8_t*>(workspace);
  int nchunks, tpc;
  // the polar kernel (72 registers, no shared-memory ring) hides its global
  // loads with more resident CTAs: 7 per SM
  chunking(B, Hkv, capacity, kcb->dev.mode == TQ_MODE_POLAR ? 148 * 7 : kLogitsCtas, &nchunks, &tpc);
  // The kernels score 4 query heads per kv head (fp16 hi / lo of each in
  // the 8 tensor-core columns); a larger group (a multiple of 4) is scored
  // 4 heads at a time: with Hq and Hkv unchanged, queries and logits offset
  // by 4 g heads address heads 4 g .. 4 g + 3 of every kv head.
  const int ngroups = (Hq / Hkv + 3) / 4;
  for (int g = 0; g < ngroups; ++g) {
    const float* qg = q + (size_t)4 * g * kcb->dev.d;
    float* lg = logits + (size_t)4 * g * capacity;
    if (kcb->dev.mode == TQ_MODE_POLAR) {
      if ((st = launched(what, tq::launch_prep_polar(kcb->dev, qg, B, Hq, Hkv, prep, s))) != TQ_OK) return st;
      st = launched(what, tq::launch_logits_polar(kcb->dev, static_cast<const uint8_t*>(kcache), B, Hq, Hkv,
                                                  capacity, rows, map, seq_lens, prep, lg, nchunks, tpc,
                                                  kcb->d_status, s));
    } else {
      if (g == 0 && app.n > 0)
        st = launched(what, tq::launch_prep_append(kcb->dev, qg, B, Hq, Hkv, prep,
                                                   static_cast<uint8_t*>(const_cast<void*>(kcache)), rows, app.x,
                                                   app.x_dtype, app.n, app.d_in, app.dst_rows, kcb->d_status, s));
      else
        st = launched(what, tq::launch_prep(kcb->dev, qg, B, Hq, Hkv, prep, s));
      if (st != TQ_OK) return st;
      if (capacity % 16 == 0)
        st = launched(what, tq::launch_logits_staged(kcb->dev, static_cast<const uint8_t*>(kcache), B, Hq, Hkv,
                                                     capacity, rows, map, seq_lens, prep, lg, nchunks, tpc,
                                                     kcb->d_status, s));
      else
        st = launched(what, tq::launch_logits(kcb->dev, static_cast<const uint8_t*>(kcache), B, Hq, Hkv, capacity,
                                              rows, seq_lens, prep, lg, nchunks, tpc, s));
    }
    if (st != TQ_OK) return st;
  }
  return ok();
}

tq_status tq_logits(const tq_codebook* kcb, const void* kcache, int32_t B, int32_t Hq, int32_t Hkv, int64_t capacity,
                    const int32_t* seq_lens, const float* q, float* logits, void* workspace, size_t ws_bytes,
                    void* stream) {
  const tq::NvtxRange nvtx_range("tq_logits");
  return logits_common("tq_logits", kcb, kcache, (int64_t)B * Hkv * capacity, tq::RowMap{}, B, Hq, Hkv, capacity,
                       seq_lens, q, logits, workspace, ws_bytes, stream);
}

tq_status tq_append_logits(const tq_codebook* kcb, void* kcache, const void* x, int32_t x_dtype, int64_t n,
                           int32_t d_in, const int64_t* dst_rows, int32_t B, int32_t Hq, int32_t Hkv, int64_t capacity,
                           const int32_t* seq_lens, const float* q, float* logits, void* workspace, size_t ws_bytes,
                           void* stream) {
  const tq::NvtxRange nvtx_range("tq_append_logits");
  const char* what = "tq_append_logits";
  if (!kcb) return fail(TQ_EINVAL, "%s: codebook is NULL", what);
  if (B <= 0 || Hkv <= 0 || capacity < 0) return fail(TQ_EINVAL, "%s: bad sizes", what);
  const int64_t rows = (int64_t)B * Hkv * capacity;
  const bool fuse = n >= 1 && n <= 4096 && kcb->dev.mode == TQ_MODE_SCALAR && kcb->dev.d == 128 &&
                    kcb->dev.extra == 0 && capacity > 0;
  if (!fuse) {
    tq_status st = quantize_common(what, kcb, kcache, rows, x, x_dtype, n, d_in, nullptr, nullptr, dst_rows, stream);
    if (st != TQ_OK) return st;
    return logits_common(what, kcb, kcache, rows, tq::RowMap{}, B, Hq, Hkv, capacity, seq_lens, q, logits, workspace,
                         ws_bytes, stream);
  }
  // the append's own checks (as tq_quantize), then the fused launch
  if (!kcache || !aligned16(kcache)) return fail(TQ_EINVAL, "%s: cache must be a 16-byte aligned device pointer", what);
  if (!x) return fail(TQ_EINVAL, "%s: x is NULL", what);
  if (x_dtype != TQ_F32 && x_dtype != TQ_BF16) return fail(TQ_EINVAL, "%s: bad dtype %d", what, x_dtype);
  if (d_in < 1 || d_in > kcb->dev.d) return fail(TQ_EINVAL, "%s: d_in = %d must be in 1..%d", what, d_in, kcb->dev.d);
  if (!dst_rows && n > rows) return fail(TQ_EINVAL, "%s: n = %lld rows exceed the cache", what, (long long)n);
  FusedAppend app;
  app.x = x;
  app.x_dtype = x_dtype;
  app.n = n;
  app.d_in = d_in;
  app.dst_rows = dst_rows;
  return logits_common(what, kcb, kcache, rows, tq::RowMap{}, B, Hq, Hkv, capacity, seq_lens, q, logits, workspace,
                       ws_bytes, stream, app);
}

// Paged layout arguments shared by the *_paged entry points.
static tq_status check_paged(const char* what, int32_t num_pages, int32_t page_size, const int32_t* block_table,
                             int32_t max_pages, int32_t Hkv, tq::RowMap* map) {
  if (!block_table) return fail(TQ_EINVAL, "%s: block_table is NULL", what);
  if (page_size < 16 || page_size % 16 || page_size > (1 << 20))
    return fail(TQ_EINVAL, "%s: page_size = %d must be a positive multiple of 16 (at most 2^20)", what, page_size);
  if (num_pages < 1 || max_pages < 1) return fail(TQ_EINVAL, "%s: num_pages and max_pages must be positive", what);
  if (Hkv < 1 || (int64_t)num_pages * Hkv * page_size >= (1ll << 40))
    return fail(TQ_EINVAL, "%s: cache too large", what);
  if ((int64_t)max_pages * page_size >= (1ll << 31))
    return fail(TQ_EINVAL, "%s: max_pages * page_size must be below 2^31 tokens", what);
  map->table = block_table;
  map->page = page_size;
  map->max_pages = max_pages;
  map->num_pages = num_pages;
  map->page_shift = -1;
  for (int k = 4; k <= 20; ++k)
    if (page_size == (1 << k)) map->page_shift = k;
  return TQ_OK;
}

tq_status tq_logits_paged(const tq_codebook* kcb, const void* kcache, int32_t num_pages, int32_t page_size,
                          const int32_t* block_table, int32_t max_pages, int32_t B, int32_t Hq, int32_t Hkv,
                          const int32_t* seq_lens, const float* q, float* logits, void* workspace, size_t ws_bytes,
                          void* stream) {
  const tq::NvtxRange nvtx_range("tq_logits_paged");
  tq::RowMap map;
  tq_status st = check_paged("tq_logits_paged", num_pages, page_size, block_table, max_pages, Hkv, &map);
  if (st != TQ_OK) return st;
  return logits_common("tq_logits_paged", kcb, kcache, (int64_t)num_pages * Hkv * page_size, map, B, Hq, Hkv,
                       (int64_t)max_pages * page_size, seq_lens, q, logits, workspace, ws_bytes, stream);
}

tq_status tq_append_paged(const tq_codebook* cb, void* cache, int32_t num_pages, int32_t page_size,
                          const int32_t* block_table, int32_t max_pages, int32_t B, int32_t Hkv,
                          const int32_t* seq_lens, const void* x, int32_t x_dtype, int32_t d_in, void* stream) {
  const tq::NvtxRange nvtx_range("tq_append_paged");
  tq::AppendDst dst = {};
  tq_status st = check_paged("tq_append_paged", num_pages, page_size, block_table, max_pages, Hkv, &dst.map);
  if (st != TQ_OK) return st;
  if (!cb) return fail(TQ_EINVAL, "tq_append_paged: codebook is NULL");
  if (B < 1 || B > 65535) return fail(TQ_EINVAL, "tq_append_paged: bad B = %d", B);
  if (!seq_lens) return fail(TQ_EINVAL, "tq_append_paged: seq_lens is NULL");
  dst.seq_lens = seq_lens;
  dst.Hkv = Hkv;
  return quantize_common("tq_append_paged", cb, cache, (int64_t)num_pages * Hkv * page_size, x, x_dtype,
                         (int64_t)B * Hkv, d_in, nullptr, nullptr, nullptr, stream, &dst);
}

tq_status tq_advance_lengths(int32_t* seq_lens, int32_t B, int32_t delta, void* stream) {
  const tq::NvtxRange nvtx_range("tq_advance_lengths");
  if (!seq_lens || B < 1) return fail(TQ_EINVAL, "tq_advance_lengths: bad arguments");
  return launched("tq_advance_lengths", tq::launch_advance_lengths(seq_lens, B, delta, static_cast<cudaStream_t>(stream)));
}

// Split of the context of a decode-attention launch and the workspace it
// writes: the query fragments, then one partial per (sequence, kv head,
// chunk, warp).  The launch and every workspace bound use this one helper;
// without a value codebook it gives the largest split any value codebook
// can get (a value codebook only ever lowers the resident-CTA target).
// Groups of more than 4 query heads per kv head keep one partial region per
// 4-head group (group_stride floats apart).
static int64_t attn_workspace_bytes(const tq_codebook* kcb, const tq_codebook* vcb, int32_t B, int32_t Hq,
                                    int32_t Hkv, int64_t capacity, int* nchunks_out = nullptr,
                                    int* tpc_out = nullptr, int64_t* group_stride_out = nullptr) {
  int nchunks, tpc;
  chunking(B, Hkv, capacity, attn_ctas(kcb, vcb), &nchunks, &tpc);
  if (nchunks_out) *nchunks_out = nchunks;
  if (tpc_out) *tpc_out = tpc;
  const int64_t ngroups = (Hq / std::max(Hkv, 1) + 3) / 4;
  const int64_t prep = tq::align256((int64_t)B * Hkv * tq::prep_block_bytes(kcb->dev.d));
  const int64_t stride = (int64_t)B * Hkv * nchunks * tq::kAttnWarps * tq::partial_floats(kcb->dev.d);
  if (group_stride_out) *group_stride_out = stride;
  return prep + std::max<int64_t>(1, ngroups) * stride * 4;
}

size_t tq_decode_attention_workspace(const tq_codebook* kcb, int32_t B, int32_t Hq, int32_t Hkv, int64_t capacity) {
  if (!kcb || B <= 0 || Hkv <= 0 || Hq <= 0 || capacity < 0) return 0;
  return (size_t)attn_workspace_bytes(kcb, nullptr, B, Hq, Hkv, capacity);
}

static tq_status attn_common(const char* what, const tq_codebook* kcb, const tq_codebook* vcb, const void* kcache,
                             const void* vcache, int64_t rows, const tq::RowMap& map, int32_t B, int32_t Hq,
                             int32_t Hkv, int64_t capacity, const int32_t* seq_lens, const float* q, float scale,
                             float* out, void* workspace, size_t ws_bytes, void* stream) {
  tq_status st;
  // keys: with the QJL term (PROD, 2.5 / 3.5-bit mixed included) or MSE-only
  if ((st = check_scoring_codebook(kcb, kcb && kcb->dev.kind == TQ_KIND_MSE ? TQ_KIND_MSE : TQ_KIND_PROD,
                                   "tq_decode_attention(keys)", true)) != TQ_OK)
    return st;
  // values: MSE kind; mixed-bit (an extra bit on d/4 coordinates) in scalar mode
  const bool mixed_values = vcb && vcb->dev.extra != 0;
  if (mixed_values) {
    if (vcb->dev.kind != TQ_KIND_MSE) return fail(TQ_EINVAL, "%s: the value codebook must be of kind MSE", what);
  } else if ((st = check_scoring_codebook(vcb, TQ_KIND_MSE, "tq_decode_attention(values)")) != TQ_OK) {
    return st;
  }
  if (kcb->dev.kind == TQ_KIND_MSE || kcb->dev.extra != 0 || mixed_values) {
    if (kcb->dev.mode != TQ_MODE_SCALAR || vcb->dev.mode != TQ_MODE_SCALAR)
      return fail(TQ_EUNSUPPORTED, "%s: MSE-only and mixed-bit caches are attended in scalar mode only", what);
    if (!tq::attn_staged_supports(kcb->dev, vcb->dev))
      return fail(TQ_EUNSUPPORTED,
                  "%s: this key/value pair is not implemented (MSE-only or mixed-bit keys take 3- or 4-bit values; "
                  "mixed-bit values take 2 or 3 bits, extra = d/4, with keys that have the QJL term)",
                  what);
    if (capacity % 16 != 0 && !map.table)
      return fail(TQ_EUNSUPPORTED, "%s: MSE-only and mixed-bit caches need a capacity that is a multiple of 16", what);
    int dev = -1;
    cudaGetDevice(&dev);
    if (dev != vcb->device) return fail(TQ_EINVAL, "%s: value codebook lives on another device", what);
  }
  if ((st = check_heads(what, B, Hq, Hkv, capacity)) != TQ_OK) return st;
  if (!kcache || !vcache || !seq_lens || !q || !out || !workspace)
    return fail(TQ_EINVAL, "%s: NULL device pointer", what);
  if (!aligned16(kcache) || !aligned16(vcache) || !aligned16(q) || !aligned16(out) || !aligned16(workspace))
    return fail(TQ_EINVAL, "%s: device pointers must be 16-byte aligned", what);
  if (!std::isfinite(scale)) return fail(TQ_EINVAL, "%s: scale must be finite", what);
  int nchunks, tpc;
  int64_t gstride;
  if (ws_bytes < (size_t)attn_workspace_bytes(kcb, vcb, B, Hq, Hkv, capacity, &nchunks, &tpc, &gstride))
    return fail(TQ_ENOMEM, "%s: workspace too small", what);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* prep = static_cast<uint8_t*>(workspace);
  float* parts = reinterpret_cast<float*>(
      prep + tq::align256((int64_t)B * Hkv * tq::prep_block_bytes(kcb->dev.d)));
  if (kcb->dev.mode != vcb->dev.mode)
    return fail(TQ_EUNSUPPORTED, "%s: keys and values must use the same stage-1 mode", what);
  const float sl2 = scale * 1.4426950408889634f;
  // 4 query heads per kv head per launch (see logits_common); head group g
  // writes its partials gstride floats after group g - 1's
  const int ngroups = (Hq / Hkv + 3) / 4;
  for (int g = 0; g < ngroups; ++g) {
    const float* qg = q + (size_t)4 * g * kcb->dev.d;
    float* pg = parts + (size_t)g * gstride;
    if (kcb->dev.mode == TQ_MODE_POLAR) {
      if ((st = launched("tq_decode_attention/prep", tq::launch_prep_polar(kcb->dev, qg, B, Hq, Hkv, prep, s))) !=
          TQ_OK)
        return st;
      if (capacity % 16 == 0 || map.table)
        st = launched("tq_decode_attention",
                      tq::launch_attn_polar_staged(kcb->dev, vcb->dev, static_cast<const uint8_t*>(kcache),
                                                   static_cast<const uint8_t*>(vcache), B, Hq, Hkv, capacity, rows,
                                                   map, seq_lens, prep, sl2, pg, nchunks, tpc, kcb->d_status, s));
      else
        st = launched("tq_decode_attention",
                      tq::launch_attn_polar(kcb->dev, vcb->dev, static_cast<const uint8_t*>(kcache),
                                            static_cast<const uint8_t*>(vcache), B, Hq, Hkv, capacity, rows,
                                            seq_lens, prep, sl2, pg, nchunks, tpc, s));
    } else {
      if ((st = launched("tq_decode_attention/prep", tq::launch_prep(kcb->dev, qg, B, Hq, Hkv, prep, s))) != TQ_OK)
        return st;
      if (capacity % 16 == 0 || map.table)
        st = launched("tq_decode_attention",
                      tq::launch_attn_staged(kcb->dev, vcb->dev, static_cast<const uint8_t*>(kcache),
                                             static_cast<const uint8_t*>(vcache), B, Hq, Hkv, capacity, rows, map,
                                             seq_lens, prep, sl2, pg, nchunks, tpc, kcb->d_status, s));
      else
        st = launched("tq_decode_attention",
                      tq::launch_attn(kcb->dev, vcb->dev, static_cast<const uint8_t*>(kcache),
                                      static_cast<const uint8_t*>(vcache), B, Hq, Hkv, capacity, rows, seq_lens,
                                      prep, sl2, pg, nchunks, tpc, s));
    }
    if (st != TQ_OK) return st;
  }
  return launched("tq_decode_attention/merge",
                  tq::launch_attn_merge(vcb->dev, parts, B, Hq, Hkv, nchunks * tq::kAttnWarps, gstride, out, s));
}

tq_status tq_decode_attention(const tq_codebook* kcb, const tq_codebook* vcb, const void* kcache, const void* vcache,
                              int32_t B, int32_t Hq, int32_t Hkv, int64_t capacity, const int32_t* seq_lens,
                              const float* q, float scale, float* out, void* workspace, size_t ws_bytes,
                              void* stream) {
  const tq::NvtxRange nvtx_range("tq_decode_attention");
  return attn_common("tq_decode_attention", kcb, vcb, kcache, vcache, (int64_t)B * Hkv * capacity, tq::RowMap{}, B,
                     Hq, Hkv, capacity, seq_lens, q, scale, out, workspace, ws_bytes, stream);
}

tq_status tq_decode_attention_paged(const tq_codebook* kcb, const tq_codebook* vcb, const void* kcache,
                                    const void* vcache, int32_t num_pages, int32_t page_size,
                                    const int32_t* block_table, int32_t max_pages, int32_t B, int32_t Hq,
                                    int32_t Hkv, const int32_t* seq_lens, const float* q, float scale, float* out,
                                    void* workspace, size_t ws_bytes, void* stream) {
  const tq::NvtxRange nvtx_range("tq_decode_attention_paged");
  tq::RowMap map;
  tq_status st = check_paged("tq_decode_attention_paged", num_pages, page_size, block_table, max_pages, Hkv, &map);
  if (st != TQ_OK) return st;
  return attn_common("tq_decode_attention_paged", kcb, vcb, kcache, vcache, (int64_t)num_pages * Hkv * page_size,
                     map, B, Hq, Hkv, (int64_t)max_pages * page_size, seq_lens, q, scale, out, workspace, ws_bytes,
                     stream);
}

size_t tq_search_workspace(const tq_codebook* cb, int64_t n_db, int32_t nq, int32_t k) {
  if (!cb || nq <= 0 || n_db <= 0 || k < 1) return 0;
  if (tq::search_tc_applies(cb->dev, k)) return (size_t)tq::search_tc_workspace_bytes(cb->dev, n_db, nq, k, cb->sms);
  return (size_t)tq::search_workspace_bytes(cb->dev, n_db, nq, k, cb->sms);
}

tq_status tq_search(const tq_codebook* cb, const void* db_cache, int64_t n_db, const float* q, int32_t nq,
                    int32_t d_in, int32_t k, int32_t* ids, float* scores, void* workspace, size_t ws_bytes,
                    void* stream) {
  const tq::NvtxRange nvtx_range("tq_search");
  if (!cb) return fail(TQ_EINVAL, "tq_search: codebook is NULL");
  if (cb->dev.kind != TQ_KIND_PROD) return fail(TQ_EINVAL, "tq_search: the database codebook must be of kind PROD");
  if (cb->dev.mode != TQ_MODE_SCALAR || cb->dev.extra != 0)
    return fail(TQ_EUNSUPPORTED, "tq_search: only scalar-mode databases without extra bits are searched");
  if (cb->dev.d != 256) return fail(TQ_EUNSUPPORTED, "tq_search: only d = 256 is implemented");
  if (n_db <= 0 || n_db >= (1ll << 31) || nq <= 0 || d_in < 1 || d_in > cb->dev.d || k < 1 || k > 32)
    return fail(TQ_EINVAL, "tq_search: bad sizes (n_db %lld, nq %d, d_in %d, k %d; k must be 1..32)",
                (long long)n_db, nq, d_in, k);
  if (!db_cache || !q || !ids || !scores || !workspace) return fail(TQ_EINVAL, "tq_search: NULL device pointer");
  if (!aligned16(db_cache) || !aligned16(workspace)) return fail(TQ_EINVAL, "tq_search: buffers must be 16-byte aligned");
  if (ws_bytes < tq_search_workspace(cb, n_db, nq, k)) return fail(TQ_ENOMEM, "tq_search: workspace too small");
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != cb->device) return fail(TQ_EINVAL, "tq_search: codebook lives on another device");
  if (tq::search_tc_applies(cb->dev, k))
    return launched("tq_search", tq::launch_search_tc(cb->dev, static_cast<const uint8_t*>(db_cache), n_db, q, nq, d_in,
                                                      k, ids, scores, static_cast<uint8_t*>(workspace), cb->sms,
                                                      cb->d_status, static_cast<cudaStream_t>(stream)));
  return launched("tq_search", tq::launch_search(cb->dev, static_cast<const uint8_t*>(db_cache), n_db, q, nq, d_in, k,
                                                ids, scores, static_cast<uint8_t*>(workspace), cb->sms,
                                                static_cast<cudaStream_t>(stream)));
}

tq_status tq_search_fallbacks(const tq_codebook* cb, const void* workspace, int32_t k, int32_t* count) {
  if (!cb || !workspace || !count) return fail(TQ_EINVAL, "tq_search_fallbacks: NULL argument");
  if (!tq::search_tc_applies(cb->dev, k)) {
    *count = -1;
    return ok();
  }
  cudaError_t e = cudaDeviceSynchronize();
  unsigned v = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&v, static_cast<const unsigned*>(workspace) + 2, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(TQ_ECUDA, "tq_search_fallbacks: %s", cudaGetErrorString(e));
  *count = (int32_t)v;
  return ok();
}

}  // extern "C"
