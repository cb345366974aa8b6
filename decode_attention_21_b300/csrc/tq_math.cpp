// Host-side setup mathematics of a codebook: generator, Haar rotation and
// Lloyd-Max solver.  Plain C++17 in fp64; nothing here runs per vector.
//
// Rotation: [suzuke] "TurboQuant: compressing AI consciousness", 第一步 -- a
// random orthogonal matrix makes every coordinate ~N(0, 1/d); [xujun]
// note-189244, 第一步 -- the law is a concentrated Beta distribution.
// Codebooks: [suzuke] 第二步 -- each value is coded with the Max-Lloyd
// algorithm on its known law.
#include "tq_math.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <stdexcept>
#include <utility>

namespace tqm {

uint64_t splitmix64(uint64_t seed, uint64_t k) {
  uint64_t z = seed + (k + 1) * 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

std::vector<double> gaussians(uint64_t seed, size_t count) {
  std::vector<double> out(count + 1);
  const double two53 = 1.0 / 9007199254740992.0;  // 2^-53
  for (size_t pair = 0; 2 * pair < count; ++pair) {
    const double u1 = (double)((splitmix64(seed, 2 * pair) >> 11) + 1) * two53;  // (0, 1]
    const double u2 = (double)(splitmix64(seed, 2 * pair + 1) >> 11) * two53;    // [0, 1)
    const double r = std::sqrt(-2.0 * std::log(u1));
    const double a = 2.0 * M_PI * u2;
    out[2 * pair] = r * std::cos(a);
    out[2 * pair + 1] = r * std::sin(a);
  }
  out.resize(count);
  return out;
}

float round_bf16(double v) {
  float f = (float)v;
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
  std::memcpy(&f, &u, 4);
  return f;
}

std::vector<double> haar_rotation(int d, uint64_t seed) {
  std::vector<double> A = gaussians(seed, (size_t)d * d);  // row-major G
  std::vector<std::vector<double>> refl(d);
  std::vector<double> rdiag(d);
  for (int k = 0; k < d; ++k) {
    double nrm = 0.0;
    for (int i = k; i < d; ++i) nrm += A[(size_t)i * d + k] * A[(size_t)i * d + k];
    nrm = std::sqrt(nrm);
    const double akk = A[(size_t)k * d + k];
    const double alpha = akk > 0 ? -nrm : nrm;
    std::vector<double> v(d - k);
    for (int i = k; i < d; ++i) v[i - k] = A[(size_t)i * d + k];
    v[0] -= alpha;
    double vn2 = 0.0;
    for (double e : v) vn2 += e * e;
    if (vn2 > 0.0) {
      for (int j = k; j < d; ++j) {
        double s = 0.0;
        for (int i = k; i < d; ++i) s += v[i - k] * A[(size_t)i * d + j];
        s *= 2.0 / vn2;
        for (int i = k; i < d; ++i) A[(size_t)i * d + j] -= s * v[i - k];
      }
    } else {
      v.assign(d - k, 0.0);
    }
    rdiag[k] = A[(size_t)k * d + k];
    refl[k] = std::move(v);
  }
  // Q = H_0 H_1 ... H_{d-1}: apply the reflectors to the identity, last first.
  std::vector<double> Q((size_t)d * d, 0.0);
  for (int i = 0; i < d; ++i) Q[(size_t)i * d + i] = 1.0;
  for (int k = d - 1; k >= 0; --k) {
    const std::vector<double>& v = refl[k];
    double vn2 = 0.0;
    for (double e : v) vn2 += e * e;
    if (vn2 == 0.0) continue;
    for (int j = 0; j < d; ++j) {
      double s = 0.0;
      for (int i = k; i < d; ++i) s += v[i - k] * Q[(size_t)i * d + j];
      s *= 2.0 / vn2;
      for (int i = k; i < d; ++i) Q[(size_t)i * d + j] -= s * v[i - k];
    }
  }
  for (int j = 0; j < d; ++j) {
    if (rdiag[j] < 0.0)
      for (int i = 0; i < d; ++i) Q[(size_t)i * d + j] = -Q[(size_t)i * d + j];
  }
  return Q;
}

// ------------------------------------------------------------- quadrature
namespace {

struct GaussLegendre {
  std::vector<double> x, w;
  explicit GaussLegendre(int n) : x(n), w(n) {
    // Newton iteration on the Legendre polynomial P_n from Chebyshev-like guesses.
    for (int i = 0; i < n; ++i) {
      double z = std::cos(M_PI * (i + 0.75) / (n + 0.5));
      double dp = 0.0;
      for (int it = 0; it < 100; ++it) {
        double p0 = 1.0, p1 = z;
        for (int k = 2; k <= n; ++k) {
          const double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
          p0 = p1;
          p1 = p2;
        }
        dp = n * (z * p1 - p0) / (z * z - 1.0);
        const double dz = p1 / dp;
        z -= dz;
        if (std::fabs(dz) < 1e-16) break;
      }
      {
        double p0 = 1.0, p1 = z;
        for (int k = 2; k <= n; ++k) {
          const double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
          p0 = p1;
          p1 = p2;
        }
        dp = n * (z * p1 - p0) / (z * z - 1.0);
      }
      x[i] = z;
      w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
    }
  }
};

const GaussLegendre& gl() {
  static const GaussLegendre g(160);
  return g;
}

// (integral of f, integral of t f) over [a, b]
template <class F>
std::pair<double, double> moments(const F& f, double a, double b) {
  const GaussLegendre& g = gl();
  const double h = 0.5 * (b - a), mid = 0.5 * (a + b);
  double p = 0.0, m = 0.0;
  for (size_t i = 0; i < g.x.size(); ++i) {
    const double t = mid + h * g.x[i];
    const double v = g.w[i] * f(t);
    p += v;
    m += v * t;
  }
  return {h * p, h * m};
}

template <class F>
Quantizer lloyd(const F& f, double lo, double hi, int L) {
  Quantizer q;
  q.c.assign(L, 0.0);
  if (L == 1) {
    auto pm = moments(f, lo, hi);
    q.c[0] = pm.second / pm.first;
    return q;
  }
  // equal-probability start from a cumulative table
  const int NG = 4096;
  std::vector<double> cdf(NG + 1, 0.0);
  for (int i = 0; i < NG; ++i)
    cdf[i + 1] = cdf[i] + moments(f, lo + (hi - lo) * i / NG, lo + (hi - lo) * (i + 1) / NG).first;
  q.t.assign(L - 1, 0.0);
  for (int k = 1; k < L; ++k) {
    const double target = cdf[NG] * k / L;
    int i = 0;
    while (i < NG - 1 && cdf[i + 1] < target) ++i;
    const double fr = (target - cdf[i]) / std::max(cdf[i + 1] - cdf[i], 1e-300);
    q.t[k - 1] = lo + (hi - lo) * (i + fr) / NG;
  }
  std::vector<double> edges(L + 1);
  double best = 1e300;
  int since = 0;
  for (int it = 0; it < 400000; ++it) {
    edges[0] = lo;
    edges[L] = hi;
    for (int k = 0; k < L - 1; ++k) edges[k + 1] = q.t[k];
    for (int k = 0; k < L; ++k) {
      auto pm = moments(f, edges[k], edges[k + 1]);
      q.c[k] = pm.second / pm.first;
    }
    double moved = 0.0;
    for (int k = 0; k < L - 1; ++k) {
      const double nt = 0.5 * (q.c[k] + q.c[k + 1]);
      moved = std::max(moved, std::fabs(nt - q.t[k]));
      q.t[k] = nt;
    }
    if (moved < 1e-15) break;
    if (moved < 0.5 * best) {
      best = moved;
      since = 0;
    } else if (++since > 2000 && best < 1e-13) {
      break;
    }
  }
  edges[0] = lo;
  edges[L] = hi;
  for (int k = 0; k < L - 1; ++k) edges[k + 1] = q.t[k];
  for (int k = 0; k < L; ++k) {
    auto pm = moments(f, edges[k], edges[k + 1]);
    q.c[k] = pm.second / pm.first;
  }
  return q;
}

std::mutex g_cache_mu;
std::map<std::pair<int, int>, Quantizer> g_beta_cache, g_polar_cache;

}  // namespace

Quantizer lloyd_max_beta(int d, int L) {
  {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    auto it = g_beta_cache.find({d, L});
    if (it != g_beta_cache.end()) return it->second;
  }
  const double e = 0.5 * (d - 3);
  Quantizer q = lloyd([e](double t) { return std::pow(std::max(0.0, 1.0 - t * t), e); }, -1.0, 1.0, L);
  // the law is symmetric: average with the mirror image to remove round-off
  Quantizer s = q;
  for (int k = 0; k < L; ++k) s.c[k] = 0.5 * (q.c[k] - q.c[L - 1 - k]);
  for (int k = 0; k < L - 1; ++k) s.t[k] = 0.5 * (q.t[k] - q.t[L - 2 - k]);
  std::lock_guard<std::mutex> lk(g_cache_mu);
  g_beta_cache[{d, L}] = s;
  return s;
}

Quantizer lloyd_max_polar(int k, int L) {
  {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    auto it = g_polar_cache.find({k, L});
    if (it != g_polar_cache.end()) return it->second;
  }
  const double e = k - 1.0;
  Quantizer q = lloyd([e](double p) { return e == 0.0 ? 1.0 : std::pow(std::sin(2.0 * p), e); }, 0.0, 0.5 * M_PI, L);
  std::lock_guard<std::mutex> lk(g_cache_mu);
  g_polar_cache[{k, L}] = q;
  return q;
}

}  // namespace tqm
