// Host-side setup mathematics of a codebook (C++17, fp64, libm only).
#pragma once
#include <cstddef>
#include <cstdint>
#include <vector>

namespace tqm {

// k-th output of the splitmix64 stream seeded with `seed` (Vigna's generator).
uint64_t splitmix64(uint64_t seed, uint64_t k);

// First `count` N(0,1) draws of stream `seed` (Box-Muller on output pairs).
std::vector<double> gaussians(uint64_t seed, size_t count);

// Round to fp32 then to bfloat16, both to nearest even.
float round_bf16(double v);

// Haar rotation: Householder QR of the seeded Gaussian matrix, Q * diag(sign(diag R)).
std::vector<double> haar_rotation(int d, uint64_t seed);

// Lloyd-Max tables with L cells (centroids L, interior boundaries L-1).
struct Quantizer {
  std::vector<double> c, t;
};
// Law of one coordinate of a uniform point on S^{d-1} (Beta((d-1)/2, (d-1)/2) on [-1, 1]).
Quantizer lloyd_max_beta(int d, int L);
// Polar angle between two child radii gathering k coordinates each: density
// proportional to sin^(k-1)(2 psi) on [0, pi/2].
Quantizer lloyd_max_polar(int k, int L);

}  // namespace tqm
