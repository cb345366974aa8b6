"""Lloyd-Max ("Max-Lloyd") scalar codebooks on known densities (oracle side).

[suzuke] 第二步: each angle is coded with the Max-Lloyd algorithm at b-1 bits;
[xujun] 第一步: after the random rotation every coordinate follows a highly
concentrated Beta law, and the angle laws are known, so no per-block
normalisation constants are stored.

A Lloyd-Max quantizer with L cells on a density f alternates the two optimality
conditions until they hold together:

* nearest-neighbour: every interior boundary is the midpoint of its two
  neighbouring centroids, ``t_k = (c_{k-1} + c_k) / 2``;
* centroid: every reproduction value is the conditional mean of its cell,
  ``c_k = int_{t_k}^{t_{k+1}} t f(t) dt / int_{t_k}^{t_{k+1}} f(t) dt``.

Densities used here:

* Beta_d (scalar mode): a fixed coordinate t of a uniform point on S^{d-1} has
  ``f_d(t) = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)) * (1 - t^2)^((d-3)/2)`` on
  [-1, 1], i.e. (t+1)/2 ~ Beta((d-1)/2, (d-1)/2).  Its CDF is the regularised
  incomplete beta function and ``int t f_d = -C_d (1-t^2)^((d-1)/2) / (d-1)``.
  N(0, 1/d) ([suzuke] 第一步) is its large-d limit.
* N(0,1): used only to pin the solver to Max's published table.
* uniform on [0, 2 pi): first-level polar angle.
* ``f(psi) ∝ sin^(k-1)(2 psi)`` on [0, pi/2]: polar angle between two child
  radii that each gather k coordinates (cos^2 psi ~ Beta(k/2, k/2)).
"""
import functools
import math

import numpy as np
from scipy import integrate, special


class BetaCoord:
    """Law of one coordinate of a uniform point on S^{d-1}."""

    def __init__(self, d):
        self.d = d
        self.a = (d - 1) / 2.0
        self.lo, self.hi = -1.0, 1.0
        self.C = math.exp(special.gammaln(d / 2.0) - special.gammaln((d - 1) / 2.0)) / math.sqrt(math.pi)
        self.second_moment = 1.0 / d

    def pdf(self, t):
        return self.C * (1.0 - t * t) ** ((self.d - 3) / 2.0)

    def cdf(self, t):
        return special.betainc(self.a, self.a, (np.clip(t, -1.0, 1.0) + 1.0) / 2.0)

    def pmoment(self, a, b):
        """int_a^b t f(t) dt (closed form)."""
        e = (self.d - 1) / 2.0
        return self.C / (self.d - 1) * ((1.0 - a * a) ** e - (1.0 - b * b) ** e)

    def quantile(self, p):
        return 2.0 * special.betaincinv(self.a, self.a, p) - 1.0


class Gaussian:
    """N(0, 1) on the real line (used to pin the solver)."""

    lo, hi = -math.inf, math.inf
    second_moment = 1.0

    def pdf(self, t):
        return np.exp(-0.5 * t * t) / math.sqrt(2.0 * math.pi)

    def cdf(self, t):
        return special.ndtr(t)

    def pmoment(self, a, b):
        return self.pdf(a) - self.pdf(b)

    def quantile(self, p):
        return special.ndtri(p)


class Uniform:
    def __init__(self, lo, hi):
        self.lo, self.hi = lo, hi
        self.second_moment = (hi ** 3 - lo ** 3) / (3.0 * (hi - lo))

    def pdf(self, t):
        return np.where((t >= self.lo) & (t <= self.hi), 1.0 / (self.hi - self.lo), 0.0)

    def cdf(self, t):
        return np.clip((t - self.lo) / (self.hi - self.lo), 0.0, 1.0)

    def pmoment(self, a, b):
        return (b * b - a * a) / (2.0 * (self.hi - self.lo))

    def quantile(self, p):
        return self.lo + p * (self.hi - self.lo)


_GL = np.polynomial.legendre.leggauss(160)


class PolarAngle:
    """psi = atan(rho_b / rho_a) where each child radius gathers k coordinates.

    cos^2 psi ~ Beta(k/2, k/2), hence f(psi) ∝ sin^(k-1)(2 psi) on [0, pi/2].
    """

    def __init__(self, k):
        self.k = k
        self.lo, self.hi = 0.0, math.pi / 2.0
        h = k / 2.0
        # normaliser: int_0^{pi/2} sin^(k-1)(2psi) dpsi = 2^(k-2) B(k/2, k/2)
        self.Z = math.exp((k - 2) * math.log(2.0) + special.betaln(h, h))

    def pdf(self, p):
        return np.sin(2.0 * p) ** (self.k - 1) / self.Z

    def cdf(self, p):
        p = np.clip(p, 0.0, math.pi / 2.0)
        return special.betainc(self.k / 2.0, self.k / 2.0, np.sin(p) ** 2)

    def pmoment(self, a, b):
        # Gauss-Legendre on [a, b]: the integrand is smooth and cells are short
        x, w = _GL
        h = 0.5 * (b - a)
        p = a + h * (x + 1.0)
        return h * float(np.dot(w, p * self.pdf(p)))

    def quantile(self, p):
        return math.asin(math.sqrt(special.betaincinv(self.k / 2.0, self.k / 2.0, p)))


def lloyd_max(dens, L, tol=1e-15, max_iter=400000):
    """Solve the L-level Lloyd-Max quantizer of ``dens``.

    Returns (centroids[L], boundaries[L-1], iterations).  Starts from the
    equal-probability partition and alternates the centroid and midpoint
    conditions until no value moves by more than ``tol`` (in the units of t),
    or until the step has stopped shrinking for 2000 iterations (round-off
    floor, far below 1e-12).
    """
    if L == 1:
        c = dens.pmoment(dens.lo, dens.hi) / 1.0
        return np.array([c]), np.zeros(0), 0
    t = np.array([dens.quantile(k / L) for k in range(1, L)], dtype=np.float64)
    c = np.zeros(L)
    it = 0
    best, since = math.inf, 0
    for it in range(1, max_iter + 1):
        edges = np.concatenate(([dens.lo], t, [dens.hi]))
        F = dens.cdf(edges)
        for k in range(L):
            c[k] = dens.pmoment(edges[k], edges[k + 1]) / (F[k + 1] - F[k])
        t_new = 0.5 * (c[:-1] + c[1:])
        moved = np.max(np.abs(t_new - t))
        t = t_new
        if moved < tol:
            break
        if moved < 0.5 * best:
            best, since = moved, 0
        else:
            since += 1
            if since > 2000 and best < 1e-13:
                break
    edges = np.concatenate(([dens.lo], t, [dens.hi]))
    F = dens.cdf(edges)
    for k in range(L):
        c[k] = dens.pmoment(edges[k], edges[k + 1]) / (F[k + 1] - F[k])
    return c.copy(), t.copy(), it


def distortion(dens, c, t):
    """E[(X - Q(X))^2] for the quantizer (c, t), by adaptive quadrature."""
    edges = np.concatenate(([dens.lo], t, [dens.hi]))
    tot = 0.0
    for k in range(len(c)):
        a, b = edges[k], edges[k + 1]
        tot += integrate.quad(lambda x: (x - c[k]) ** 2 * dens.pdf(x), a, b, epsabs=1e-17, epsrel=1e-13, limit=400)[0]
    return tot


def symmetrize(c, t):
    """Average a codebook of a symmetric density with its mirror image (removes
    round-off asymmetry so that c[k] == -c[L-1-k] and t[k] == -t[L-2-k])."""
    c = 0.5 * (c - c[::-1])
    t = 0.5 * (t - t[::-1])
    return c, t


@functools.lru_cache(maxsize=None)
def scalar_codebook(d, bits):
    """fp32 tables of the Beta_d Lloyd-Max quantizer with 2**bits cells.

    Returns (centroids fp32[2**bits], boundaries fp32[2**bits - 1]).  The
    middle boundary of a symmetric codebook is exactly 0.
    """
    c, t, _ = lloyd_max(BetaCoord(d), 2 ** bits)
    c, t = symmetrize(c, t)
    return c.astype(np.float32), t.astype(np.float32)
