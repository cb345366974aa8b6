"""Recursive-polar stage 1 ("PolarQuant") of a rotated unit vector (oracle side).

[xujun] 第一步 / [suzuke] 第二步 / [cnyes] 極坐標的妙用: coordinates are paired
into (radius, angle); the radii are paired again, recursively, until one final
radius and d-1 angles remain; every angle is Lloyd-Max coded on its known law.

For d = 2**D and a rotated row y:

* level 1: pair i = (y[2i], y[2i+1]) gives radius rho_1[i] and the full-circle
  angle theta_i in [0, 2 pi) (uniform law, so its Lloyd-Max quantizer is the
  uniform one: cells [2 pi k / L, 2 pi (k+1) / L), midpoint centroids);
* level l >= 2: child radii (rho_a, rho_b) = (rho_{l-1}[2j], rho_{l-1}[2j+1])
  give rho_l[j] = sqrt(rho_a^2 + rho_b^2) and psi = atan(rho_b / rho_a) in
  [0, pi/2] with density ∝ sin^(k-1)(2 psi), k = 2**(l-1).

Every angle gets ``bits`` bits (b-1 for keys, b for values).  Angles are coded
open-loop from the exact radii.

Decisions are taken in fp32 exactly as the kernel takes them, so both sides
agree bit for bit: radii are computed with separately rounded fp32 products,
sum and square root, and "angle >= boundary t" is the exact sign of
rho_b cos t - rho_a sin t >= 0 with (cos t, sin t) held as fp32 (a zero
determinant is a tie and goes to the upper cell).  Level-1 angles first get
their quadrant from the signs, then the same test runs inside the quadrant.

Decoding walks the tree from the root radius (1 for a unit row):
rho_a = rho cos psi_hat, rho_b = rho sin psi_hat, and the leaves are
(rho cos theta_hat, rho sin theta_hat).
"""
import functools
import math

import numpy as np

from .codebook import PolarAngle, lloyd_max


@functools.lru_cache(maxsize=None)
def angle_codebook(k, L):
    c, t, _ = lloyd_max(PolarAngle(k), L)
    return c, t


class PolarTables:
    def __init__(self, d, bits):
        D = int(round(math.log2(d)))
        assert 2 ** D == d and D >= 1
        self.d, self.D, self.bits = d, D, bits
        L = 2 ** bits
        self.L = L
        # level 1: uniform quantizer on [0, 2 pi)
        self.cent = {1: (2.0 * np.arange(L) + 1.0) * math.pi / L}
        self.bound = {1: 2.0 * math.pi * np.arange(1, L) / L}
        for lev in range(2, D + 1):
            self.cent[lev], self.bound[lev] = angle_codebook(2 ** (lev - 1), L)
        # fp32 values both sides use
        self.cent32 = {k: v.astype(np.float32) for k, v in self.cent.items()}
        self.bound32 = {k: v.astype(np.float32) for k, v in self.bound.items()}
        self.bcos = {k: np.cos(v.astype(np.float64)).astype(np.float32) for k, v in self.bound32.items()}
        self.bsin = {k: np.sin(v.astype(np.float64)).astype(np.float32) for k, v in self.bound32.items()}

    def n_angles(self, lev):
        return self.d >> lev


def _ge(rb, ra, c, s):
    """Exact sign test rb*c - ra*s >= 0 on fp32 inputs (products exact in fp64)."""
    return (rb.astype(np.float64) * np.float64(c) - ra.astype(np.float64) * np.float64(s)) >= 0.0


def _radius(a, b):
    a = a.astype(np.float32)
    b = b.astype(np.float32)
    return np.sqrt((a * a) + (b * b)).astype(np.float32)


def polar_encode(tab, y):
    """Codes [N, d-1] (level 1 first, then level 2, ...) of rotated rows y [N, d]."""
    y32 = np.asarray(y, dtype=np.float32)
    L = tab.L
    a, b = y32[:, 0::2], y32[:, 1::2]
    # quadrant (exact sign logic) and rotation into the first quadrant
    q = np.zeros(a.shape, dtype=np.int64)
    q[(a <= 0) & (b > 0)] = 1
    q[(a < 0) & (b <= 0)] = 2
    q[(a >= 0) & (b < 0)] = 3
    ar = np.where(q == 0, a, np.where(q == 1, b, np.where(q == 2, -a, -b)))
    br = np.where(q == 0, b, np.where(q == 1, -a, np.where(q == 2, -b, a)))
    if L == 2:
        idx1 = q // 2
    elif L == 4:
        idx1 = q
    else:
        per = L // 4
        cnt = np.zeros(a.shape, dtype=np.int64)
        for j in range(1, per):
            cnt += _ge(br, ar, tab.bcos[1][j - 1], tab.bsin[1][j - 1])
        idx1 = q * per + cnt
    codes = [idx1]
    rho = _radius(a, b)
    for lev in range(2, tab.D + 1):
        ra, rb = rho[:, 0::2], rho[:, 1::2]
        cnt = np.zeros(ra.shape, dtype=np.int64)
        for k in range(L - 1):
            cnt += _ge(rb, ra, tab.bcos[lev][k], tab.bsin[lev][k])
        codes.append(cnt)
        rho = _radius(ra, rb)
    return np.concatenate(codes, axis=1)


def polar_decode(tab, idx, root=None):
    """Reconstruction [N, d] from codes [N, d-1] (root radius 1 unless given)."""
    N = idx.shape[0]
    offs = [0]
    for lev in range(1, tab.D + 1):
        offs.append(offs[-1] + tab.n_angles(lev))
    rho = np.ones((N, 1)) if root is None else np.asarray(root, dtype=np.float64).reshape(N, 1)
    for lev in range(tab.D, 1, -1):
        c = tab.cent32[lev].astype(np.float64)[idx[:, offs[lev - 1]:offs[lev]]]
        nxt = np.empty((N, 2 * rho.shape[1]))
        nxt[:, 0::2] = rho * np.cos(c)
        nxt[:, 1::2] = rho * np.sin(c)
        rho = nxt
    th = tab.cent32[1].astype(np.float64)[idx[:, :offs[1]]]
    y = np.empty((N, tab.d))
    y[:, 0::2] = rho * np.cos(th)
    y[:, 1::2] = rho * np.sin(th)
    return y


def exact_angles(y):
    """Unquantized (level-ordered) angles of rows y, for reconstruction checks."""
    y = np.asarray(y, dtype=np.float64)
    a, b = y[:, 0::2], y[:, 1::2]
    out = [np.mod(np.arctan2(b, a), 2.0 * math.pi)]
    rho = np.hypot(a, b)
    while rho.shape[1] > 1:
        ra, rb = rho[:, 0::2], rho[:, 1::2]
        out.append(np.arctan2(rb, ra))
        rho = np.hypot(ra, rb)
    return np.concatenate(out, axis=1)


def decode_angles(d, ang, root=None):
    """Inverse of ``exact_angles`` (float angles instead of codes)."""
    N = ang.shape[0]
    D = int(round(math.log2(d)))
    offs = [0]
    for lev in range(1, D + 1):
        offs.append(offs[-1] + (d >> lev))
    rho = np.ones((N, 1)) if root is None else np.asarray(root, dtype=np.float64).reshape(N, 1)
    for lev in range(D, 1, -1):
        c = ang[:, offs[lev - 1]:offs[lev]]
        nxt = np.empty((N, 2 * rho.shape[1]))
        nxt[:, 0::2] = rho * np.cos(c)
        nxt[:, 1::2] = rho * np.sin(c)
        rho = nxt
    th = ang[:, :offs[1]]
    y = np.empty((N, d))
    y[:, 0::2] = rho * np.cos(th)
    y[:, 1::2] = rho * np.sin(th)
    return y
