"""Pins of the oracle's generator, rotation and Lloyd-Max solver (CPU only).

Each check ties the oracle to something other than itself: published test
vectors, closed forms, textbook tables, distribution tests and the figures the
pages print (tests/golden/pages_values.txt).
"""
import math

import numpy as np
import pytest
from scipy import integrate, stats

from oracle import codebook as cbk
from oracle.rng import gaussians, round_bf16, splitmix64
from oracle.rotation import haar_rotation, qjl_matrix
from tests.conftest import golden_values

G = golden_values()


# ----------------------------------------------------------------- generator
def test_splitmix64_reference_outputs():
    # Vigna's splitmix64 reference program: seed 1234567 prints
    # 6457827717110365317, 3203168211198807973, 9817491932198370423, ...
    out = splitmix64(1234567, np.arange(3))
    assert [int(v) for v in out] == [6457827717110365317, 3203168211198807973, 9817491932198370423]
    # seed 0 starts 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4
    out0 = splitmix64(0, np.arange(2))
    assert [int(v) for v in out0] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4]


def test_box_muller_is_standard_normal():
    g = gaussians(7, 200001)
    assert len(g) == 200001
    assert abs(g.mean()) < 0.01 and abs(g.var() - 1.0) < 0.01
    assert stats.kstest(g, "norm").pvalue > 1e-3
    # counter-based: a prefix does not depend on the requested length
    assert np.array_equal(gaussians(7, 10), g[:10])


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 37.0
    x[:4] = [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -1.0 - 2.0 ** -8, 0.0]  # exact ties
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(round_bf16(x), ref.astype(np.float64))


# ------------------------------------------------------------------ rotation
@pytest.mark.parametrize("d", [8, 128, 256])
def test_rotation_is_orthogonal(d):
    P = haar_rotation(d, 1)
    assert np.max(np.abs(P.T @ P - np.eye(d))) < 1e-12
    x = np.random.default_rng(1).standard_normal((16, d))
    y32 = (x.astype(np.float32) @ P.T.astype(np.float32))
    assert np.max(np.abs(np.linalg.norm(y32, axis=1) / np.linalg.norm(x, axis=1) - 1.0)) < 1e-6


def test_rotated_coordinate_law_is_beta_and_variance_1_over_d():
    # a fixed unit input, many seeds: coordinates are exchangeable with variance
    # 1/d ([suzuke] 第一步) and follow the Beta law the codebook is solved on
    d = 16
    x = np.zeros(d)
    x[3] = 1.0
    ys = np.array([haar_rotation(d, s) @ x for s in range(1000, 3000)])
    assert abs(ys.var() * d - G["rotated_coordinate_variance_times_d"]) < 0.05
    dens = cbk.BetaCoord(d)
    assert stats.kstest(ys[:, 5], dens.cdf).pvalue > 1e-3
    # a wrong exponent in the density would be rejected
    wrong = cbk.BetaCoord(d + 6)
    assert stats.kstest(ys[:, 5], wrong.cdf).pvalue < 1e-3


def test_qjl_matrix_is_bf16_exact_gaussian():
    S = qjl_matrix(128, 128, 2)
    assert np.array_equal(S, round_bf16(S))
    assert abs(S.var() - 1.0) < 0.02


# ---------------------------------------------------------------- Lloyd-Max
# J. Max, "Quantizing for minimum distortion", IRE Trans. Inf. Theory 6 (1960),
# table for the unit normal density: positive output levels, positive interior
# boundaries and mean squared error.
MAX_1960 = {
    2: ([0.7980], [], 0.3634),
    4: ([0.4528, 1.510], [0.9816], 0.1175),
    8: ([0.2451, 0.7560, 1.344, 2.152], [0.5006, 1.050, 1.748], 0.03454),
    16: ([0.1284, 0.3881, 0.6568, 0.9424, 1.256, 1.618, 2.069, 2.733],
         [0.2582, 0.5224, 0.7996, 1.099, 1.437, 1.844, 2.401], 0.009497),
}


@pytest.mark.parametrize("L", [2, 4, 8, 16])
def test_solver_reproduces_max_table_on_gaussian(L):
    c, t, _ = cbk.lloyd_max(cbk.Gaussian(), L)
    xs, ts, D = MAX_1960[L]
    assert np.allclose(c[L // 2:], xs, atol=1.5e-3)
    assert np.allclose(t[L // 2:], ts, atol=1.5e-3)
    assert abs(cbk.distortion(cbk.Gaussian(), c, t) / D - 1.0) < 1e-3


def test_one_bit_closed_forms():
    # N(0,1): c = sqrt(2/pi), D = 1 - 2/pi
    c, t, _ = cbk.lloyd_max(cbk.Gaussian(), 2)
    assert abs(c[1] - math.sqrt(2 / math.pi)) < 1e-13
    # Beta_d: c = E|t| = 2 C_d / (d - 1), D = 1/d - c^2
    for d in (8, 128, 256):
        dens = cbk.BetaCoord(d)
        c, t, _ = cbk.lloyd_max(dens, 2)
        Cd = math.gamma(d / 2) / (math.sqrt(math.pi) * math.gamma((d - 1) / 2)) if d < 300 else dens.C
        assert abs(c[1] - 2 * Cd / (d - 1)) < 1e-13
        assert abs(cbk.distortion(dens, c, t) - (1.0 / d - c[1] ** 2)) < 1e-13


@pytest.mark.parametrize("d,b", [(128, 1), (128, 2), (128, 3), (128, 4), (256, 3), (8, 3)])
def test_fixed_point_conditions(d, b):
    dens = cbk.BetaCoord(d)
    c, t, _ = cbk.lloyd_max(dens, 2 ** b)
    edges = np.concatenate(([-1.0], t, [1.0]))
    scale = 1.0 / math.sqrt(d)
    for k in range(2 ** b):
        num = integrate.quad(lambda x: x * dens.pdf(x), edges[k], edges[k + 1], epsabs=1e-18, epsrel=1e-14, limit=400)[0]
        den = integrate.quad(dens.pdf, edges[k], edges[k + 1], epsabs=1e-18, epsrel=1e-14, limit=400)[0]
        assert abs(num / den - c[k]) < 1e-12 * scale * 10
    assert np.max(np.abs(t - 0.5 * (c[:-1] + c[1:]))) < 1e-12 * scale
    assert np.all(np.diff(c) > 0)


def test_distortion_against_page_figures():
    d = 128
    ratios = {}
    for b in (1, 2, 3, 4):
        dens = cbk.BetaCoord(d)
        c, t, _ = cbk.lloyd_max(dens, 2 ** b)
        D = cbk.distortion(dens, c, t) * d          # E||u - u_hat||^2 for unit u
        ratios[b] = D * 4 ** b
        assert ratios[b] <= G["distortion_ratio_bound_all_bits"] + 0.02
        if b == 3:
            assert abs(D - G["mse_3bit_unit_vectors"]) < 0.006
    assert abs(ratios[1] - G["distortion_ratio_1bit"]) < 0.01
    # large-d Gaussian limit: sqrt(d)-scaled Beta codebook -> Max's table
    c, t, _ = cbk.lloyd_max(cbk.BetaCoord(1 << 16), 8)
    assert np.allclose(c[4:] * 256.0, MAX_1960[8][0], atol=2e-3)


def test_uniform_density_gives_uniform_quantizer():
    dens = cbk.Uniform(0.0, 2 * math.pi)
    c, t, _ = cbk.lloyd_max(dens, 8)
    assert np.allclose(t, 2 * math.pi * np.arange(1, 8) / 8, atol=1e-12)
    assert np.allclose(c, (2 * np.arange(8) + 1) * math.pi / 8, atol=1e-12)


def test_polar_angle_law():
    # psi = atan(rho_b / rho_a) with k coordinates under each child radius
    rng = np.random.default_rng(3)
    for k in (1, 2, 8, 32):
        x = rng.standard_normal((40000, 2 * k))
        ra = np.linalg.norm(x[:, :k], axis=1)
        rb = np.linalg.norm(x[:, k:], axis=1)
        psi = np.arctan2(rb, ra)
        dens = cbk.PolarAngle(k)
        assert stats.kstest(psi, dens.cdf).pvalue > 1e-3
        assert abs(integrate.quad(dens.pdf, 0, math.pi / 2)[0] - 1.0) < 1e-10


def test_symmetric_scalar_codebook_tables():
    for b in (1, 2, 3, 4):
        c, t = cbk.scalar_codebook(128, b)
        assert c.dtype == np.float32 and len(c) == 2 ** b and len(t) == 2 ** b - 1
        assert np.array_equal(c, -c[::-1]) and np.array_equal(t, -t[::-1])
        assert t[len(t) // 2] == 0.0
