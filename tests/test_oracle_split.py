"""Pins of the oracle's outlier-channel split (CPU only).

The split compresses an outlier channel group A and the remaining channels B
as two independent instances of the method (A with one more bit) and scores
with the sum of the two estimates.  What fixes it independently of the code:
unbiasedness over the sketch draws (each group's estimator is unbiased, so
the sum is; a wrong per-group norm, constant kq or channel map biases it),
the block structure of the combined rotation, a packed record written out by
hand, the bit count, and the variance argument for giving the outlier group
the extra bit.
"""
import math

import numpy as np
import pytest

from oracle import estimate, layout, quant, split


def _rng(seed):
    return np.random.default_rng(seed)


@pytest.mark.parametrize("d,E,bits", [(32, 8, 2), (128, 32, 2), (128, 64, 3)])
def test_split_estimator_is_unbiased_over_sketch_draws(d, E, bits):
    # Fixed rotation seeds, S_A and S_B redrawn per trial: the mean estimate
    # must equal the exact inner product within 3 standard errors.
    r = _rng(5)
    out = r.choice(d, size=E, replace=False)
    x = r.standard_normal(d)
    x[out] *= 10.0
    q = x + 0.5 * r.standard_normal(d)       # aligned pair: a large <q, x>
    exact = float(q @ x)
    ests = []
    for t in range(400):
        scb = split.SplitCodebook(d, bits, out, seed_pi=11, seed_s=1000 + 2 * t)
        code = split.quantize(scb, x[None, :])
        ests.append(float(estimate.estimate(scb, q[None, :], code, use_fp16_norms=False)[0, 0]))
    ests = np.array(ests)
    se = ests.std(ddof=1) / math.sqrt(len(ests))
    assert abs(ests.mean() - exact) <= 3.0 * se + 1e-9 * abs(exact)
    # and the estimate is not trivially exact: the sketch term does vary
    assert ests.std() > 1e-6 * abs(exact)


def test_split_without_sketch_shrinks_each_group_by_its_own_factor():
    # MSE-only scoring (QJL term dropped) of isotropic groups: the expected
    # estimate over the rotation is (1 - D_A) <q_A, x_A> + (1 - D_B) <q_B, x_B>,
    # D_g the stage-1 distortion of group g on unit vectors (fixed by the
    # group's codebook: the A group has one bit more, so it shrinks less).
    d, E, bits = 32, 8, 2
    r = _rng(8)
    out = np.arange(E)
    x = r.standard_normal(d)
    q = r.standard_normal(d)
    qa, qb = float(q[:E] @ x[:E]), float(q[E:] @ x[E:])
    ests = []
    for t in range(600):
        scb = split.SplitCodebook(d, bits, out, seed_pi=3 + 2 * t, seed_s=7)
        code = split.quantize(scb, x[None, :])
        ests.append(float(estimate.estimate(scb, q[None, :], code, use_fp16_norms=False, qjl=False)[0, 0]))
    from oracle import codebook as cbk
    DA = cbk.distortion(cbk.BetaCoord(E), *[v.astype(np.float64) for v in cbk.scalar_codebook(E, bits)]) * E
    DB = cbk.distortion(cbk.BetaCoord(d - E), *[v.astype(np.float64) for v in cbk.scalar_codebook(d - E, bits - 1)]) * (d - E)
    want = (1 - DA) * qa + (1 - DB) * qb
    ests = np.array(ests)
    se = ests.std(ddof=1) / math.sqrt(len(ests))
    assert abs(ests.mean() - want) <= 3.5 * se


def test_split_rotation_is_block_structured_and_orthogonal():
    d, E = 128, 32
    out = _rng(2).choice(d, size=E, replace=False)
    scb = split.SplitCodebook(d, 3, out)
    M = scb.full_rotation()
    assert np.allclose(M @ M.T, np.eye(d), atol=1e-12)
    x = _rng(3).standard_normal((4, d))
    y, n = split.rotate(scb, x)
    assert np.allclose(n[:, 0], np.linalg.norm(x[:, out], axis=1))
    assert np.allclose(n[:, 1], np.linalg.norm(np.delete(x, out, axis=1), axis=1))
    # rotated coordinates 0..E-1 see only the outlier channels, the rest only the others
    x2 = x.copy()
    x2[:, np.delete(np.arange(d), out)] += 1.0
    y2, _ = split.rotate(scb, x2)
    assert np.array_equal(y[:, :E], y2[:, :E])
    z = x @ M.T
    assert np.allclose(y[:, :E] * n[:, :1], z[:, :E]) and np.allclose(y[:, E:] * n[:, 1:], z[:, E:])
    S = scb.full_sketch()
    assert not S[:E, E:].any() and not S[E:, :E].any()


def test_split_record_written_out_by_hand():
    # d = 128, E = 32, b = 2: group A codes are 2-bit (idx_A[j] = j % 4),
    # group B codes 1-bit (idx_B[j] = j % 2); sign rows: A all +1, B +1 where
    # j % 3 == 0.  Record: 4 word columns x 2 planes (top code bit, signs),
    # then the extra word of column 0 (low bit of the A codes).
    scb = split.SplitCodebook(128, 2, list(range(100, 132 - 4)) + [0, 1, 2, 3])
    jA, jB = np.arange(32), np.arange(96)
    ca = {"idx": (jA % 4)[None, :], "sigma": np.ones((1, 32), bool),
          "n16": np.array([1.5], np.float16), "g16": np.array([0.25], np.float16)}
    cb_ = {"idx": (jB % 2)[None, :], "sigma": (jB % 3 == 0)[None, :],
           "n16": np.array([2.0], np.float16), "g16": np.array([0.5], np.float16)}
    rec, norms = split.pack(scb, {"groups": [ca, cb_]})
    want = [0xCCCCCCCC, 0xFFFFFFFF,      # column 0: A codes' top bits (j % 4 in {2, 3}), A signs
            0xAAAAAAAA, 0x49249249,      # column 1: B coordinates 0..31: odd j; j % 3 == 0
            0xAAAAAAAA, 0x92492492,      # column 2: B 32..63: signs where j % 3 == 1
            0xAAAAAAAA, 0x24924924,      # column 3: B 64..95: signs where j % 3 == 2
            0xAAAAAAAA]                  # extra word: low bits of the A codes (odd j)
    assert rec.shape == (1, 9) and [int(w) for w in rec[0]] == want
    assert [int(v) for v in norms[0]] == [0x3E00, 0x3400, 0x4000, 0x3800]
    back = split.unpack(scb, rec, norms)["groups"]
    assert np.array_equal(back[0]["idx"], ca["idx"]) and np.array_equal(back[1]["sigma"], cb_["sigma"])


@pytest.mark.parametrize("E,bits,want", [(32, 2, 2.75), (64, 2, 3.0), (32, 3, 3.75), (64, 3, 4.0)])
def test_split_bit_count(E, bits, want):
    scb = split.SplitCodebook(128, bits, range(E))
    assert scb.bits_per_coordinate() == want
    rows = 1024
    per_row = (split.cache_bytes(scb, rows) - 0) * 8 / rows / 128
    assert abs(per_row - want) < 1e-9


def test_split_gives_outlier_heavy_keys_a_smaller_error_than_one_codebook():
    # Keys whose energy sits in E outlier channels (x 10): the split puts
    # those channels in their own group with one more bit and its own norm.
    # Its inner-product error variance is then about D(b+1) / D(b) ~ 1/4 of
    # the single b-bit instance's (per-group variance ~ n_g^2 |q_g|^2 D_g / d_g).
    d, E, bits, N = 128, 32, 2, 400
    r = _rng(4)
    out = r.choice(d, size=E, replace=False)
    X = r.standard_normal((N, d))
    X[:, out] *= 10.0
    Q = r.standard_normal((8, d))
    exact = Q @ X.T
    scb = split.SplitCodebook(d, bits, out)
    e_split = estimate.estimate(scb, Q, split.quantize(scb, X)) - exact
    plain = quant.Codebook(d, bits, "prod")
    e_plain = estimate.estimate(plain, Q, quant.quantize(plain, X)) - exact
    ratio = np.mean(e_split ** 2) / np.mean(e_plain ** 2)
    assert ratio < 0.5
