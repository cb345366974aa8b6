"""Pins of the oracle's encoder, QJL estimator, polar mode, layout and consumers.

CPU only.  Brute force on tiny inputs, the estimator's unbiasedness over many
sketch seeds, the bias without QJL (2/pi at one bit), exact attention/search
as the bit width grows, and hand-built layout examples.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import estimate, layout, polar, quant
from oracle import codebook as cbk
from tests.conftest import golden_values
from decode_attention_21_b300 import workloads as wl

G = golden_values()


def unit_rows(n, d, seed):
    x = np.random.default_rng(seed).standard_normal((n, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


# ------------------------------------------------------------- scalar stage 1
def test_d8_brute_force_scalar_encoder():
    cb = quant.Codebook(8, 3, kind="prod")       # b' = 2 bits per coordinate
    y = unit_rows(64, 8, 5)
    idx, yhat = quant.stage1_scalar(cb, y)
    c = cb.c.astype(np.float64)
    words = np.array(list(itertools.product(range(4), repeat=8)))   # 65536 codewords
    recon = c[words]
    for r in range(len(y)):
        err = np.sum((recon - y[r]) ** 2, axis=1)
        assert np.array_equal(words[np.argmin(err)], idx[r])
        assert np.allclose(recon[np.argmin(err)], yhat[r])


def test_encoder_tie_goes_to_upper_cell():
    cb = quant.Codebook(128, 3, kind="mse")
    y = np.zeros((1, 128))
    y[0, :7] = cb.t.astype(np.float64)
    idx, _ = quant.stage1_scalar(cb, y)
    assert list(idx[0, :7]) == list(range(1, 8))
    assert idx[0, 7] == 4     # y = 0 sits on the middle boundary


def test_unit_vector_mse_at_three_bits():
    # stage 1 alone at 3 bits on unit vectors ([suzuke] MSE 0.03 at 3 bits)
    cb = quant.Codebook(128, 3, kind="mse")
    x = np.random.default_rng(2).standard_normal((20000, 128))
    code = quant.quantize(cb, x)
    y, _ = quant.rotate(cb, x)
    mse = np.mean(np.sum((y - code["yhat"]) ** 2, axis=1))
    D = cbk.distortion(cbk.BetaCoord(128), cb.c.astype(np.float64), cb.t.astype(np.float64)) * 128
    assert abs(mse - D) < 0.003
    assert abs(mse - G["mse_3bit_unit_vectors"]) < 0.006


def test_rotation_makes_outliers_harmless():
    # same distortion with and without huge outlier channels: data-oblivious
    cb = quant.Codebook(128, 3, kind="mse")
    x = np.random.default_rng(3).standard_normal((4000, 128))
    x2 = x.copy()
    x2[:, :4] *= 20.0
    e = []
    for xx in (x, x2):
        code = quant.quantize(cb, xx)
        y, _ = quant.rotate(cb, xx)
        e.append(np.mean(np.sum((y - code["yhat"]) ** 2, axis=1)))
    assert abs(e[0] - e[1]) < 0.004


def test_mixed_bits_codes():
    cb = quant.Codebook(128, 3, kind="prod", extra=32)
    y = unit_rows(200, 128, 4)
    idx, yhat = quant.stage1_scalar(cb, y)
    assert idx[:, :32].max() <= 7 and idx[:, 32:].max() <= 3
    # the extra bit lowers the error on the first quarter
    e_hi = np.mean((y[:, :32] - yhat[:, :32]) ** 2)
    e_lo = np.mean((y[:, 32:] - yhat[:, 32:]) ** 2)
    assert e_hi < 0.5 * e_lo


# ----------------------------------------------------------------- QJL / est
def _tiny():
    x = wl.gaussian_outlier_keys(4096)
    q = wl.queries((8, 128), name="tiny_q")
    return x, q


def test_estimator_unbiased_over_sketch_seeds():
    """Mean over 1000 S seeds within 3 standard errors of <q, x> for nearly all pairs."""
    x, q = _tiny()
    cb = quant.Codebook(128, 3, kind="prod", seed_s=1000)
    y, n = quant.rotate(cb, x)
    idx, yhat = quant.stage1_scalar(cb, y)
    r = y - yhat
    gam = np.linalg.norm(r, axis=1)
    q1 = q.astype(np.float64) @ cb.Pi.T
    base = (q1 @ yhat.T) * n[None, :]
    true = q.astype(np.float64) @ x.astype(np.float64).T
    from oracle.rotation import qjl_matrix
    s1 = np.zeros_like(true)
    s2 = np.zeros_like(true)
    T = 1000
    for seed in range(1000, 1000 + T):
        S = qjl_matrix(128, 128, seed)
        sig = np.where(r @ S.T >= 0, 1.0, -1.0)
        est = base + ((q1 @ S.T) @ sig.T) * (gam * n * cb.qjl_const)[None, :]
        s1 += est
        s2 += est * est
    mean = s1 / T
    se = np.sqrt(np.maximum(s2 / T - mean ** 2, 0) / T)
    zz = (mean - true) / se
    assert np.mean(np.abs(zz) > 3) <= 0.005
    assert abs(np.mean(zz)) < 0.1


@pytest.mark.parametrize("bits", [2, 3])
def test_bias_without_qjl_and_with_qjl(bits):
    """Slope of est on <q,x>: 1 - D_{b'} without QJL (2/pi at b' = 1), 1 with it."""
    cb = quant.Codebook(128, bits, kind="prod")
    x = np.random.default_rng(9).standard_normal((3000, 128))
    q = np.random.default_rng(10).standard_normal((16, 128))
    code = quant.quantize(cb, x)
    true = (q @ x.T).ravel()
    no = estimate.estimate(cb, q, code, use_fp16_norms=False, qjl=False).ravel()
    yes = estimate.estimate(cb, q, code, use_fp16_norms=False, qjl=True).ravel()
    slope_no = np.dot(no, true) / np.dot(true, true)
    slope_yes = np.dot(yes, true) / np.dot(true, true)
    D = cbk.distortion(cbk.BetaCoord(128), cb.c.astype(np.float64), cb.t.astype(np.float64)) * 128
    assert abs(slope_no - (1.0 - D)) < 0.02
    if bits == 2:
        assert abs(slope_no - G["mse_1bit_inner_product_bias"]) < 0.02
    assert abs(slope_yes - 1.0) < 0.03


# -------------------------------------------------------------------- polar
def test_polar_reconstruction_from_exact_angles():
    for d in (8, 128, 256):
        y = unit_rows(50, d, 11)
        ang = polar.exact_angles(y)
        assert ang.shape == (50, d - 1)
        assert np.max(np.abs(polar.decode_angles(d, ang) - y)) < 1e-12


def test_polar_encoder_d8_brute_force():
    tab = polar.PolarTables(8, 2)
    y = unit_rows(300, 8, 12)
    idx = polar.polar_encode(tab, y)
    ang = polar.exact_angles(y)
    offs = [0, 4, 6, 7]
    for lev in (1, 2, 3):
        a = ang[:, offs[lev - 1]:offs[lev]]
        cells = np.searchsorted(tab.bound[lev], a, side="right")
        # away from the (fp32-rounded) boundaries the code is the atan2 cell
        dist = np.min(np.abs(a[..., None] - tab.bound[lev][None, None, :]), axis=-1)
        ok = dist > 1e-5
        assert ok.mean() > 0.99
        assert np.array_equal(cells[ok], idx[:, offs[lev - 1]:offs[lev]][ok])
        # each angle's code is its nearest centroid
        cen = np.argmin(np.abs(a[..., None] - tab.cent[lev][None, None, :]), axis=-1)
        if lev == 1:
            # circular distance for the full-circle angle
            diff = np.abs(a[..., None] - tab.cent[lev][None, None, :])
            diff = np.minimum(diff, 2 * math.pi - diff)
            cen = np.argmin(diff, axis=-1)
        assert np.array_equal(cen[ok], idx[:, offs[lev - 1]:offs[lev]][ok])


def test_polar_error_decreases_with_bits():
    y = unit_rows(2000, 128, 13)
    errs = []
    for b in (1, 2, 3, 4):
        tab = polar.PolarTables(128, b)
        yh = polar.polar_decode(tab, polar.polar_encode(tab, y))
        errs.append(np.mean(np.sum((yh - y) ** 2, axis=1)))
    assert all(errs[i + 1] < errs[i] for i in range(3))


def _centroid_angles(tab, idx):
    """Level-ordered centroid angles of codes idx, each level from its own table."""
    out, off = [], 0
    for lev in range(1, tab.D + 1):
        n = tab.n_angles(lev)
        out.append(tab.cent32[lev].astype(np.float64)[idx[:, off:off + n]])
        off += n
    return np.concatenate(out, axis=1)


@pytest.mark.parametrize("d,bits", [(8, 1), (8, 3), (128, 2), (256, 3)])
def test_polar_decode_is_the_tree_walk_of_the_centroid_angles(d, bits):
    # [xujun] 第一步 / [suzuke] 第二步: decoding replaces every angle by its
    # cell's centroid and walks the radius tree back down; decode_angles is
    # pinned separately by the exact arctan2 round trip, so a swapped cos/sin
    # or a level read from the wrong table in polar_decode shows up here
    tab = polar.PolarTables(d, bits)
    rng = np.random.default_rng(21 + d + bits)
    idx = rng.integers(0, tab.L, size=(300, d - 1))
    got = polar.polar_decode(tab, idx)
    want = polar.decode_angles(d, _centroid_angles(tab, idx))
    assert np.max(np.abs(got - want)) < 1e-12
    roots = rng.uniform(0.5, 2.0, size=300)
    got = polar.polar_decode(tab, idx, root=roots)
    want = polar.decode_angles(d, _centroid_angles(tab, idx), root=roots)
    assert np.max(np.abs(got - want)) < 1e-12


@pytest.mark.parametrize("bits", [1, 2])
def test_polar_decode_d8_written_out_by_hand(bits):
    # d = 8: four level-1 angles t0..t3 (pairs (y0,y1) .. (y6,y7)), two level-2
    # angles a (over the radii of pairs 0,1) and b (pairs 2,3), one level-3
    # angle c (over the two level-2 radii); root radius 1.  Every code word.
    tab = polar.PolarTables(8, bits)
    L = tab.L
    words = np.array(list(itertools.product(range(L), repeat=7)))
    th = tab.cent32[1].astype(np.float64)[words[:, 0:4]]
    a = tab.cent32[2].astype(np.float64)[words[:, 4]]
    b = tab.cent32[2].astype(np.float64)[words[:, 5]]
    c = tab.cent32[3].astype(np.float64)[words[:, 6]]
    cos, sin = np.cos, np.sin
    want = np.stack([
        cos(c) * cos(a) * cos(th[:, 0]), cos(c) * cos(a) * sin(th[:, 0]),
        cos(c) * sin(a) * cos(th[:, 1]), cos(c) * sin(a) * sin(th[:, 1]),
        sin(c) * cos(b) * cos(th[:, 2]), sin(c) * cos(b) * sin(th[:, 2]),
        sin(c) * sin(b) * cos(th[:, 3]), sin(c) * sin(b) * sin(th[:, 3]),
    ], axis=1)
    got = polar.polar_decode(tab, words)
    assert np.max(np.abs(got - want)) < 1e-12
    # the level-2 and level-3 laws differ (sin^1(2 psi) vs sin^3(2 psi)), so a
    # level decoded with another level's table would not match
    assert not np.allclose(tab.cent32[2], tab.cent32[3])


def test_polar_quadrant_rule():
    tab = polar.PolarTables(8, 3)
    # points on the axes and at 45 degrees: ties go to the upper cell; the zero
    # pair sits in quadrant 0 and ties with the 45-degree boundary
    pts = [(1, 0), (0, 1), (-1, 0), (0, -1), (1, 1), (-1, -1), (0, 0)]
    y = np.zeros((len(pts), 8), dtype=np.float32)
    for i, (a, b) in enumerate(pts):
        y[i, 0], y[i, 1] = a, b
        y[i, 2] = 1.0
    idx = polar.polar_encode(tab, y)[:, 0]
    assert list(idx) == [0, 2, 4, 6, 1, 5, 1]


# ------------------------------------------------------------------- layout
def test_layout_hand_example():
    cb = quant.Codebook(128, 3, kind="prod")      # 2 code planes + sign plane
    code = {"idx": np.zeros((1, 128), dtype=np.int64), "sigma": np.zeros((1, 128), dtype=bool),
            "n16": np.array([1.5], dtype=np.float16), "g16": np.array([0.25], dtype=np.float16)}
    code["idx"][0, 5] = 2        # binary 10: plane 0 bit
    code["idx"][0, 40] = 1       # binary 01: plane 1 bit
    code["sigma"][0, 127] = True
    rec, norms = layout.pack(cb, code)
    assert rec.shape == (1, 12)
    expect = np.zeros(12, dtype=np.uint32)
    expect[0 * 3 + 0] = 1 << 5           # word (c=0, p=0)
    expect[1 * 3 + 1] = 1 << 8           # word (c=1, p=1), coordinate 40 = 32 + 8
    expect[3 * 3 + 2] = 1 << 31          # word (c=3, p=2) = sign plane
    assert np.array_equal(rec[0], expect)
    assert norms[0, 0] == 0x3E00 and norms[0, 1] == 0x3400


@pytest.mark.parametrize("kind,bits,mode,extra", [("prod", 2, "scalar", 0), ("prod", 4, "scalar", 0),
                                                  ("mse", 3, "scalar", 0), ("prod", 3, "scalar", 32),
                                                  ("prod", 3, "polar", 0), ("mse", 3, "polar", 0)])
def test_layout_round_trip(kind, bits, mode, extra):
    cb = quant.Codebook(128, bits, kind=kind, mode=mode, extra=extra)
    x = np.random.default_rng(14).standard_normal((37, 128))
    code = quant.quantize(cb, x)
    buf = layout.write_cache(cb, 50, code, row_ids=np.arange(37) + 5)
    assert buf.nbytes == layout.cache_bytes(cb, 50)
    back = layout.read_cache(cb, 50, buf, row_ids=np.arange(37) + 5)
    assert np.array_equal(back["idx"], code["idx"])
    assert np.array_equal(back["n16"], code["n16"])
    if kind == "prod":
        assert np.array_equal(back["sigma"], code["sigma"])
        assert np.array_equal(back["g16"], code["g16"])
    quant.decode_codes(cb, back)
    assert np.allclose(back["yhat"], code["yhat"])


def test_polar_slots_d128():
    s = layout.polar_slots(128)
    assert s[0] == 0 and s[15] == 15 and s[16] == 32       # level 1 angles 0..15 in word 0
    assert s[64] == 16                                     # first level-2 angle
    assert s[126] == 31                                    # root angle: word 0, bit 31
    assert sorted(s[124:126]) == [63, 95]                  # level 6: words 1 and 2, bit 31


# ---------------------------------------------------------------- consumers
def test_high_bit_estimates_approach_exact_inner_products():
    # the error std roughly halves per extra bit (distortion ~ 4^-b) and the
    # MSE-only part becomes exact
    x = np.random.default_rng(15).standard_normal((500, 128))
    q = np.random.default_rng(16).standard_normal((4, 128))
    true = q @ x.T
    rel = []
    for b in (5, 6, 7):
        cb = quant.Codebook(128, b, kind="prod")
        code = quant.quantize(cb, x)
        est = estimate.estimate(cb, q, code, use_fp16_norms=False)
        rel.append(np.std(est - true) / np.std(true))
    assert rel[2] < 0.04
    assert 1.6 < rel[0] / rel[1] < 2.5 and 1.6 < rel[1] / rel[2] < 2.5
    cb = quant.Codebook(128, 7, kind="mse")
    est = estimate.estimate(cb, q, quant.quantize(cb, x), use_fp16_norms=False)
    assert np.max(np.abs(est - true)) < 0.03 * np.max(np.abs(true))


def test_attention_matches_exact_softmax_attention_at_high_bits():
    B, Hq, Hkv, T, d = 2, 4, 2, 64, 128
    rng = np.random.default_rng(17)
    K = rng.standard_normal((B * Hkv * T, d))
    V = rng.standard_normal((B * Hkv * T, d))
    q = rng.standard_normal((B, Hq, d))
    seq = np.array([64, 37])
    cbk_ = quant.Codebook(d, 7, kind="prod")
    cbv_ = quant.Codebook(d, 6, kind="mse", seed_pi=7)
    kc, vc = quant.quantize(cbk_, K), quant.quantize(cbv_, V)
    scale = 1.0 / math.sqrt(d)
    o = estimate.attention(cbk_, cbv_, kc, vc, q, seq, Hkv, T, scale)
    for b in range(B):
        for h in range(Hq):
            base = (b * Hkv + h // (Hq // Hkv)) * T
            Kb, Vb = K[base:base + seq[b]], V[base:base + seq[b]]
            s = scale * (Kb @ q[b, h])
            p = np.exp(s - s.max())
            ref = (p / p.sum()) @ Vb
            err = np.sqrt(np.mean((o[b, h] - ref) ** 2))
            assert err < 0.06 * np.sqrt(np.mean(ref ** 2))


def test_attention_single_token_returns_its_value():
    d = 128
    cbk_ = quant.Codebook(d, 3, kind="prod")
    cbv_ = quant.Codebook(d, 3, kind="mse")
    K = np.random.default_rng(18).standard_normal((4, d))
    V = np.random.default_rng(19).standard_normal((4, d))
    kc, vc = quant.quantize(cbk_, K), quant.quantize(cbv_, V)
    q = np.random.default_rng(20).standard_normal((1, 2, d))
    o = estimate.attention(cbk_, cbv_, kc, vc, q, np.array([1]), 1, 4, 0.1)
    vhat = (vc["yhat"][0] * float(vc["n16"][0])) @ cbv_.Pi
    assert np.allclose(o[0, 0], vhat) and np.allclose(o[0, 1], vhat)


def test_search_topk_brute_force_and_ties():
    cb = quant.Codebook(128, 4, kind="prod")
    x = np.random.default_rng(21).standard_normal((3000, 100))
    q = np.random.default_rng(22).standard_normal((5, 100))
    code = quant.quantize(cb, x)
    ids, sc = estimate.search(cb, code, q, 10, block=700)
    full = estimate.estimate(cb, q, code)
    for i in range(5):
        order = sorted(range(3000), key=lambda j: (-full[i, j], j))[:10]
        assert list(ids[i]) == order
        assert np.allclose(sc[i], full[i, order])
    s = np.array([[1.0, 3.0, 3.0, 2.0]])
    i2, _ = estimate.topk(s, 3)
    assert list(i2[0]) == [1, 2, 3]


def test_search_recall_high_bits():
    x = wl.search_rows(4000, "db")
    q = wl.search_rows(50, "search_q")
    cb = quant.Codebook(256, 7, kind="prod")
    ids, _ = estimate.search(cb, quant.quantize(cb, x), q, 10)
    true = np.argmax(q.astype(np.float64) @ x.astype(np.float64).T, axis=1)
    assert estimate.recall_1_at_k(true, ids)[10] >= 0.98


def test_dense_logits_brute_force():
    """The unquantized comparator against a plain Python triple loop (tiny case,
    GQA group 2, a short sequence)."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, cap, d = 2, 4, 2, 5, 8
    K = rng.standard_normal((B, Hkv, cap, d))
    q = rng.standard_normal((B, Hq, d))
    lens = [5, 3]
    got = estimate.dense_logits(K, q, lens, Hkv, cap)
    for b in range(B):
        for h in range(Hq):
            for t in range(cap):
                if t >= lens[b]:
                    assert np.isnan(got[b, h, t])
                    continue
                want = 0.0
                for i in range(d):
                    want += float(q[b, h, i]) * float(K[b, h // 2, t, i])
                assert abs(got[b, h, t] - want) <= 1e-12 * (1 + abs(want))


def test_block_table_generator_assigns_distinct_pages():
    """The paged-cache inputs: each sequence's first ceil(len / page) entries
    are distinct pages of the pool (no page shared between sequences), the
    rest are -1, and the same seed gives the same table."""
    B, max_pages, num_pages, ps = 4, 9, 40, 16
    lens = [144, 1, 0, 77]
    t = wl.block_table(B, max_pages, num_pages, ps, lens)
    assert t.shape == (B, max_pages) and t.dtype == np.int32
    used = []
    for b, L in enumerate(lens):
        n = -(-L // ps)
        assert np.all(t[b, n:] == -1)
        assert np.all((t[b, :n] >= 0) & (t[b, :n] < num_pages))
        used.extend(t[b, :n].tolist())
    assert len(used) == len(set(used))
    assert np.array_equal(t, wl.block_table(B, max_pages, num_pages, ps, lens))
