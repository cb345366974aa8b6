"""Outlier-channel split: two independent instances of the method on two
channel groups (oracle side, fp64).

TEST INFRASTRUCTURE ONLY (see the package header).

The pages quote cache sizes and scores at 2.5 and 3.5 bits per coordinate
([xujun] 社区验证: 2.5-bit and 3.5-bit caches; [suzuke] 實際跑出來的數據:
3.5 bits matches FP16 on LongBench, 2.5 bits loses 1.2%) without describing
how a fractional width arises.  The reading taken here: the input channels
are split into an outlier group A (a caller-given list of E channels) and the
rest B; each group is compressed as its own vector by its own instance of
the whole method, and group A gets one more bit per coordinate:

* group g has dimension d_g, its own rotation Pi_g (Haar, d_g x d_g), its
  own Lloyd-Max codebook on the law of a rotated coordinate of a
  d_g-dimensional unit vector, its own sketch S_g (m_g = d_g rows) and its
  own stored norms n_g = ||x_g||, gamma_g = ||r_g||;
* seeds: group A uses (seed_pi, seed_s), group B (seed_pi + 1, seed_s + 1);
* the estimate of <q, x> is the sum of the two groups' estimates,
  est_A(q_A, x_A) + est_B(q_B, x_B), with q_g the query's channels of group g.

Each group's estimate is unbiased over its S_g, so the sum is too.  Bits per
coordinate: (E (b + 1) + (d - E) b) / d for the codes plus 4 fp16 norms per
vector (64 / d).

Packed form (the project's own layout, like the rest of ``layout``): the
record of a d = 128 vector whose first E rotated coordinates are group A's
(in order) and the rest group B's, i.e. the mixed-bit record with E
extended coordinates; the norm entry is four fp16 values n_A, gamma_A, n_B,
gamma_B (8 bytes).
"""
import math

import numpy as np

from . import quant


class SplitCodebook:
    """Two quant.Codebook instances over the channel groups (A: outliers)."""

    split = True
    mode = "scalar"

    def __init__(self, d, bits, outliers, kind="prod", seed_pi=1, seed_s=2):
        A = [int(c) for c in outliers]
        assert len(set(A)) == len(A) and all(0 <= c < d for c in A) and 0 < len(A) < d
        B = [c for c in range(d) if c not in set(A)]
        self.d, self.bits, self.kind = d, bits, kind
        self.extra = len(A)
        self.b1 = bits - 1 if kind == "prod" else bits
        self.channels = (np.array(A, dtype=np.int64), np.array(B, dtype=np.int64))
        self.groups = (quant.Codebook(len(A), bits + 1, kind, seed_pi=seed_pi, seed_s=seed_s),
                       quant.Codebook(len(B), bits, kind, seed_pi=seed_pi + 1, seed_s=seed_s + 1))

    def bits_per_coordinate(self, norm_bits=16):
        """Code bits plus the groups' stored norms, per coordinate."""
        E, d = self.extra, self.d
        norms = (2 if self.kind == "prod" else 1) * 2 * norm_bits
        return (E * (self.bits + 1) + (d - E) * self.bits + norms) / d

    def full_rotation(self):
        """The d x d orthogonal map x -> (Pi_A x_A, Pi_B x_B): rotated
        coordinates 0..E-1 are group A's, the rest group B's."""
        d, E = self.d, self.extra
        A, B = self.channels
        M = np.zeros((d, d))
        M[np.ix_(np.arange(E), A)] = self.groups[0].Pi
        M[np.ix_(np.arange(E, d), B)] = self.groups[1].Pi
        return M

    def full_sketch(self):
        """The block-diagonal d x d sketch diag(S_A, S_B) in rotated order."""
        d, E = self.d, self.extra
        S = np.zeros((d, d))
        S[:E, :E] = self.groups[0].S
        S[E:, E:] = self.groups[1].S
        return S

    def qjl_consts(self):
        return tuple(math.sqrt(math.pi / 2.0) / g.m for g in self.groups)


def quantize(scb, x):
    """Each group's channels of raw rows x [N, d] compressed by its own instance."""
    x = np.asarray(x, dtype=np.float64)
    return {"groups": [quant.quantize(g, x[:, ch]) for g, ch in zip(scb.groups, scb.channels)]}


def encode_rotated(scb, y, n):
    """From rotated rows y [N, d] (group A's unit vector in columns 0..E-1,
    group B's in the rest) and the groups' norms n [N, 2]."""
    y = np.asarray(y, dtype=np.float64)
    n = np.asarray(n, dtype=np.float64)
    E = scb.extra
    return {"groups": [quant.encode_rotated(scb.groups[0], y[:, :E], n[:, 0]),
                       quant.encode_rotated(scb.groups[1], y[:, E:], n[:, 1])]}


def rotate(scb, x):
    """(y [N, d], n [N, 2]): each group rotated by its Pi_g and normalised by
    its own norm, group A in columns 0..E-1."""
    parts = [quant.rotate(g, np.asarray(x, dtype=np.float64)[:, ch]) for g, ch in zip(scb.groups, scb.channels)]
    return np.concatenate([parts[0][0], parts[1][0]], axis=1), np.stack([parts[0][1], parts[1][1]], axis=1)


def estimate(scb, q, code, rows=None, use_fp16_norms=True, qjl=True):
    """Sum of the groups' estimates for query rows q [Q, d] -> [Q, N]."""
    from .estimate import estimate as est
    q = np.asarray(q, dtype=np.float64)
    return sum(est(g, q[:, ch], c, rows, use_fp16_norms, qjl)
               for g, ch, c in zip(scb.groups, scb.channels, code["groups"]))


def pack(scb, code):
    """(records uint32 [N, W], norms uint16 [N, 4]) in the mixed-bit record
    layout with E extended coordinates."""
    from . import layout
    ca, cb_ = code["groups"]
    view = _RecordView(scb)
    merged = {"idx": np.concatenate([ca["idx"], cb_["idx"]], axis=1)}
    if scb.kind == "prod":
        merged["sigma"] = np.concatenate([ca["sigma"], cb_["sigma"]], axis=1)
    merged["n16"] = ca["n16"]
    merged["g16"] = ca.get("g16", ca["n16"])
    rec, _ = layout.pack(view, merged)
    cols = [ca["n16"], ca["g16"], cb_["n16"], cb_["g16"]] if scb.kind == "prod" else [ca["n16"], cb_["n16"]]
    norms = np.stack([c.view(np.uint16) for c in cols], axis=1)
    return rec, norms


def unpack(scb, rec, norms):
    """Inverse of ``pack``."""
    from . import layout
    view = _RecordView(scb)
    E = scb.extra
    one = np.zeros((rec.shape[0], 2), dtype=np.uint16)
    m = layout.unpack(view, rec, one)
    out = []
    k = 2 if scb.kind == "prod" else 1
    for gi, sl in enumerate((slice(0, E), slice(E, scb.d))):
        c = {"idx": m["idx"][:, sl]}
        if scb.kind == "prod":
            c["sigma"] = m["sigma"][:, sl]
            c["g16"] = norms[:, gi * k + 1].copy().view(np.float16)
        c["n16"] = norms[:, gi * k].copy().view(np.float16)
        out.append(quant.decode_codes(scb.groups[gi], c))
    return {"groups": out}


class _RecordView:
    """The record geometry of a split codebook, as ``layout`` reads it."""

    mode = "scalar"

    def __init__(self, scb):
        self.d, self.b1, self.kind, self.extra = scb.d, scb.b1, scb.kind, scb.extra


def write_cache(scb, rows_total, code, row_ids=None):
    """Byte image (uint8) of a cache of ``rows_total`` rows holding ``code``."""
    from . import layout
    rec, norms = pack(scb, code)
    N = rec.shape[0]
    row_ids = np.arange(N) if row_ids is None else np.asarray(row_ids)
    W = layout.record_words(_RecordView(scb))
    nb = 2 * norms.shape[1]
    off = ((rows_total * W * 4 + 255) // 256) * 256
    buf = np.zeros(off + rows_total * nb, dtype=np.uint8)
    buf[: rows_total * W * 4].view(np.uint32).reshape(rows_total, W)[row_ids] = rec
    buf[off:].view(np.uint16).reshape(rows_total, nb // 2)[row_ids] = norms
    return buf


def read_cache(scb, rows_total, buf, row_ids=None):
    """Decode rows ``row_ids`` of a split cache byte image (uint8)."""
    from . import layout
    W = layout.record_words(_RecordView(scb))
    k = 4 if scb.kind == "prod" else 2
    off = ((rows_total * W * 4 + 255) // 256) * 256
    planes = buf[: rows_total * W * 4].view(np.uint32).reshape(rows_total, W)
    nview = buf[off: off + rows_total * 2 * k].view(np.uint16).reshape(rows_total, k)
    sel = slice(None) if row_ids is None else np.asarray(row_ids)
    return unpack(scb, planes[sel], nview[sel])


def cache_bytes(scb, rows):
    from . import layout
    W = layout.record_words(_RecordView(scb))
    return ((rows * W * 4 + 255) // 256) * 256 + rows * (8 if scb.kind == "prod" else 4)
