"""TurboQuant compression of one batch of vectors (oracle side, fp64).

Pipeline ([suzuke] 技術上怎麼做到的, 第一步..第三步; [xujun] 两步绝杀):

1. rotate: y = Pi x / n with n = ||x|| (n = 0 gives y = 0);
2. stage 1 (scalar mode, "TurboQuant-MSE" per coordinate): a Lloyd-Max code
   per rotated coordinate, b-1 bits for keys (kind "prod"), b bits for values
   (kind "mse");  idx_i = #{k : y_i >= t_k}, so a tie goes to the upper cell;
3. QJL (kind "prod" only, [xujun] 第二步 / [cnyes] 1 bit 掃尾): the residual
   r = y - yhat is sketched by S and only sign(S r) is kept (z = 0 counts as
   +1), together with gamma = ||r||.

n and gamma are stored as fp16 (round to nearest even); the scores use the
stored fp16 values.  The recursive-polar stage 1 is in ``polar``.

Mixed bits ([xujun] 社区验证 2.5-bit / 3.5-bit figures): the first ``extra``
rotated coordinates (exchangeable after Pi) get one more stage-1 bit from a
codebook with twice as many cells.
"""
import math

import numpy as np

from . import codebook as cbk
from .rotation import haar_rotation, qjl_matrix


class Codebook:
    """Everything the method fixes before the first vector arrives."""

    def __init__(self, d, bits, kind="prod", mode="scalar", seed_pi=1, seed_s=2, m=None, extra=0):
        assert kind in ("prod", "mse") and mode in ("scalar", "polar")
        self.d, self.bits, self.kind, self.mode = d, bits, kind, mode
        self.b1 = bits - 1 if kind == "prod" else bits
        assert self.b1 >= 1
        self.m = m if m is not None else d
        self.extra = extra
        self.seed_pi, self.seed_s = seed_pi, seed_s
        self.Pi = haar_rotation(d, seed_pi)
        self.S = qjl_matrix(self.m, d, seed_s) if kind == "prod" else None
        self.qjl_const = math.sqrt(math.pi / 2.0) / self.m
        if mode == "scalar":
            self.c, self.t = cbk.scalar_codebook(d, self.b1)
            if extra:
                self.c_x, self.t_x = cbk.scalar_codebook(d, self.b1 + 1)
        else:
            from .polar import PolarTables
            assert extra == 0
            self.polar = PolarTables(d, self.b1)


def stage1_scalar(cb, y):
    """Scalar Lloyd-Max codes and reproduction values of rotated rows y [N, d]."""
    t = cb.t.astype(np.float64)
    idx = np.sum(y[..., None] >= t, axis=-1).astype(np.int64)
    yhat = cb.c.astype(np.float64)[idx]
    if cb.extra:
        E = cb.extra
        tx = cb.t_x.astype(np.float64)
        idx_x = np.sum(y[:, :E, None] >= tx, axis=-1).astype(np.int64)
        idx[:, :E] = idx_x
        yhat[:, :E] = cb.c_x.astype(np.float64)[idx_x]
    return idx, yhat


def rotate(cb, x):
    """(y, n): y = Pi x / ||x|| row-wise, x zero-padded to d columns."""
    x = np.asarray(x, dtype=np.float64)
    if x.shape[1] < cb.d:
        x = np.concatenate([x, np.zeros((x.shape[0], cb.d - x.shape[1]))], axis=1)
    n = np.linalg.norm(x, axis=1)
    y = x @ cb.Pi.T
    inv = np.divide(1.0, n, out=np.zeros_like(n), where=n > 0)
    return y * inv[:, None], n


def encode_rotated(cb, y, n):
    """Stage 1 + QJL from already rotated, unit-norm rows y [N, d] (fp64 or fp32)."""
    y = np.asarray(y, dtype=np.float64)
    out = {"n": np.asarray(n, dtype=np.float64)}
    if cb.mode == "scalar":
        idx, yhat = stage1_scalar(cb, y)
    else:
        from .polar import polar_encode, polar_decode
        idx = polar_encode(cb.polar, y)
        yhat = polar_decode(cb.polar, idx)
    out["idx"], out["yhat"] = idx, yhat
    if cb.kind == "prod":
        r = y - yhat
        out["gamma"] = np.linalg.norm(r, axis=1)
        z = r @ cb.S.T
        out["z"] = z
        out["sigma"] = z >= 0.0
    out["n16"] = out["n"].astype(np.float16)
    if cb.kind == "prod":
        out["g16"] = out["gamma"].astype(np.float16)
    return out


def quantize(cb, x):
    """Full compression of raw rows x [N, d_in] (d_in <= d)."""
    y, n = rotate(cb, x)
    return encode_rotated(cb, y, n)


def dequantize_rotated(cb, code, use_fp16_norms=True):
    """n * yhat in the rotated domain (the MSE reconstruction of Pi x)."""
    n = code["n16"].astype(np.float64) if use_fp16_norms else code["n"]
    return code["yhat"] * n[:, None]


def decode_codes(cb, code):
    """Add the reproduction values ``yhat`` to unpacked codes (in place)."""
    idx = code["idx"]
    if cb.mode == "polar":
        from .polar import polar_decode
        code["yhat"] = polar_decode(cb.polar, idx)
    else:
        yhat = cb.c.astype(np.float64)[np.minimum(idx, len(cb.c) - 1)]
        if cb.extra:
            yhat[:, :cb.extra] = cb.c_x.astype(np.float64)[idx[:, :cb.extra]]
        code["yhat"] = yhat
    return code
