"""Seeded random rotation Pi and QJL projection S (oracle side).

[suzuke] 第一步 / [xujun] 第一步: every vector is multiplied by a random
orthogonal matrix so that its coordinates become identically distributed
(≈ N(0, 1/d), exactly the Beta law of a coordinate of a uniform point on the
sphere) whatever the input looks like; the method is data-oblivious.

Pi is Haar-distributed: G (d x d, iid N(0,1) from stream ``seed_pi``, row-major)
is factored G = QR by Householder QR and Pi = Q diag(sign(diag R)), the unique
orthogonal factor with a positive-diagonal R.  The rotated vector is y = Pi x.

S (m x d) is the Johnson-Lindenstrauss sign-sketch matrix of [xujun] 第二步:
iid N(0,1) from stream ``seed_s`` (row-major), each draw rounded to fp32 and
then to bfloat16 (both round-to-nearest-even) so that it is held exactly by
the tensor-core path.
"""
import numpy as np

from .rng import gaussians, round_bf16


def haar_rotation(d, seed_pi):
    """Pi as fp64 [d, d] (rows are the output coordinates)."""
    G = gaussians(seed_pi, d * d).reshape(d, d)
    Q, R = np.linalg.qr(G)
    s = np.sign(np.diag(R))
    s[s == 0] = 1.0
    return Q * s[None, :]


def qjl_matrix(m, d, seed_s):
    """S as fp64 [m, d] holding bfloat16-exact values."""
    return round_bf16(gaussians(seed_s, m * d)).reshape(m, d)
