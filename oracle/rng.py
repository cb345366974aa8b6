"""Counter-based splitmix64 and Box-Muller Gaussians (oracle side).

The pages draw the rotation Pi and the QJL projection S at random
([suzuke] 第一步: "乘以一個隨機正交矩陣"; [xujun] 第二步: Johnson-Lindenstrauss
transform) without naming a generator.  Both sides of this project therefore
implement one published counter-based generator independently:

* splitmix64 (S. Vigna, public-domain reference code): the k-th output (k >= 0)
  of the stream seeded with ``seed`` is ``mix(seed + (k + 1) * 0x9E3779B97F4A7C15)``
  with ``mix(z) = z ^ (z >> 31)`` after the two xor-shift-multiply rounds
  (30, 0xBF58476D1CE4E5B9) and (27, 0x94D049BB133111EB), all mod 2**64.
* uniforms from the top 53 bits: ``u = (z >> 11) * 2**-53`` in [0, 1); the
  first uniform of a pair uses ``((z >> 11) + 1) * 2**-53`` in (0, 1] so the
  logarithm is finite.
* Box-Muller: normal pair k takes stream outputs 2k and 2k+1:
  ``g[2k] = sqrt(-2 ln u1) cos(2 pi u2)``, ``g[2k+1] = sqrt(-2 ln u1) sin(2 pi u2)``.
"""
import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed, k):
    """k-th output(s) of the splitmix64 stream seeded with ``seed`` (uint64)."""
    k = np.asarray(k, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (k + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def gaussians(seed, count):
    """First ``count`` N(0,1) draws (fp64) of stream ``seed``."""
    npairs = (count + 1) // 2
    k = np.arange(2 * npairs, dtype=np.uint64)
    z = splitmix64(seed, k)
    top = (z >> np.uint64(11)).astype(np.float64)
    u1 = (top[0::2] + 1.0) * 2.0 ** -53
    u2 = top[1::2] * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    return out[:count]


def round_bf16(a):
    """Round fp64/fp32 values to the nearest bfloat16 (ties to even), as fp64."""
    f = np.asarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)
