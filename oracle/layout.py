"""Byte layout of the packed bit-plane cache (oracle side, written independently).

The pages fix no layout; this is the project's format, which the CUDA path
writes and reads and which the oracle writes here from its own codes.

A cache holding R rows is one byte buffer:

    [ R records of 4*W bytes ][ pad to 256 B ][ R norm entries ]

Record of one row (W uint32 words, little-endian):
  * code planes p = 0 .. P-1 (plane 0 = most significant bit of the stage-1
    index); for kind "prod" a final plane holds the QJL signs (bit = 1 for +1);
  * word (c, p) sits at word offset c * P + p, c = 0 .. d/32 - 1, and its bit
    j belongs to coordinate (or sign row, or polar angle slot) 32 c + j;
  * mixed bits: the first E coordinates carry (b'+1)-bit indices; the P code
    planes hold their top b' bits and E/32 trailing words hold their lowest bit
    (word d/32*P + e/32, bit e%32 for coordinate e < E).
Norm entry: kind "prod": fp16 n then fp16 gamma (4 bytes); kind "mse": fp16 n.

Polar mode replaces coordinates by angle slots.  For d = 2**D (D >= 5) the
d-1 angles split into d/32 subtrees of 32 leaves; subtree s keeps its 31
angles in word s, bits 0-15 level 1, 16-23 level 2, 24-27 level 3, 28-29
level 4 and 30 level 5, each level in index order; the d/32 - 1 angles above
the subtrees go, root first and level by level (heap order), to bit 31 of
words 0, 1, ...; the last word's bit 31 is zero.
"""
import numpy as np


def n_planes(cb):
    return cb.b1 + (1 if cb.kind == "prod" else 0)


def record_words(cb):
    w = (cb.d // 32) * n_planes(cb)
    if cb.extra:
        w += cb.extra // 32
    return w


def norm_bytes(cb):
    return 4 if cb.kind == "prod" else 2


def cache_bytes(cb, rows):
    planes = rows * record_words(cb) * 4
    return ((planes + 255) // 256) * 256 + rows * norm_bytes(cb)


def polar_slots(d):
    """Slot (32*word + bit) of each level-ordered polar angle."""
    D = d.bit_length() - 1
    assert 2 ** D == d and D >= 5
    nsub = d // 32
    slots = []
    base_bit = {1: 0, 2: 16, 3: 24, 4: 28, 5: 30}
    per_sub = {1: 16, 2: 8, 3: 4, 4: 2, 5: 1}
    for lev in range(1, 6):
        for j in range(d >> lev):
            s, r = divmod(j, per_sub[lev])
            slots.append(32 * s + base_bit[lev] + r)
    # top tree in heap order: root (level D) first
    top = []
    for lev in range(D, 5, -1):
        top.extend([(lev, j) for j in range(d >> lev)])
    top_slot = {key: 32 * i + 31 for i, key in enumerate(top)}
    for lev in range(6, D + 1):
        for j in range(d >> lev):
            slots.append(top_slot[(lev, j)])
    slots = np.array(slots, dtype=np.int64)
    assert len(slots) == d - 1 and len(set(slots.tolist())) == d - 1
    return slots


def _bits_to_words(bits):
    """bits [N, 32*k] (0/1) -> uint32 words [N, k], bit j of word c = bits[32c+j]."""
    N, nb = bits.shape
    b = bits.reshape(N, nb // 32, 32).astype(np.uint64)
    return (b << np.arange(32, dtype=np.uint64)).sum(axis=2).astype(np.uint32)


def _words_to_bits(words):
    w = words.astype(np.uint64)[:, :, None]
    return ((w >> np.arange(32, dtype=np.uint64)) & np.uint64(1)).reshape(words.shape[0], -1).astype(np.int64)


def pack(cb, code):
    """(records uint32 [N, W], norms uint16 [N, 2 or 1]) of one coded batch."""
    idx = code["idx"]
    N, d = idx.shape[0], cb.d
    if cb.mode == "polar":
        slots = polar_slots(d)
        full = np.zeros((N, d), dtype=np.int64)
        full[:, slots] = idx
        idx = full
    P = n_planes(cb)
    words = np.zeros((N, d // 32, P), dtype=np.uint32)
    top = idx.copy()
    if cb.extra:
        top[:, :cb.extra] = idx[:, :cb.extra] >> 1
    for p in range(cb.b1):
        plane = (top >> (cb.b1 - 1 - p)) & 1
        words[:, :, p] = _bits_to_words(plane)
    if cb.kind == "prod":
        words[:, :, cb.b1] = _bits_to_words(code["sigma"].astype(np.int64))
    rec = words.reshape(N, -1)
    if cb.extra:
        lsb = _bits_to_words((idx[:, :cb.extra] & 1))
        rec = np.concatenate([rec, lsb], axis=1)
    if cb.kind == "prod":
        norms = np.stack([code["n16"].view(np.uint16), code["g16"].view(np.uint16)], axis=1)
    else:
        norms = code["n16"].view(np.uint16)[:, None]
    return rec, norms


def unpack(cb, rec, norms):
    """Inverse of ``pack``: dict with idx, sigma (prod), n16, g16 (prod)."""
    N, d = rec.shape[0], cb.d
    P = n_planes(cb)
    words = rec[:, :(d // 32) * P].reshape(N, d // 32, P)
    idx = np.zeros((N, d), dtype=np.int64)
    for p in range(cb.b1):
        idx = (idx << 1) | _words_to_bits(words[:, :, p])
    out = {}
    if cb.extra:
        lsb = _words_to_bits(rec[:, (d // 32) * P:])
        idx[:, :cb.extra] = (idx[:, :cb.extra] << 1) | lsb
    if cb.mode == "polar":
        idx = idx[:, polar_slots(d)]
    out["idx"] = idx
    if cb.kind == "prod":
        out["sigma"] = _words_to_bits(words[:, :, cb.b1]).astype(bool)
        out["n16"] = norms[:, 0].copy().view(np.float16)
        out["g16"] = norms[:, 1].copy().view(np.float16)
    else:
        out["n16"] = norms[:, 0].copy().view(np.float16)
    return out


def write_cache(cb, rows_total, code, row_ids=None):
    """Byte image (uint8) of a cache of ``rows_total`` rows holding ``code``."""
    rec, norms = pack(cb, code)
    N = rec.shape[0]
    row_ids = np.arange(N) if row_ids is None else np.asarray(row_ids)
    buf = np.zeros(cache_bytes(cb, rows_total), dtype=np.uint8)
    W = record_words(cb)
    planes = buf[: rows_total * W * 4].view(np.uint32).reshape(rows_total, W)
    planes[row_ids] = rec
    off = ((rows_total * W * 4 + 255) // 256) * 256
    nb = norm_bytes(cb)
    nview = buf[off: off + rows_total * nb].view(np.uint16).reshape(rows_total, nb // 2)
    nview[row_ids] = norms
    return buf


def read_cache(cb, rows_total, buf, row_ids=None):
    """Decode rows ``row_ids`` of a cache byte image (uint8)."""
    W = record_words(cb)
    planes = buf[: rows_total * W * 4].view(np.uint32).reshape(rows_total, W)
    off = ((rows_total * W * 4 + 255) // 256) * 256
    nb = norm_bytes(cb)
    nview = buf[off: off + rows_total * nb].view(np.uint16).reshape(rows_total, nb // 2)
    sel = slice(None) if row_ids is None else np.asarray(row_ids)
    return unpack(cb, planes[sel], nview[sel])
