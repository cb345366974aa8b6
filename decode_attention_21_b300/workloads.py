"""Seeded synthetic inputs shared by the tests, the benchmark and the CPU checker.

This module only draws numbers; it holds none of the compression or scoring
arithmetic.  Every array is reproducible from (seed, name, indices) with
NumPy's PCG64, chunk by chunk, so a GPU run and a CPU check can regenerate the
same slice independently.

Workloads (shapes of the pages' own cases):

* ``gaussian_outlier_keys``: fp32 keys ~N(0, I) with a few seeded channels
  scaled up (tiny estimator check: 4096 x 128, 4 channels x20).
* ``llama_kv``: bf16-valued keys or values shaped like one Llama-3.1-8B
  layer (8 KV heads, head_dim 128): N(0,1) times a per-(kv-head, channel)
  log-normal(0,1) scale, with 2% of the channels (3 of 128, seeded, without
  replacement) scaled x10.
* ``queries``: fp32 ~N(0, I).
* ``block_table``: a paged cache's page assignment: the pages of all
  sequences are a seeded random permutation of the pool (so consecutive
  pages of a sequence are scattered), entries past each sequence's last page
  are -1.
* ``search_mixture``: database and held-out queries from a Gaussian mixture
  (1000 centres ~N(0, I) in d=200, within-cluster sigma 0.3), unit-normalised;
  a synthetic stand-in for the 200-dimensional GloVe vectors.
"""
import numpy as np

DATA_SEED = 20261202

_NAMES = {"keys": 1, "values": 2, "queries": 3, "scale": 4, "outliers": 5,
          "centres": 6, "db": 7, "search_q": 8, "tiny_keys": 9, "tiny_q": 10, "append": 11, "pages": 12}


def _rng(seed, name, *idx):
    return np.random.default_rng([int(seed), _NAMES[name], *[int(i) for i in idx]])


def to_bf16(a):
    """Round fp32 values to bfloat16 (nearest, ties to even); returns fp32."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def gaussian_outlier_keys(n=4096, d=128, n_outlier=4, factor=20.0, seed=DATA_SEED):
    r = _rng(seed, "tiny_keys")
    k = r.standard_normal((n, d)).astype(np.float32)
    ch = r.choice(d, size=n_outlier, replace=False)
    k[:, ch] *= np.float32(factor)
    return k


def queries(shape, seed=DATA_SEED, name="queries"):
    return _rng(seed, name).standard_normal(shape).astype(np.float32)


def llama_channel_scale(h, d=128, seed=DATA_SEED, which="keys", outlier_frac=0.02, factor=10.0):
    """Per-channel scale of kv head ``h``: exp(N(0,1)), 2% channels x10."""
    r = _rng(seed, "scale", h, 0 if which == "keys" else 1)
    s = np.exp(r.standard_normal(d))
    n_out = max(1, int(round(outlier_frac * d)))
    ch = r.choice(d, size=n_out, replace=False)
    s[ch] *= factor
    return s


def layer_outlier_channels(Hkv, E, d=128, seed=DATA_SEED, which="keys"):
    """The E channels of largest RMS scale over the layer's Hkv kv heads (a
    caller's calibration of the channel groups for an outlier-channel split)."""
    rms = np.sqrt(np.mean([llama_channel_scale(h, d, seed, which) ** 2 for h in range(Hkv)], axis=0))
    return np.argsort(-rms, kind="stable")[:E].astype(np.int32)


def llama_kv_slice(b, h, t0, t1, d=128, seed=DATA_SEED, which="keys"):
    """bf16-valued rows t0..t1-1 of sequence b, kv head h (fp32 array [t1-t0, d]).

    Rows are drawn in blocks of 4096 tokens so any slice can be regenerated.
    """
    out = np.empty((t1 - t0, d), dtype=np.float32)
    s = llama_channel_scale(h, d, seed, which)
    blk = 4096
    for bi in range(t0 // blk, (t1 + blk - 1) // blk):
        r = _rng(seed, which, b, h, bi)
        x = r.standard_normal((blk, d)) * s[None, :]
        a, e = max(t0, bi * blk), min(t1, (bi + 1) * blk)
        out[a - t0:e - t0] = x[a - bi * blk:e - bi * blk]
    return to_bf16(out)


def search_centres(n_centres=1000, d_in=200, seed=DATA_SEED):
    return _rng(seed, "centres").standard_normal((n_centres, d_in))


def search_rows(n, which="db", n_centres=1000, d_in=200, sigma=0.3, seed=DATA_SEED, block=1 << 16, start=0):
    """Rows start..start+n-1 of the mixture (fp32, unit-normalised), in blocks."""
    C = search_centres(n_centres, d_in, seed)
    out = np.empty((n, d_in), dtype=np.float32)
    for bi in range(start // block, (start + n + block - 1) // block):
        r = _rng(seed, which, bi)
        j = r.integers(0, n_centres, size=block)
        x = C[j] + sigma * r.standard_normal((block, d_in))
        x /= np.linalg.norm(x, axis=1, keepdims=True)
        a, e = max(start, bi * block), min(start + n, (bi + 1) * block)
        out[a - start:e - start] = x[a - bi * block:e - bi * block]
    return out


def llama_kv_torch(n, d, kv_head, seed=DATA_SEED, which="keys", device="cuda", generator_offset=0):
    """Same recipe as ``llama_kv_slice`` drawn on the GPU with torch's Philox
    generator (for benchmark-sized caches that are never checked row by row):
    N(0,1) times the per-(kv-head, channel) scale, rounded to bf16."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + _NAMES[which] * 7919 + int(kv_head) * 104729 + int(generator_offset))
    s = torch.from_numpy(llama_channel_scale(kv_head, d, seed, which)).to(device=device, dtype=torch.float32)
    x = torch.randn(n, d, generator=g, device=device, dtype=torch.float32) * s
    return x.to(torch.bfloat16)


def block_table(B, max_pages, num_pages, page_size, lens, seed=DATA_SEED):
    """int32 [B, max_pages] page ids: sequence b's pages 0..ceil(lens[b] /
    page_size) - 1 are distinct pages drawn from a seeded permutation of
    range(num_pages); the other entries are -1."""
    need = [-(-int(L) // page_size) for L in lens]
    assert max(need) <= max_pages and sum(need) <= num_pages
    perm = _rng(seed, "pages", B, max_pages, num_pages).permutation(num_pages)
    t = np.full((B, max_pages), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        t[b, : need[b]] = perm[k: k + need[b]]
        k += need[b]
    return t
