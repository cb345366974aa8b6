"""GPU parity: the CUDA path (called through the C ABI) against the oracle on
the same seeded inputs.

* quantize from identical rotated fp32 rows: stage-1 codes bit-exact; QJL
  signs bit-exact except near-ties |z| < 1e-5 * gamma * ||s_j||; fp16 norms
  exact (n) or within one ulp (gamma, fp32 vs fp64 accumulation);
* quantize end to end (fp32 and bf16 inputs): <= 0.1% differing code or sign
  bits, each differing code within 1e-4 / sqrt(d) of a boundary;
* logits / attention: the GPU scores the oracle's own packed cache; per
  (sequence, head) row max |diff| <= 1e-3 * max |oracle|, median relative
  error <= 1e-4 (fp32 accumulation vs fp64).
"""
import math

import numpy as np
import pytest
import torch

from decode_attention_21_b300 import tq
from decode_attention_21_b300 import workloads as wl
from oracle import estimate, layout, quant

pytestmark = pytest.mark.gpu

KIND = {"prod": tq.KIND_PROD, "mse": tq.KIND_MSE}
MODE = {"scalar": tq.MODE_SCALAR, "polar": tq.MODE_POLAR}


def pair(d, bits, kind="prod", mode="scalar", extra=0, seed_pi=1, seed_s=2):
    ocb = quant.Codebook(d, bits, kind=kind, mode=mode, extra=extra, seed_pi=seed_pi, seed_s=seed_s)
    gcb = tq.Codebook(d, bits, KIND[kind], MODE[mode], seed_pi, seed_s, extra=extra)
    return ocb, gcb


def gpu_cache(gcb, rows):
    return torch.zeros(tq.cache_bytes(gcb, rows), dtype=torch.uint8, device="cuda")


def read_back(ocb, rows, buf):
    return layout.read_cache(ocb, rows, buf.cpu().numpy())


def sign_ties(ocb, code, rows=None):
    """Mask of QJL sign bits whose oracle projection is a near-tie."""
    z = code["z"] if rows is None else code["z"][rows]
    g = code["gamma"] if rows is None else code["gamma"][rows]
    sn = np.linalg.norm(ocb.S, axis=1)
    return np.abs(z) < 1e-5 * g[:, None] * sn[None, :]


CASES = [(128, 2, "prod", "scalar", 0), (128, 3, "prod", "scalar", 0), (128, 4, "prod", "scalar", 0),
         (128, 1, "mse", "scalar", 0), (128, 3, "mse", "scalar", 0), (128, 4, "mse", "scalar", 0),
         (128, 3, "prod", "scalar", 32), (128, 2, "prod", "scalar", 64), (256, 2, "prod", "scalar", 0),
         (256, 4, "prod", "scalar", 0), (128, 3, "prod", "polar", 0), (128, 3, "mse", "polar", 0),
         (128, 4, "mse", "polar", 0), (256, 3, "prod", "polar", 0)]


@pytest.mark.parametrize("d,bits,kind,mode,extra", CASES)
def test_quantize_rotated_bit_exact(d, bits, kind, mode, extra):
    ocb, gcb = pair(d, bits, kind, mode, extra)
    n = 1000 + 37
    x = np.random.default_rng(d * 10 + bits).standard_normal((n, d)) * 3.0
    y, nrm = quant.rotate(ocb, x)
    y32 = y.astype(np.float32)
    n32 = nrm.astype(np.float32)
    code = quant.encode_rotated(ocb, y32.astype(np.float64), n32.astype(np.float64))
    rows = n + 5
    perm = np.random.default_rng(1).permutation(rows)[:n]
    cache = gpu_cache(gcb, rows)
    tq.tq_quantize_rotated(gcb, cache, rows, torch.from_numpy(y32).cuda(), torch.from_numpy(n32).cuda(), n,
                           dst_rows=torch.from_numpy(perm.astype(np.int64)).cuda())
    torch.cuda.synchronize()
    got = read_back(ocb, rows, cache)
    sel = np.argsort(perm)
    inv = np.empty(n, dtype=np.int64)
    inv[:] = perm
    g_idx = got["idx"][inv]
    assert np.array_equal(g_idx, code["idx"])
    assert np.array_equal(got["n16"][inv], code["n16"])
    if kind == "prod":
        diff = got["sigma"][inv] != code["sigma"]
        assert not np.any(diff & ~sign_ties(ocb, code))
        g16 = got["g16"][inv].astype(np.float64)
        assert np.all(np.abs(g16 - code["g16"].astype(np.float64)) <= np.spacing(code["g16"]).astype(np.float64) * 1.01)
    del sel


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,bits,kind,mode,extra", [(128, 3, "prod", "scalar", 0), (128, 4, "prod", "scalar", 0),
                                                    (128, 3, "mse", "scalar", 0), (128, 2, "prod", "scalar", 32),
                                                    (256, 2, "prod", "scalar", 0), (128, 3, "prod", "polar", 0)])
def test_quantize_end_to_end(dtype, d, bits, kind, mode, extra):
    ocb, gcb = pair(d, bits, kind, mode, extra)
    d_in = 200 if d == 256 else d
    if dtype == "f32":
        x = wl.gaussian_outlier_keys(4096, d_in)
    else:
        x = wl.llama_kv_slice(0, 1, 0, 4096, d_in)
    code = quant.quantize(ocb, x.astype(np.float64))
    cache = gpu_cache(gcb, len(x))
    xt = torch.from_numpy(x).cuda()
    if dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    tq.tq_quantize(gcb, cache, len(x), xt, len(x), d_in)
    torch.cuda.synchronize()
    got = read_back(ocb, len(x), cache)
    code_bits = (got["idx"] != code["idx"])
    nbits = code["idx"].size * ocb.b1
    flips = code_bits.sum()
    if kind == "prod":
        flips += (got["sigma"] != code["sigma"]).sum()
        nbits += code["sigma"].size
    assert flips <= 1e-3 * nbits
    if mode == "scalar" and code_bits.any():
        y, _ = quant.rotate(ocb, x.astype(np.float64))
        t = ocb.t.astype(np.float64)
        dist = np.min(np.abs(y[code_bits][:, None] - t[None, :]), axis=1)
        assert np.all(dist < 1e-4 / math.sqrt(d))
    n_ref = np.linalg.norm(x.astype(np.float64), axis=1)
    assert np.allclose(got["n16"].astype(np.float64), n_ref, rtol=1e-3)


def oracle_cache(ocb, rows, x):
    code = quant.quantize(ocb, x)
    return code, layout.write_cache(ocb, rows, code)


def rowwise_ok(got, ref, tol=1e-3, med=1e-4):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref), axis=-1, keepdims=True)
    assert np.all(np.abs(got - ref) <= tol * scale + 1e-30), float(np.max(np.abs(got - ref) / scale))
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3 * scale)
    assert np.median(rel) <= med, float(np.median(rel))


@pytest.mark.parametrize("mode", ["scalar", "polar"])
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("B,Hq,Hkv,cap,lens", [(1, 8, 2, 4096, [4096]), (2, 4, 1, 1000, [1000, 1]),
                                               (3, 6, 3, 333, [333, 17, 0]), (1, 2, 2, 64, [49]),
                                               (2, 16, 2, 1000, [1000, 513]), (1, 12, 1, 336, [336]),
                                               (1, 32, 2, 256, [250])])
def test_logits_parity(bits, B, Hq, Hkv, cap, lens, mode):
    ocb, gcb = pair(128, bits, mode=mode)
    rows = B * Hkv * cap
    x = wl.gaussian_outlier_keys(rows, 128)
    code, img = oracle_cache(ocb, rows, x.astype(np.float64))
    q = wl.queries((B, Hq, 128), name="tiny_q")
    ref = estimate.logits(ocb, code, q.astype(np.float64), lens, Hkv, cap)
    kc = torch.from_numpy(img).cuda()
    ws = torch.empty(tq.tq_logits_workspace(gcb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, cap), float("nan"), device="cuda")
    tq.tq_logits(gcb, kc, B, Hq, Hkv, cap, torch.tensor(lens, dtype=torch.int32, device="cuda"),
                 torch.from_numpy(q).cuda(), out, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        L = lens[b]
        assert np.all(np.isnan(got[b, :, L:]))
        if L:
            rowwise_ok(got[b, :, :L], ref[b, :, :L])


@pytest.mark.parametrize("mode", ["scalar", "polar"])
def test_logits_tiny_estimator_config_all_pairs(mode):
    """The tiny estimator check as the configuration states it: 4096 fp32 keys
    ~N(0, I) with 4 outlier channels x20, 8 fp32 queries, b = 3 (2-bit stage 1
    + 1-bit QJL, m = 128), logits for all 8 x 4096 pairs: one kv head shared by
    the 8 query heads (a group of 8, scored 4 heads per launch)."""
    ocb, gcb = pair(128, 3, mode=mode)
    T = 4096
    x = wl.gaussian_outlier_keys(T, 128)
    code, img = oracle_cache(ocb, T, x.astype(np.float64))
    q = wl.queries((1, 8, 128), name="tiny_q")
    ref = estimate.estimate(ocb, q[0].astype(np.float64), code)           # [8, 4096]: every pair
    ws = torch.empty(tq.tq_logits_workspace(gcb, 1, 8, 1), dtype=torch.uint8, device="cuda")
    out = torch.full((1, 8, T), float("nan"), device="cuda")
    tq.tq_logits(gcb, torch.from_numpy(img).cuda(), 1, 8, 1, T, torch.tensor([T], dtype=torch.int32, device="cuda"),
                 torch.from_numpy(q).cuda(), out, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()[0]
    assert np.all(np.isfinite(got))
    rowwise_ok(got, ref)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("B,Hq,Hkv,cap,lens", [(1, 8, 2, 4096, [4096]), (3, 6, 3, 333, [333, 17, 0]),
                                               (2, 4, 1, 1000, [1000, 1])])
def test_logits_parity_mse_only_keys(bits, B, Hq, Hkv, cap, lens):
    """TurboQuant-MSE keys (b-bit stage 1, no QJL term): est = n <q', yhat>."""
    ocb, gcb = pair(128, bits, kind="mse")
    rows = B * Hkv * cap
    x = wl.gaussian_outlier_keys(rows, 128)
    code, img = oracle_cache(ocb, rows, x.astype(np.float64))
    q = wl.queries((B, Hq, 128), name="tiny_q")
    ref = estimate.logits(ocb, code, q.astype(np.float64), lens, Hkv, cap)
    ws = torch.empty(tq.tq_logits_workspace(gcb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, cap), float("nan"), device="cuda")
    tq.tq_logits(gcb, torch.from_numpy(img).cuda(), B, Hq, Hkv, cap, torch.tensor(lens, dtype=torch.int32, device="cuda"),
                 torch.from_numpy(q).cuda(), out, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        L = lens[b]
        assert np.all(np.isnan(got[b, :, L:]))
        if L:
            rowwise_ok(got[b, :, :L], ref[b, :, :L])


@pytest.mark.parametrize("bits,extra", [(2, 32), (3, 32), (2, 64), (3, 64), (4, 32)])
@pytest.mark.parametrize("B,Hq,Hkv,cap,lens", [(1, 8, 2, 4096, [4096]), (3, 6, 3, 333, [333, 17, 0])])
def test_logits_parity_mixed_bits(bits, extra, B, Hq, Hkv, cap, lens):
    """Mixed-bit keys (2.5 / 3.5-bit points): the first `extra` rotated
    coordinates carry one more stage-1 bit."""
    ocb, gcb = pair(128, bits, extra=extra)
    rows = B * Hkv * cap
    x = wl.gaussian_outlier_keys(rows, 128)
    code, img = oracle_cache(ocb, rows, x.astype(np.float64))
    q = wl.queries((B, Hq, 128), name="tiny_q")
    ref = estimate.logits(ocb, code, q.astype(np.float64), lens, Hkv, cap)
    ws = torch.empty(tq.tq_logits_workspace(gcb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, cap), float("nan"), device="cuda")
    tq.tq_logits(gcb, torch.from_numpy(img).cuda(), B, Hq, Hkv, cap, torch.tensor(lens, dtype=torch.int32, device="cuda"),
                 torch.from_numpy(q).cuda(), out, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        L = lens[b]
        assert np.all(np.isnan(got[b, :, L:]))
        if L:
            rowwise_ok(got[b, :, :L], ref[b, :, :L])


def tiled_code(code, reps):
    """The oracle's code arrays repeated ``reps`` times along the rows."""
    n = code["n"].shape[0]
    return {k: (np.tile(v, (reps,) + (1,) * (v.ndim - 1)) if isinstance(v, np.ndarray) and v.shape[:1] == (n,) else v)
            for k, v in code.items()}


@pytest.mark.parametrize("bits", [3, 4])
def test_logits_long_context_every_position(bits):
    """Context 131072 for 2 sequences x 2 kv heads: chunks of more tiles than
    the staging ring holds, so stages are refilled.  The cache repeats 4096
    oracle-coded keys, so every one of the 2 x 8 x 131072 outputs has an
    oracle value (that of its source key)."""
    B, Hq, Hkv, cap, lens = 2, 8, 2, 131072, [131072, 100003]
    ocb, gcb = pair(128, bits)
    x = wl.gaussian_outlier_keys(4096, 128)
    code = quant.quantize(ocb, x.astype(np.float64))
    reps = B * Hkv * cap // 4096
    img = layout.write_cache(ocb, B * Hkv * cap, tiled_code(code, reps))
    q = wl.queries((B, Hq, 128), name="tiny_q")
    G = Hq // Hkv
    ref = np.stack([estimate.estimate(ocb, q[b].astype(np.float64), code) for b in range(B)])   # [B, Hq, 4096]
    ws = torch.empty(tq.tq_logits_workspace(gcb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, cap), float("nan"), device="cuda")
    tq.tq_logits(gcb, torch.from_numpy(img).cuda(), B, Hq, Hkv, cap, torch.tensor(lens, dtype=torch.int32, device="cuda"),
                 torch.from_numpy(q).cuda(), out, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        L = lens[b]
        assert np.all(np.isnan(got[b, :, L:]))
        for h in range(Hq):
            # rows of (b, kv head h // G) start at a multiple of 4096: position t holds key t mod 4096
            want = np.tile(ref[b, h], cap // 4096)[:L]
            rowwise_ok(got[b, h, :L][None], want[None])


@pytest.mark.parametrize("kb,vb,mode", [(3, 3, "scalar"), (4, 3, "scalar"), (2, 2, "scalar"), (3, 4, "scalar"),
                                        (3, 1, "scalar"), (3, 3, "polar"), (4, 2, "polar"), (2, 4, "polar")])
@pytest.mark.parametrize("B,Hq,Hkv,cap,lens", [(2, 8, 2, 2048, [2048, 1500]), (3, 4, 1, 300, [300, 1, 0]),
                                               (1, 4, 4, 5000, [4999]), (2, 16, 2, 1024, [1024, 700]),
                                               (1, 8, 1, 300, [299])])
def test_attention_parity(kb, vb, mode, B, Hq, Hkv, cap, lens):
    okc, gkc = pair(128, kb, "prod", mode=mode)
    ovc, gvc = pair(128, vb, "mse", mode=mode, seed_pi=1)
    rows = B * Hkv * cap
    K = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="keys") for h in range(B * Hkv)])
    V = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="values") for h in range(B * Hkv)])
    kcode, kimg = oracle_cache(okc, rows, K.astype(np.float64))
    vcode, vimg = oracle_cache(ovc, rows, V.astype(np.float64))
    q = wl.queries((B, Hq, 128))
    scale = 1.0 / math.sqrt(128)
    ref = estimate.attention(okc, ovc, kcode, vcode, q.astype(np.float64), lens, Hkv, cap, scale)
    ws = torch.empty(tq.tq_decode_attention_workspace(gkc, B, Hq, Hkv, cap), dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    tq.tq_decode_attention(gkc, gvc, torch.from_numpy(kimg).cuda(), torch.from_numpy(vimg).cuda(), B, Hq, Hkv, cap,
                           torch.tensor(lens, dtype=torch.int32, device="cuda"), torch.from_numpy(q).cuda(), scale,
                           out, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        if lens[b] == 0:
            assert np.all(got[b] == 0)
        else:
            rowwise_ok(got[b], ref[b])


@pytest.mark.parametrize("kkind,kbits,kextra", [("mse", 3, 0), ("mse", 4, 0), ("mse", 2, 0), ("prod", 3, 32),
                                                ("prod", 4, 32), ("prod", 2, 64), ("prod", 4, 64)])
@pytest.mark.parametrize("vb", [3, 4])
@pytest.mark.parametrize("B,Hq,Hkv,cap,lens", [(2, 8, 2, 2048, [2048, 1500]), (3, 4, 1, 304, [300, 1, 0])])
def test_attention_parity_key_variants(kkind, kbits, kextra, vb, B, Hq, Hkv, cap, lens):
    """Decode attention over MSE-only keys (no QJL term) and over mixed-bit
    keys (the first `extra` rotated coordinates carry one more stage-1 bit),
    with 3- or 4-bit values."""
    okc, gkc = pair(128, kbits, kkind, extra=kextra)
    ovc, gvc = pair(128, vb, "mse", seed_pi=1)
    rows = B * Hkv * cap
    K = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="keys") for h in range(B * Hkv)])
    V = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="values") for h in range(B * Hkv)])
    kcode, kimg = oracle_cache(okc, rows, K.astype(np.float64))
    vcode, vimg = oracle_cache(ovc, rows, V.astype(np.float64))
    q = wl.queries((B, Hq, 128))
    scale = 1.0 / math.sqrt(128)
    ref = estimate.attention(okc, ovc, kcode, vcode, q.astype(np.float64), lens, Hkv, cap, scale)
    ws = torch.empty(tq.tq_decode_attention_workspace(gkc, B, Hq, Hkv, cap), dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    tq.tq_decode_attention(gkc, gvc, torch.from_numpy(kimg).cuda(), torch.from_numpy(vimg).cuda(), B, Hq, Hkv, cap,
                           torch.tensor(lens, dtype=torch.int32, device="cuda"), torch.from_numpy(q).cuda(), scale,
                           out, ws)
    torch.cuda.synchronize()
    tq.tq_check_device(gkc)
    got = out.cpu().numpy()
    for b in range(B):
        if lens[b] == 0:
            assert np.all(got[b] == 0)
        else:
            rowwise_ok(got[b], ref[b])


@pytest.mark.parametrize("kbits,kextra,vbits", [(3, 32, 3), (3, 0, 3), (2, 32, 2), (4, 0, 2), (4, 32, 3), (2, 0, 3)])
@pytest.mark.parametrize("B,Hq,Hkv,cap,lens", [(2, 8, 2, 2048, [2048, 1500]), (3, 4, 1, 304, [300, 1, 0])])
def test_attention_parity_mixed_bit_values(kbits, kextra, vbits, B, Hq, Hkv, cap, lens):
    """Decode attention over mixed-bit value caches (the first d/4 rotated
    coordinates carry one more stage-1 bit: the 2.5 / 3.5-bit points), with
    keys that carry the QJL term, mixed-bit or not."""
    okc, gkc = pair(128, kbits, "prod", extra=kextra)
    ovc, gvc = pair(128, vbits, "mse", extra=32, seed_pi=1)
    rows = B * Hkv * cap
    K = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="keys") for h in range(B * Hkv)])
    V = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="values") for h in range(B * Hkv)])
    kcode, kimg = oracle_cache(okc, rows, K.astype(np.float64))
    vcode, vimg = oracle_cache(ovc, rows, V.astype(np.float64))
    q = wl.queries((B, Hq, 128))
    scale = 1.0 / math.sqrt(128)
    ref = estimate.attention(okc, ovc, kcode, vcode, q.astype(np.float64), lens, Hkv, cap, scale)
    ws = torch.empty(tq.tq_decode_attention_workspace(gkc, B, Hq, Hkv, cap), dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    tq.tq_decode_attention(gkc, gvc, torch.from_numpy(kimg).cuda(), torch.from_numpy(vimg).cuda(), B, Hq, Hkv, cap,
                           torch.tensor(lens, dtype=torch.int32, device="cuda"), torch.from_numpy(q).cuda(), scale,
                           out, ws)
    torch.cuda.synchronize()
    tq.tq_check_device(gkc)
    got = out.cpu().numpy()
    for b in range(B):
        if lens[b] == 0:
            assert np.all(got[b] == 0)
        else:
            rowwise_ok(got[b], ref[b])


def test_attention_key_variants_unsupported_pairs():
    """MSE-only or mixed-bit keys with 1- or 2-bit values, mixed-bit values with
    MSE-only keys or at 1 bit, and any of these at a capacity that is not a
    multiple of 16 are rejected before any launch."""
    _, gk = pair(128, 3, "mse")
    _, gm = pair(128, 3, "prod", extra=32)
    _, gv2 = pair(128, 2, "mse", seed_pi=1)
    _, gv3 = pair(128, 3, "mse", seed_pi=1)
    _, gvx = pair(128, 3, "mse", extra=32, seed_pi=1)
    _, gvx1 = pair(128, 1, "mse", extra=32, seed_pi=1)
    _, gk3 = pair(128, 3, "prod")
    B, Hq, Hkv = 1, 4, 1
    sl = torch.tensor([10], dtype=torch.int32, device="cuda")
    q = torch.zeros((B, Hq, 128), device="cuda")
    out = torch.zeros((B, Hq, 128), device="cuda")
    for kcb, vcb, cap in ((gk, gv2, 64), (gm, gv2, 64), (gk, gv3, 40), (gm, gv3, 40), (gk, gvx, 64),
                          (gk3, gvx1, 64), (gk3, gvx, 40)):
        kc = torch.zeros(tq.cache_bytes(kcb, cap), dtype=torch.uint8, device="cuda")
        vc = torch.zeros(tq.cache_bytes(vcb, cap), dtype=torch.uint8, device="cuda")
        ws = torch.empty(tq.tq_decode_attention_workspace(kcb, B, Hq, Hkv, cap), dtype=torch.uint8, device="cuda")
        with pytest.raises(tq.TqError) as e:
            tq.tq_decode_attention(kcb, vcb, kc, vc, B, Hq, Hkv, cap, sl, q, 0.1, out, ws)
        assert e.value.status == tq.TQ_EUNSUPPORTED


def test_attention_long_context_ring_refill():
    """2 sequences x 8 kv heads at context 16384: chunks of more tiles than
    the staging ring holds.  Keys and values repeat 4096 oracle-coded rows;
    the oracle attends over the repeated codes in full."""
    B, Hq, Hkv, cap, lens = 2, 32, 8, 16384, [16384, 12001]
    okc, gkc = pair(128, 3, "prod")
    ovc, gvc = pair(128, 3, "mse", seed_pi=1)
    K = wl.llama_kv_slice(0, 0, 0, 4096, which="keys")
    V = wl.llama_kv_slice(0, 0, 0, 4096, which="values")
    reps = B * Hkv * cap // 4096
    kcode = tiled_code(quant.quantize(okc, K.astype(np.float64)), reps)
    vcode = tiled_code(quant.quantize(ovc, V.astype(np.float64)), reps)
    rows = B * Hkv * cap
    kimg = layout.write_cache(okc, rows, kcode)
    vimg = layout.write_cache(ovc, rows, vcode)
    q = wl.queries((B, Hq, 128))
    scale = 1.0 / math.sqrt(128)
    ref = estimate.attention(okc, ovc, kcode, vcode, q.astype(np.float64), lens, Hkv, cap, scale)
    ws = torch.empty(tq.tq_decode_attention_workspace(gkc, B, Hq, Hkv, cap), dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    tq.tq_decode_attention(gkc, gvc, torch.from_numpy(kimg).cuda(), torch.from_numpy(vimg).cuda(), B, Hq, Hkv, cap,
                           torch.tensor(lens, dtype=torch.int32, device="cuda"), torch.from_numpy(q).cuda(), scale,
                           out, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        rowwise_ok(got[b], ref[b])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,Hq,Hkv,cap,lens", [(1, 32, 8, 4096, [4096]), (3, 6, 3, 333, [333, 17, 0]),
                                               (2, 4, 4, 1001, [1000, 1001])])
def test_logits_dense_comparator(dtype, B, Hq, Hkv, cap, lens):
    """Unquantized logits (fp32 or bf16 keys) against the oracle's plain dot products."""
    from oracle import rng as orng
    K = np.stack([np.stack([wl.llama_kv_slice(0, h, 0, cap, which="keys") for h in range(Hkv)])
                  for _ in range(B)]).astype(np.float64)
    Kt = torch.from_numpy(K.astype(np.float32))
    if dtype == "bf16":
        Kt = Kt.to(torch.bfloat16)
        K = orng.round_bf16(K)
    q = wl.queries((B, Hq, 128))
    ref = estimate.dense_logits(K, q.astype(np.float64), lens, Hkv, cap)
    out = torch.full((B, Hq, cap), float("nan"), device="cuda")
    tq.tq_logits_dense(Kt.cuda(), B, Hq, Hkv, cap, torch.tensor(lens, dtype=torch.int32, device="cuda"),
                       torch.from_numpy(q).cuda(), out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        L = lens[b]
        assert np.all(np.isnan(got[b, :, L:]))
        if L:
            rowwise_ok(got[b, :, :L], ref[b, :, :L], tol=1e-4, med=1e-4)


def test_invalid_arguments_return_status_without_launch():
    _, gcb = pair(128, 3)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    kc = torch.zeros(tq.cache_bytes(gcb, 64), dtype=torch.uint8, device="cuda")
    q = torch.zeros(1, 4, 128, device="cuda")
    out = torch.zeros(1, 4, 64, device="cuda")
    sl = torch.tensor([64], dtype=torch.int32, device="cuda")
    with pytest.raises(tq.TqError) as e:
        tq.tq_logits(gcb, kc, 1, 4, 1, 64, sl, q, out, ws)       # workspace too small
    assert e.value.status == tq.TQ_ENOMEM
    ws = torch.empty(tq.tq_logits_workspace(gcb, 1, 4, 1), dtype=torch.uint8, device="cuda")
    with pytest.raises(tq.TqError) as e:
        tq.tq_logits(gcb, kc, 1, 6, 1, 64, sl, q, out, ws)       # G = 6: above 4, not a multiple of 4
    assert e.value.status == tq.TQ_EUNSUPPORTED
    with pytest.raises(tq.TqError) as e:
        tq.tq_logits(gcb, kc, 1, 20, 1, 64, sl, q, out, ws)      # G = 20 > 16
    assert e.value.status == tq.TQ_EUNSUPPORTED
    with pytest.raises(tq.TqError) as e:
        tq.tq_logits(gcb, kc, 1, 6, 4, 64, sl, q, out, ws)       # Hq not a multiple of Hkv
    assert e.value.status == tq.TQ_EINVAL
    with pytest.raises(tq.TqError) as e:
        tq.tq_quantize(gcb, kc, 64, q.view(-1, 128), 4, 129)     # d_in > d
    assert e.value.status == tq.TQ_EINVAL
    _, pcb = pair(128, 3, "mse", mode="polar")
    with pytest.raises(tq.TqError) as e:
        tq.tq_logits(pcb, kc, 1, 4, 1, 64, sl, q, out, ws)       # MSE-only keys in polar mode
    assert e.value.status == tq.TQ_EUNSUPPORTED
    with pytest.raises(tq.TqError) as e:                         # values of kind PROD
        tq.tq_decode_attention(gcb, gcb, kc, kc, 1, 4, 1, 64, sl, q, 0.1, out, ws)
    assert e.value.status == tq.TQ_EINVAL
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("bits,kind,extra", [(2, "prod", 0), (3, "prod", 0), (4, "prod", 0), (4, "mse", 0),
                                             (3, "prod", 32), (2, "prod", 64)])
@pytest.mark.parametrize("n", [1, 8, 128])
def test_quantize_decode_step_appends(dtype, bits, kind, extra, n):
    """A decode step's few rows (one CTA per row, coded while the previous
    kernel runs): the same bars as the batch paths, scattered destinations."""
    ocb, gcb = pair(128, bits, kind, "scalar", extra)
    x = wl.llama_kv_slice(0, 3, 0, n)
    xt = torch.from_numpy(x).cuda()
    if dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    x64 = xt.float().cpu().numpy().astype(np.float64)
    code = quant.quantize(ocb, x64)
    rows = n + 50
    perm = np.random.default_rng(n + bits).permutation(rows)[:n]
    cache = gpu_cache(gcb, rows)
    tq.tq_quantize(gcb, cache, rows, xt, n, 128, dst_rows=torch.from_numpy(perm.astype(np.int64)).cuda())
    tq.tq_check_device(gcb)
    got = read_back(ocb, rows, cache)
    bad = got["idx"][perm] != code["idx"]
    flips = bad.sum()
    nbits = code["idx"].size * ocb.b1
    if kind == "prod":
        flips += (got["sigma"][perm] != code["sigma"]).sum()
        nbits += code["sigma"].size
    assert flips <= max(1, 1e-3 * nbits)
    if bad.any():
        y, _ = quant.rotate(ocb, x64)
        t = ocb.t.astype(np.float64)
        tx = ocb.t_x.astype(np.float64) if extra else t
        for r, cidx in zip(*np.nonzero(bad)):
            tt = tx if cidx < extra else t
            assert np.min(np.abs(y[r, cidx] - tt)) < 1e-4 / math.sqrt(128)
    assert np.allclose(got["n16"][perm].astype(np.float64), np.linalg.norm(x64, axis=1), rtol=1e-3)
    if kind == "prod":
        assert np.allclose(got["g16"][perm].astype(np.float64), code["gamma"], rtol=2e-3, atol=1e-4)


@pytest.mark.parametrize("bits,kind,extra", [(2, "prod", 0), (3, "prod", 0), (4, "prod", 0), (3, "mse", 0),
                                             (4, "mse", 0), (3, "prod", 32), (2, "prod", 64)])
@pytest.mark.parametrize("n", [2048, 5000 + 37])
def test_quantize_tensor_core_path(bits, kind, extra, n):
    """bf16 batches of >= 2048 rows take the tcgen05 kernel: <= 0.1% differing
    bits against the oracle, scattered destination rows, ragged last tile."""
    ocb, gcb = pair(128, bits, kind, "scalar", extra)
    x = np.concatenate([wl.llama_kv_slice(0, h, 0, 4096) for h in range(2)])[:n]
    code = quant.quantize(ocb, x.astype(np.float64))
    rows = n + 100
    perm = np.random.default_rng(n).permutation(rows)[:n]
    cache = gpu_cache(gcb, rows)
    tq.tq_quantize(gcb, cache, rows, torch.from_numpy(x).cuda().to(torch.bfloat16), n, 128,
                   dst_rows=torch.from_numpy(perm.astype(np.int64)).cuda())
    tq.tq_check_device(gcb)
    got = read_back(ocb, rows, cache)
    g_idx = got["idx"][perm]
    flips = (g_idx != code["idx"]).sum()
    nbits = code["idx"].size * ocb.b1
    if kind == "prod":
        flips += (got["sigma"][perm] != code["sigma"]).sum()
        nbits += code["sigma"].size
    assert flips <= 1e-3 * nbits, flips / nbits
    n_ref = np.linalg.norm(x.astype(np.float64), axis=1)
    assert np.allclose(got["n16"][perm].astype(np.float64), n_ref, rtol=1e-3)
    if kind == "prod":
        assert np.allclose(got["g16"][perm].astype(np.float64), code["gamma"], rtol=2e-3, atol=1e-4)


@pytest.mark.parametrize("d,dtype", [(256, "f32"), (256, "bf16"), (128, "f32")])
@pytest.mark.parametrize("bits,kind", [(2, "prod"), (3, "prod"), (4, "prod"), (4, "mse")])
@pytest.mark.parametrize("n", [2048, 4096 + 77])
def test_quantize_tensor_core_path_tmem_operands(d, dtype, bits, kind, n):
    """Batches of >= 2048 rows that take the tcgen05 kernel with X in tensor
    memory: d = 256 (the search database, 200 coordinates zero-padded), fp32
    or bf16, and d = 128 fp32: <= 0.1% differing bits against the oracle,
    each differing code near a boundary, scattered destination rows, ragged
    last tile."""
    ocb, gcb = pair(d, bits, kind, "scalar", 0)
    d_in = 200 if d == 256 else 128
    x = wl.search_rows(n, "db") if d == 256 else np.concatenate(
        [wl.llama_kv_slice(0, h, 0, 4096) for h in range(2)])[:n]
    xt = torch.from_numpy(x).cuda()
    if dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    x64 = xt.float().cpu().numpy().astype(np.float64)
    code = quant.quantize(ocb, x64)
    rows = n + 100
    perm = np.random.default_rng(n + bits).permutation(rows)[:n]
    cache = gpu_cache(gcb, rows)
    tq.tq_quantize(gcb, cache, rows, xt, n, d_in, dst_rows=torch.from_numpy(perm.astype(np.int64)).cuda())
    tq.tq_check_device(gcb)
    got = read_back(ocb, rows, cache)
    g_idx = got["idx"][perm]
    bad = g_idx != code["idx"]
    flips = bad.sum()
    nbits = code["idx"].size * ocb.b1
    if kind == "prod":
        flips += (got["sigma"][perm] != code["sigma"]).sum()
        nbits += code["sigma"].size
    assert flips <= 1e-3 * nbits, flips / nbits
    if bad.any():
        y, _ = quant.rotate(ocb, x64)
        t = ocb.t.astype(np.float64)
        dist = np.min(np.abs(y[bad][:, None] - t[None, :]), axis=1)
        assert np.all(dist < 1e-4 / math.sqrt(d))
    n_ref = np.linalg.norm(x64, axis=1)
    assert np.allclose(got["n16"][perm].astype(np.float64), n_ref, rtol=1e-3)
    if kind == "prod":
        assert np.allclose(got["g16"][perm].astype(np.float64), code["gamma"], rtol=2e-3, atol=1e-4)


def polar_tie_distance(ocb, y):
    """Per level-ordered angle of unit rows y: how far (in the rotated space)
    the point sits from the nearest cell boundary of its level, i.e. the
    angular distance to the boundary times the radius of its node."""
    from oracle import polar
    tab = ocb.polar
    ang = polar.exact_angles(y)
    a, b = y[:, 0::2], y[:, 1::2]
    rho = np.hypot(a, b)
    radii = [rho]
    while rho.shape[1] > 1:
        rho = np.hypot(rho[:, 0::2], rho[:, 1::2])
        radii.append(rho)
    radii = np.concatenate(radii, axis=1)
    dist = np.empty_like(ang)
    off = 0
    for lev in range(1, tab.D + 1):
        cnt = tab.d >> lev
        bnd = tab.bound[lev].astype(np.float64)
        if lev == 1:                                   # the full circle wraps at 0 = 2 pi
            bnd = np.concatenate([[0.0], bnd, [2.0 * math.pi]])
        sl = slice(off, off + cnt)
        dist[:, sl] = np.min(np.abs(ang[:, sl, None] - bnd[None, None, :]), axis=2) * radii[:, sl]
        off += cnt
    return dist


@pytest.mark.parametrize("d,dtype,bits,kind", [(128, "bf16", 2, "prod"), (128, "bf16", 3, "prod"),
                                               (128, "bf16", 4, "prod"), (128, "f32", 3, "prod"),
                                               (128, "bf16", 1, "mse"), (128, "bf16", 3, "mse"),
                                               (128, "bf16", 4, "mse"), (128, "f32", 4, "mse"),
                                               (256, "f32", 3, "prod"), (256, "bf16", 4, "prod"),
                                               (256, "f32", 4, "mse")])
@pytest.mark.parametrize("n", [2048, 4096 + 37])
def test_quantize_polar_tensor_core_path(d, dtype, bits, kind, n):
    """Polar-mode batches of >= 2048 rows (tcgen05 rotation and sketch, the
    angle tree on the CUDA cores): <= 0.1% differing bits against the
    oracle, each differing angle code a near-tie (its point within 1e-4 /
    sqrt(d) of a cell boundary), scattered destinations, ragged last tile."""
    ocb, gcb = pair(d, bits, kind, "polar", 0)
    d_in = 200 if d == 256 else 128
    x = wl.search_rows(n, "db") if d == 256 else np.concatenate(
        [wl.llama_kv_slice(0, h, 0, 4096) for h in range(2)])[:n]
    xt = torch.from_numpy(x).cuda()
    if dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    x64 = xt.float().cpu().numpy().astype(np.float64)
    code = quant.quantize(ocb, x64)
    rows = n + 100
    perm = np.random.default_rng(n + bits).permutation(rows)[:n]
    cache = gpu_cache(gcb, rows)
    tq.tq_quantize(gcb, cache, rows, xt, n, d_in, dst_rows=torch.from_numpy(perm.astype(np.int64)).cuda())
    tq.tq_check_device(gcb)
    got = read_back(ocb, rows, cache)
    bad = got["idx"][perm] != code["idx"]
    flips = bad.sum()
    nbits = code["idx"].size * ocb.b1
    if kind == "prod":
        flips += (got["sigma"][perm] != code["sigma"]).sum()
        nbits += code["sigma"].size
    assert flips <= 1e-3 * nbits, flips / nbits
    if bad.any():
        y, _ = quant.rotate(ocb, x64)
        dist = polar_tie_distance(ocb, y)
        assert np.all(dist[bad] < 1e-4 / math.sqrt(d)), float(np.max(dist[bad]))
    n_ref = np.linalg.norm(x64, axis=1)
    assert np.allclose(got["n16"][perm].astype(np.float64), n_ref, rtol=1e-3)
    if kind == "prod":
        # a flipped angle code moves a whole subtree's reproduction, so the
        # residual norm is compared on the rows whose codes all agree
        same = ~bad.any(axis=1)
        assert same.mean() > 0.9
        assert np.allclose(got["g16"][perm][same].astype(np.float64), code["gamma"][same], rtol=2e-3, atol=1e-4)


@pytest.mark.parametrize("d,bits,kind", [(128, 4, "prod"), (128, 4, "mse"), (256, 3, "mse")])
def test_quantize_polar_exact_ties_take_the_upper_cell(d, bits, kind):
    """Level-1 pairs placed exactly on a boundary ray, and one ulp to either
    side of it: the fp32 screen of the sign test cannot decide these, so the
    exact fp64 products decide, and the codes equal the oracle's bit for bit
    (a zero determinant goes to the upper cell)."""
    ocb, gcb = pair(d, bits, kind, "polar", 0)
    tab = ocb.polar
    bc, bs = tab.bcos[1].astype(np.float32), tab.bsin[1].astype(np.float32)
    rng = np.random.default_rng(d + bits)
    n = 512
    y = np.empty((n, d), dtype=np.float32)
    for r in range(n):
        j = rng.integers(0, len(bc), size=d // 2)
        c, s_ = bc[j].copy(), bs[j].copy()
        nudge = rng.integers(-1, 2, size=d // 2)       # -1, 0, +1 ulp on the sine
        s_ = np.where(nudge > 0, np.nextafter(s_, np.float32(2)), np.where(nudge < 0, np.nextafter(s_, np.float32(-2)), s_))
        scale = np.float32(2.0) ** rng.integers(-8, 1, size=d // 2).astype(np.float32)   # exact scaling
        y[r, 0::2] = c * scale
        y[r, 1::2] = s_ * scale
    y /= np.float32(8.0)
    nrm = np.ones(n, dtype=np.float32)
    code = quant.encode_rotated(ocb, y.astype(np.float64), nrm.astype(np.float64))
    cache = gpu_cache(gcb, n)
    tq.tq_quantize_rotated(gcb, cache, n, torch.from_numpy(y).cuda(), torch.from_numpy(nrm).cuda(), n)
    tq.tq_check_device(gcb)
    got = read_back(ocb, n, cache)
    assert np.array_equal(got["idx"], code["idx"])


def kernels_of(fn):
    """Names of the CUDA kernels one call launches."""
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    return {e.name for e in prof.events() if e.device_type.name == "CUDA"}


@pytest.mark.parametrize("d,dtype,mode,n,kernel", [(128, "bf16", "scalar", 4096, "k_quantize_tc<"),
                                                   (128, "f32", "scalar", 4096, "k_quantize_tcx<128"),
                                                   (256, "f32", "scalar", 4096, "k_quantize_tcx<256"),
                                                   (256, "bf16", "scalar", 4096, "k_quantize_tcx<256"),
                                                   (128, "bf16", "polar", 4096, "k_quantize_tc<"),
                                                   (128, "f32", "polar", 4096, "k_quantize_tcx<128"),
                                                   (256, "f32", "polar", 4096, "k_quantize_tcx<256"),
                                                   (128, "bf16", "scalar", 8, "k_quantize_row<128>"),
                                                   (128, "bf16", "polar", 8, "k_quantize_simt<128>")])
def test_quantize_batches_take_the_tensor_core_kernels(d, dtype, mode, n, kernel):
    """Which kernel a batch takes: every batch of >= 2048 rows runs a tcgen05
    kernel (launch list recorded by the profiler); short batches run the
    row-wise CUDA-core kernels."""
    gcb = tq.Codebook(d, 3, tq.KIND_PROD, MODE[mode])
    d_in = 200 if d == 256 else 128
    x = torch.randn(n, d_in, device="cuda", generator=torch.Generator("cuda").manual_seed(d + n))
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    cache = gpu_cache(gcb, n)
    names = kernels_of(lambda: tq.tq_quantize(gcb, cache, n, x, n, d_in))
    tq.tq_check_device(gcb)
    assert any(kernel in nm for nm in names), names


def check_search(ocb, gcb, x, q, k, expect_fallbacks=None):
    """Top-k ids equal to the oracle's on the oracle's own packed database,
    except swaps among near-tied scores (oracle scores within 1e-5 relative);
    returns the number of queries the exact scan re-ran (-1: exact scan only)."""
    n_db, nq = x.shape[0], q.shape[0]
    code = quant.quantize(ocb, x.astype(np.float64))
    img = torch.from_numpy(layout.write_cache(ocb, n_db, code)).cuda()
    ref_ids, ref_sc = estimate.search(ocb, code, q.astype(np.float64), min(k, n_db))
    full = estimate.estimate(ocb, q.astype(np.float64), code)
    ws = torch.full((tq.tq_search_workspace(gcb, n_db, nq, k),), 0xFF, dtype=torch.uint8, device="cuda")
    ids = torch.full((nq, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((nq, k), float("nan"), device="cuda")
    tq.tq_search(gcb, img, n_db, torch.from_numpy(q).cuda(), nq, q.shape[1], k, ids, sc, ws)
    torch.cuda.synchronize()
    fallbacks = tq.tq_search_fallbacks(gcb, ws, k)
    assert tq.tq_check_device(gcb) is None
    gi, gs = ids.cpu().numpy(), sc.cpu().numpy()
    kk = min(k, n_db)
    assert np.all(gi[:, kk:] == -1)
    scale = np.max(np.abs(full))
    tol = 1e-5 * scale
    for r in range(nq):
        g_ids = gi[r, :kk]
        assert len(set(g_ids.tolist())) == kk and np.all(g_ids >= 0) and np.all(g_ids < n_db)
        # GPU scores are the estimator of the returned rows
        assert np.all(np.abs(gs[r, :kk] - full[r, g_ids]) <= tol)
        # a valid top-k: the oracle scores of the returned rows match the oracle's top-k scores
        assert np.all(np.abs(np.sort(full[r, g_ids])[::-1] - ref_sc[r]) <= tol)
        # identical ids except where the oracle's scores are near-tied
        for j in np.nonzero(g_ids != ref_ids[r])[0]:
            assert abs(full[r, g_ids[j]] - ref_sc[r, j]) <= tol
        # sorted by decreasing score
        assert np.all(np.diff(gs[r, :kk]) <= tol)
    if expect_fallbacks is not None:
        assert fallbacks == expect_fallbacks, fallbacks
    return fallbacks


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("n_db,nq,k", [(20013, 37, 10), (7, 5, 10), (4096, 8, 1), (50000, 300, 16)])
def test_search_parity(bits, n_db, nq, k):
    """d = 256, k <= 16: tensor-core candidates and exact re-ranking; on this
    data every query's top k is certified, so the exact scan re-runs none."""
    ocb, gcb = pair(256, bits)
    check_search(ocb, gcb, wl.search_rows(n_db, "db"), wl.search_rows(nq, "search_q"), k, expect_fallbacks=0)


@pytest.mark.parametrize("bits", [2, 4])
def test_search_parity_exact_scan_for_large_k(bits):
    """k > 16 runs the exact scan for every query."""
    ocb, gcb = pair(256, bits)
    check_search(ocb, gcb, wl.search_rows(6000, "db"), wl.search_rows(19, "search_q"), 20, expect_fallbacks=-1)


@pytest.mark.parametrize("bits", [2, 4])
def test_search_uncertified_queries_fall_back_to_the_exact_scan(bits):
    """40 consecutive copies of a query's best-scoring row inside one 128-row
    tile put 40 equal scores at the top of one scan part: its list of 32
    candidates is all ties, so it cannot prove the top 10 and the query is
    re-run by the exact scan; the result is still the oracle's."""
    ocb, gcb = pair(256, bits)
    x = wl.search_rows(9000, "db")
    q = wl.search_rows(12, "search_q")
    est = estimate.estimate(ocb, q.astype(np.float64), quant.quantize(ocb, x.astype(np.float64)))
    for j, tile in enumerate((8, 20, 40, 60)):   # queries 0..3
        best = int(np.argmax(est[j]))
        x[128 * tile + 10:128 * tile + 50] = x[best]
    n = check_search(ocb, gcb, x, q, 10)
    assert n >= 4, n
