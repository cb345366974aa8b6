"""GPU parity of the outlier-channel split (keys whose outlier channels form
their own group, one bit wider, with its own rotation, sketch and norms).

Same bars as the other parity tests: codes bit-exact from identical rotated
fp32 rows (signs up to near-ties, gamma within one fp16 ulp); end to end at
most 0.1% differing bits, each differing code near a boundary of its group's
codebook; logits and decode attention scored by the GPU on the oracle's own
packed cache, per row max |diff| <= 1e-3 max |ref| and median relative error
<= 1e-4.
"""
import math

import numpy as np
import pytest
import torch

from decode_attention_21_b300 import tq
from decode_attention_21_b300 import workloads as wl
from oracle import estimate, quant, split

pytestmark = pytest.mark.gpu


def outlier_channels(x, E):
    """The E channels of largest RMS over the rows x (the caller's choice)."""
    return np.argsort(-np.sqrt(np.mean(np.asarray(x, np.float64) ** 2, axis=0)), kind="stable")[:E]


def split_pair(bits, out, seed_pi=1, seed_s=2):
    scb = split.SplitCodebook(128, bits, out, seed_pi=seed_pi, seed_s=seed_s)
    gcb = tq.Codebook(128, bits, tq.KIND_PROD, tq.MODE_SCALAR, seed_pi, seed_s, outliers=out)
    return scb, gcb


def keys(rows, seed_head=0):
    return np.concatenate([wl.llama_kv_slice(0, h, 0, min(rows, 4096), which="keys")
                           for h in range(seed_head, seed_head + (rows + 4095) // 4096)])[:rows]


def sign_ties(g, c):
    sn = np.linalg.norm(g.S, axis=1)
    return np.abs(c["z"]) < 1e-5 * c["gamma"][:, None] * sn[None, :]


@pytest.mark.parametrize("E,bits", [(32, 2), (64, 2), (32, 3), (64, 3), (32, 4)])
def test_split_quantize_rotated_bit_exact(E, bits):
    n = 1000 + 37
    x = np.random.default_rng(E + bits).standard_normal((n, 128)) * 3.0
    out = np.random.default_rng(bits).choice(128, size=E, replace=False)
    x[:, out] *= 8.0
    scb, gcb = split_pair(bits, out)
    y, nrm = split.rotate(scb, x)
    y32, n32 = y.astype(np.float32), nrm.astype(np.float32)
    code = split.encode_rotated(scb, y32.astype(np.float64), n32.astype(np.float64))
    rows = n + 5
    perm = np.random.default_rng(1).permutation(rows)[:n]
    cache = torch.zeros(tq.cache_bytes(gcb, rows), dtype=torch.uint8, device="cuda")
    assert tq.cache_bytes(gcb, rows) == split.cache_bytes(scb, rows)
    tq.tq_quantize_rotated(gcb, cache, rows, torch.from_numpy(y32).cuda(), torch.from_numpy(n32).cuda(), n,
                           dst_rows=torch.from_numpy(perm.astype(np.int64)).cuda())
    torch.cuda.synchronize()
    got = split.read_cache(scb, rows, cache.cpu().numpy(), perm)["groups"]
    for g, c, w in zip(scb.groups, code["groups"], got):
        assert np.array_equal(w["idx"], c["idx"])
        assert np.array_equal(w["n16"], c["n16"])
        assert not np.any((w["sigma"] != c["sigma"]) & ~sign_ties(g, c))
        g16 = w["g16"].astype(np.float64)
        assert np.all(np.abs(g16 - c["g16"].astype(np.float64)) <= np.spacing(c["g16"]).astype(np.float64) * 1.01)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("E,bits,n", [(32, 2, 4096), (64, 3, 20000), (32, 3, 100)])
def test_split_quantize_end_to_end(dtype, E, bits, n):
    # up to 16384 rows take the short-batch kernel (one CTA per row), more
    # the row-per-warp kernel
    x = keys(n)
    out = outlier_channels(x, E)
    scb, gcb = split_pair(bits, out)
    xt = torch.from_numpy(x).cuda()
    if dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    x64 = xt.float().cpu().numpy().astype(np.float64)
    code = split.quantize(scb, x64)
    cache = torch.zeros(tq.cache_bytes(gcb, n), dtype=torch.uint8, device="cuda")
    tq.tq_quantize(gcb, cache, n, xt, n, 128)
    torch.cuda.synchronize()
    got = split.read_cache(scb, n, cache.cpu().numpy())["groups"]
    flips = nbits = 0
    y, _ = split.rotate(scb, x64)
    cols = (slice(0, E), slice(E, 128))
    for g, c, w, sl in zip(scb.groups, code["groups"], got, cols):
        bad = w["idx"] != c["idx"]
        flips += bad.sum() + (w["sigma"] != c["sigma"]).sum()
        nbits += c["idx"].size * g.b1 + c["sigma"].size
        if bad.any():
            t = g.t.astype(np.float64)
            dist = np.min(np.abs(y[:, sl][bad][:, None] - t[None, :]), axis=1)
            assert np.all(dist < 1e-4 / math.sqrt(g.d))
        assert np.allclose(w["n16"].astype(np.float64), c["n16"].astype(np.float64), rtol=2e-3)
    assert flips <= 1e-3 * nbits


def rowwise_ok(got, ref, tol=1e-3, med=1e-4):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref), axis=-1, keepdims=True)
    assert np.all(np.abs(got - ref) <= tol * scale + 1e-30), float(np.max(np.abs(got - ref) / scale))
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3 * scale)
    assert np.median(rel) <= med, float(np.median(rel))


@pytest.mark.parametrize("E,bits", [(32, 2), (64, 2), (32, 3), (64, 3), (32, 4), (64, 4)])
@pytest.mark.parametrize("B,Hq,Hkv,cap,lens", [(2, 8, 2, 1024, [1024, 700]), (3, 6, 3, 333, [333, 17, 0]),
                                               (1, 16, 2, 256, [250])])
def test_split_logits_parity(E, bits, B, Hq, Hkv, cap, lens):
    # capacity 333 takes the register-path kernel, multiples of 16 the staged one
    rows = B * Hkv * cap
    x = keys(rows)
    out = outlier_channels(x, E)
    scb, gcb = split_pair(bits, out)
    code = split.quantize(scb, x.astype(np.float64))
    img = split.write_cache(scb, rows, code)
    q = wl.queries((B, Hq, 128), name="tiny_q")
    ref = estimate.logits(scb, code, q.astype(np.float64), lens, Hkv, cap)
    ws = torch.empty(tq.tq_logits_workspace(gcb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    res = torch.full((B, Hq, cap), float("nan"), device="cuda")
    tq.tq_logits(gcb, torch.from_numpy(img).cuda(), B, Hq, Hkv, cap, torch.tensor(lens, dtype=torch.int32, device="cuda"),
                 torch.from_numpy(q).cuda(), res, ws)
    torch.cuda.synchronize()
    tq.tq_check_device(gcb)
    got = res.cpu().numpy()
    for b in range(B):
        L = lens[b]
        assert np.all(np.isnan(got[b, :, L:]))
        if L:
            rowwise_ok(got[b, :, :L], ref[b, :, :L])


@pytest.mark.parametrize("E,bits", [(32, 2), (64, 3), (32, 4)])
@pytest.mark.parametrize("vb", [3, 4])
@pytest.mark.parametrize("B,Hq,Hkv,cap,lens", [(2, 8, 2, 2048, [2048, 1500]), (3, 4, 1, 304, [300, 1, 0]),
                                               (1, 16, 2, 512, [500])])
def test_split_attention_parity(E, bits, vb, B, Hq, Hkv, cap, lens):
    rows = B * Hkv * cap
    K = keys(rows)
    V = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="values") for h in range(B * Hkv)])
    out = outlier_channels(K, E)
    scb, gkc = split_pair(bits, out)
    ovc = quant.Codebook(128, vb, "mse", seed_pi=1)
    gvc = tq.Codebook(128, vb, tq.KIND_MSE, tq.MODE_SCALAR, 1, 2)
    kcode = split.quantize(scb, K.astype(np.float64))
    kimg = split.write_cache(scb, rows, kcode)
    from oracle import layout
    vcode = quant.quantize(ovc, V.astype(np.float64))
    vimg = layout.write_cache(ovc, rows, vcode)
    q = wl.queries((B, Hq, 128))
    scale = 1.0 / math.sqrt(128)
    ref = estimate.attention(scb, ovc, kcode, vcode, q.astype(np.float64), lens, Hkv, cap, scale)
    ws = torch.empty(tq.tq_decode_attention_workspace(gkc, B, Hq, Hkv, cap), dtype=torch.uint8, device="cuda")
    res = torch.full((B, Hq, 128), float("nan"), device="cuda")
    tq.tq_decode_attention(gkc, gvc, torch.from_numpy(kimg).cuda(), torch.from_numpy(vimg).cuda(), B, Hq, Hkv, cap,
                           torch.tensor(lens, dtype=torch.int32, device="cuda"), torch.from_numpy(q).cuda(), scale,
                           res, ws)
    torch.cuda.synchronize()
    tq.tq_check_device(gkc)
    got = res.cpu().numpy()
    for b in range(B):
        if lens[b] == 0:
            assert np.all(got[b] == 0)
        else:
            rowwise_ok(got[b], ref[b])


def test_split_keys_rejected_where_not_scored():
    out = np.arange(32)
    gcb = tq.Codebook(128, 3, tq.KIND_PROD, tq.MODE_SCALAR, 1, 2, outliers=out)
    gvc = tq.Codebook(128, 3, tq.KIND_MSE, tq.MODE_SCALAR, 1, 2)
    # decode attention over split keys needs a capacity that is a multiple of 16
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    kc = torch.zeros(tq.cache_bytes(gcb, 100), dtype=torch.uint8, device="cuda")
    vc = torch.zeros(tq.cache_bytes(gvc, 100), dtype=torch.uint8, device="cuda")
    with pytest.raises(tq.TqError) as e:
        tq.tq_decode_attention(gcb, gvc, kc, vc, 1, 4, 1, 100, torch.tensor([100], dtype=torch.int32, device="cuda"),
                               torch.zeros(1, 4, 128, device="cuda"), 0.1, torch.zeros(1, 4, 128, device="cuda"), ws)
    assert e.value.status == tq.TQ_EUNSUPPORTED


@pytest.mark.parametrize("ps", [16, 256])
def test_split_logits_paged_equals_contiguous(ps):
    # the paged staged kernel copies 8-byte norm entries per page run
    B, Hq, Hkv = 2, 8, 2
    max_pages = -(-700 // ps)
    cap = max_pages * ps
    lens = [cap, 333]
    num_pages = B * max_pages + 3
    rows = B * Hkv * cap
    x = keys(rows)
    scb, gcb = split_pair(3, outlier_channels(x, 32))
    code = split.quantize(scb, x.astype(np.float64))
    table = wl.block_table(B, max_pages, num_pages, ps, lens)
    # physical row of every live logical row; other physical rows hold valid unrelated rows
    rows_p = num_pages * Hkv * ps
    filler = np.random.default_rng(5).integers(0, rows, size=rows_p)
    log, phys = [], []
    for b in range(B):
        t = np.arange(lens[b])
        for h in range(Hkv):
            log.append((b * Hkv + h) * cap + t)
            phys.append((table[b, t // ps].astype(np.int64) * Hkv + h) * ps + t % ps)
    log, phys = np.concatenate(log), np.concatenate(phys)
    pcode = {"groups": []}
    for c in code["groups"]:
        pc = {k: v[filler].copy() for k, v in c.items() if isinstance(v, np.ndarray) and v.shape[:1] == (rows,)}
        for k in pc:
            pc[k][phys] = c[k][log]
        pcode["groups"].append(pc)
    img_c = split.write_cache(scb, rows, code)
    img_p = split.write_cache(scb, rows_p, pcode)
    q = wl.queries((B, Hq, 128), name="tiny_q")
    ref = estimate.logits(scb, code, q.astype(np.float64), lens, Hkv, cap)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    qd = torch.from_numpy(q).cuda()
    ws = torch.empty(tq.tq_logits_workspace(gcb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    out_c = torch.full((B, Hq, cap), float("nan"), device="cuda")
    out_p = torch.full((B, Hq, cap), float("nan"), device="cuda")
    tq.tq_logits(gcb, torch.from_numpy(img_c).cuda(), B, Hq, Hkv, cap, sl, qd, out_c, ws)
    tq.tq_logits_paged(gcb, torch.from_numpy(img_p).cuda(), num_pages, ps, torch.from_numpy(table).cuda(), B, Hq,
                       Hkv, sl, qd, out_p, ws)
    torch.cuda.synchronize()
    tq.tq_check_device(gcb)
    got_c, got_p = out_c.cpu().numpy(), out_p.cpu().numpy()
    for b in range(B):
        L = lens[b]
        assert np.array_equal(got_p[b, :, :L], got_c[b, :, :L])
        rowwise_ok(got_p[b, :, :L], ref[b, :, :L])
