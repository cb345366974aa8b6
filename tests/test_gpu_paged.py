"""GPU parity of the paged caches and the in-place decode loop.

A paged cache holds the same packed rows as a contiguous one, scattered over
pages named by a block table.  The arithmetic is unchanged, so:

* paged logits and attention equal the contiguous calls bit for bit on a
  cache holding the same rows, and match the oracle (same bar as the
  contiguous parity tests: per-row max |diff| <= 1e-3 * max |oracle|,
  median relative error <= 1e-4);
* table entries past a sequence's last page are -1 here: reading one would
  raise the out-of-cache flag, which every test checks is clear;
* a decode loop captured once in a CUDA graph (advance the lengths, append
  the step's key and value, attend) and replayed step after step writes the
  same packed rows as the contiguous path, attends bit-identically to it, and
  matches the oracle's attention over the oracle's own codes of the same
  keys and values.
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


def pair(bits, kind="prod", mode="scalar", seed_pi=1, seed_s=2):
    ocb = quant.Codebook(128, bits, kind=kind, mode=mode, seed_pi=seed_pi, seed_s=seed_s)
    gcb = tq.Codebook(128, bits, KIND[kind], MODE[mode], seed_pi, seed_s)
    return ocb, gcb


def rowwise_ok(got, ref, tol=1e-3, med=1e-4):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref), axis=-1, keepdims=True)
    assert np.all(np.abs(got - ref) <= tol * scale + 1e-30), float(np.max(np.abs(got - ref) / scale))
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3 * scale)
    assert np.median(rel) <= med, float(np.median(rel))


def physical_rows(table, B, Hkv, cap, ps, lens):
    """Physical row of every live logical row (b, h, t < lens[b]), in logical
    order (b*Hkv + h)*cap + t, and the logical indices themselves."""
    log, phys = [], []
    for b in range(B):
        t = np.arange(lens[b])
        for h in range(Hkv):
            log.append((b * Hkv + h) * cap + t)
            phys.append((table[b, t // ps].astype(np.int64) * Hkv + h) * ps + t % ps)
    return np.concatenate(log), np.concatenate(phys)


def paged_image(ocb, code, B, Hkv, cap, ps, table, num_pages, lens):
    """Byte image of a paged cache holding the live logical rows of ``code``;
    every other physical row holds a valid but unrelated code row."""
    rows_total = num_pages * Hkv * ps
    n = code["n"].shape[0]
    filler = np.random.default_rng(7).integers(0, n, size=rows_total)
    phys_code = {k: (v[filler] if isinstance(v, np.ndarray) and v.shape[:1] == (n,) else v) for k, v in code.items()}
    log, phys = physical_rows(table, B, Hkv, cap, ps, lens)
    for k, v in code.items():
        if isinstance(v, np.ndarray) and v.shape[:1] == (n,):
            phys_code[k][phys] = v[log]
    return layout.write_cache(ocb, rows_total, phys_code)


def check_clear(gcb):
    tq.tq_check_device(gcb)   # raises on a bounded-wait timeout or an out-of-cache access


@pytest.mark.parametrize("bits,kind,mode", [(3, "prod", "scalar"), (4, "prod", "scalar"), (2, "prod", "scalar"),
                                             (3, "mse", "scalar"), (3, "prod", "polar"), (4, "prod", "polar")])
@pytest.mark.parametrize("ps", [16, 48, 128, 256])
def test_logits_paged_equals_contiguous_and_oracle(bits, kind, mode, ps):
    B, Hq, Hkv = 3, 6, 3
    max_pages = -(-1100 // ps)
    cap = max_pages * ps
    lens = [cap, 517, 0]
    num_pages = B * max_pages + 5
    ocb, gcb = pair(bits, kind, mode)
    rows = B * Hkv * cap
    x = wl.gaussian_outlier_keys(rows, 128)
    code = quant.quantize(ocb, x.astype(np.float64))
    table = wl.block_table(B, max_pages, num_pages, ps, lens)
    img_c = layout.write_cache(ocb, rows, code)
    img_p = paged_image(ocb, code, B, Hkv, cap, ps, table, num_pages, lens)
    q = wl.queries((B, Hq, 128), name="tiny_q")
    ref = estimate.logits(ocb, code, q.astype(np.float64), lens, Hkv, cap)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    qd = torch.from_numpy(q).cuda()
    ws = torch.empty(tq.tq_logits_workspace(gcb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    out_c = torch.full((B, Hq, cap), float("nan"), device="cuda")
    out_p = torch.full((B, Hq, cap), float("nan"), device="cuda")
    tq.tq_logits(gcb, torch.from_numpy(img_c).cuda(), B, Hq, Hkv, cap, sl, qd, out_c, ws)
    tq.tq_logits_paged(gcb, torch.from_numpy(img_p).cuda(), num_pages, ps, torch.from_numpy(table).cuda(), B, Hq,
                       Hkv, sl, qd, out_p, ws)
    torch.cuda.synchronize()
    check_clear(gcb)
    got_c, got_p = out_c.cpu().numpy(), out_p.cpu().numpy()
    for b in range(B):
        L = lens[b]
        assert np.all(np.isnan(got_p[b, :, L:]))
        assert np.array_equal(got_p[b, :, :L], got_c[b, :, :L])
        if L:
            rowwise_ok(got_p[b, :, :L], ref[b, :, :L])


@pytest.mark.parametrize("kb,vb,mode", [(3, 3, "scalar"), (4, 3, "scalar"), (2, 4, "scalar"), (3, 3, "polar")])
@pytest.mark.parametrize("ps", [16, 64])
def test_attention_paged_equals_contiguous_and_oracle(kb, vb, mode, ps):
    B, Hq, Hkv = 3, 8, 2
    max_pages = -(-2000 // ps)
    cap = max_pages * ps
    lens = [cap, 1001, 0]
    num_pages = B * max_pages + 3
    okc, gkc = pair(kb, "prod", mode)
    ovc, gvc = pair(vb, "mse", mode, seed_pi=1)
    rows = B * Hkv * cap
    K = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="keys") for h in range(B * Hkv)])
    V = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="values") for h in range(B * Hkv)])
    kcode = quant.quantize(okc, K.astype(np.float64))
    vcode = quant.quantize(ovc, V.astype(np.float64))
    table = wl.block_table(B, max_pages, num_pages, ps, lens)
    q = wl.queries((B, Hq, 128))
    scale = 1.0 / math.sqrt(128)
    ref = estimate.attention(okc, ovc, kcode, vcode, q.astype(np.float64), lens, Hkv, cap, scale)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    qd = torch.from_numpy(q).cuda()
    ws = torch.empty(tq.tq_decode_attention_workspace(gkc, B, Hq, Hkv, cap), dtype=torch.uint8, device="cuda")
    out_c = torch.full((B, Hq, 128), float("nan"), device="cuda")
    out_p = torch.full((B, Hq, 128), float("nan"), device="cuda")
    tq.tq_decode_attention(gkc, gvc, torch.from_numpy(layout.write_cache(okc, rows, kcode)).cuda(),
                           torch.from_numpy(layout.write_cache(ovc, rows, vcode)).cuda(), B, Hq, Hkv, cap, sl, qd,
                           scale, out_c, ws)
    tq.tq_decode_attention_paged(gkc, gvc,
                                 torch.from_numpy(paged_image(okc, kcode, B, Hkv, cap, ps, table, num_pages, lens)).cuda(),
                                 torch.from_numpy(paged_image(ovc, vcode, B, Hkv, cap, ps, table, num_pages, lens)).cuda(),
                                 num_pages, ps, torch.from_numpy(table).cuda(), B, Hq, Hkv, sl, qd, scale, out_p, ws)
    torch.cuda.synchronize()
    check_clear(gkc)
    got_c, got_p = out_c.cpu().numpy(), out_p.cpu().numpy()
    assert np.array_equal(got_p, got_c)
    for b in range(B):
        if lens[b] == 0:
            assert np.all(got_p[b] == 0)
        else:
            rowwise_ok(got_p[b], ref[b])


@pytest.mark.parametrize("mode", ["scalar", "polar"])
def test_decode_loop_in_a_cuda_graph(mode):
    """Prefill by tq_quantize into the pages, then 24 decode steps, each one
    replay of a graph captured once: advance the lengths by one, append the
    step's key and value (tq_append_paged), attend over the paged caches."""
    B, Hq, Hkv, ps, max_pages = 3, 8, 2, 32, 10
    cap = max_pages * ps
    prefill = [37, 5, 0]
    steps = 24
    final = [L + steps for L in prefill]
    num_pages = sum(-(-L // ps) for L in final) + 2
    okc, gkc = pair(3, "prod", mode)
    ovc, gvc = pair(3, "mse", mode, seed_pi=1)
    rows_total = num_pages * Hkv * ps
    table = wl.block_table(B, max_pages, num_pages, ps, final)
    # every key and value of every sequence: logical row (b*Hkv + h)*cap + t
    K = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="keys") for h in range(B * Hkv)])
    V = np.concatenate([wl.llama_kv_slice(0, h, 0, cap, which="values") for h in range(B * Hkv)])
    Kd, Vd = torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda()
    kc = torch.zeros(tq.cache_bytes(gkc, rows_total), dtype=torch.uint8, device="cuda")
    vc = torch.zeros(tq.cache_bytes(gvc, rows_total), dtype=torch.uint8, device="cuda")
    bt = torch.from_numpy(table).cuda()
    # prefill through explicit destination rows
    log, phys = physical_rows(table, B, Hkv, cap, ps, prefill)
    idx = torch.from_numpy(log).cuda()
    dst = torch.from_numpy(phys).cuda()
    tq.tq_quantize(gkc, kc, rows_total, Kd[idx].contiguous(), len(log), 128, dst_rows=dst)
    tq.tq_quantize(gvc, vc, rows_total, Vd[idx].contiguous(), len(log), 128, dst_rows=dst)
    sl = torch.tensor(prefill, dtype=torch.int32, device="cuda")
    kin = torch.zeros((B, Hkv, 128), device="cuda")
    vin = torch.zeros((B, Hkv, 128), device="cuda")
    qin = torch.zeros((B, Hq, 128), device="cuda")
    out = torch.zeros((B, Hq, 128), device="cuda")
    ws = torch.empty(tq.tq_decode_attention_workspace(gkc, B, Hq, Hkv, cap), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(128)
    Q = wl.queries((steps, B, Hq, 128))

    def step_inputs(i):
        # token prefill[b] + i of every (b, h)
        t = torch.tensor([prefill[b] + i for b in range(B)], device="cuda")
        rows = (torch.arange(B, device="cuda")[:, None] * Hkv + torch.arange(Hkv, device="cuda")[None, :]) * cap \
            + t[:, None]
        kin.copy_(Kd[rows])
        vin.copy_(Vd[rows])
        qin.copy_(torch.from_numpy(Q[i]).cuda())

    s = torch.cuda.Stream()

    def step():
        tq.tq_advance_lengths(sl, B, 1, stream=s)
        tq.tq_append_paged(gkc, kc, num_pages, ps, bt, B, Hkv, sl, kin, 128, stream=s)
        tq.tq_append_paged(gvc, vc, num_pages, ps, bt, B, Hkv, sl, vin, 128, stream=s)
        tq.tq_decode_attention_paged(gkc, gvc, kc, vc, num_pages, ps, bt, B, Hq, Hkv, sl, qin, scale, out, ws,
                                     stream=s)

    torch.cuda.synchronize()
    # the first step runs eagerly (the attention's first call does one-time setup), the rest replay a graph
    outs = []
    with torch.cuda.stream(s):
        step_inputs(0)
        step()
        s.synchronize()
        outs.append(out.clone())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        for i in range(1, steps):
            step_inputs(i)
            g.replay()
            outs.append(out.clone())
    torch.cuda.synchronize()
    check_clear(gkc)
    check_clear(gvc)
    assert sl.cpu().tolist() == final
    # contiguous path on the same keys and values (same per-row quantize kernel)
    live_log, live_phys = physical_rows(table, B, Hkv, cap, ps, final)
    rows_c = B * Hkv * cap
    kcc = torch.zeros(tq.cache_bytes(gkc, rows_c), dtype=torch.uint8, device="cuda")
    vcc = torch.zeros(tq.cache_bytes(gvc, rows_c), dtype=torch.uint8, device="cuda")
    li = torch.from_numpy(live_log).cuda()
    tq.tq_quantize(gkc, kcc, rows_c, Kd[li].contiguous(), len(live_log), 128, dst_rows=li)
    tq.tq_quantize(gvc, vcc, rows_c, Vd[li].contiguous(), len(live_log), 128, dst_rows=li)
    # the pages hold exactly the packed rows of the contiguous cache
    for gcb, paged, contig, nb in ((gkc, kc, kcc, 4), (gvc, vc, vcc, 2)):
        assert torch.equal(packed_rows(gcb, paged, rows_total, live_phys, nb),
                           packed_rows(gcb, contig, rows_c, live_log, nb))
    # the oracle codes the same keys and values itself; the loop's codes
    # differ from them at most in rare boundary cases (fp32 vs fp64 rotation)
    kcode = quant.quantize(okc, K.astype(np.float64))
    vcode = quant.quantize(ovc, V.astype(np.float64))
    for ocb, paged in ((okc, kc), (ovc, vc)):
        got = layout.read_cache(ocb, rows_total, paged.cpu().numpy(), row_ids=live_phys)
        ref_idx = (kcode if ocb is okc else vcode)["idx"][live_log]
        assert (got["idx"] != ref_idx).sum() <= 1e-3 * ref_idx.size
    wsc = torch.empty_like(ws)
    outc = torch.zeros_like(out)
    for i in range(steps):
        lens_i = [prefill[b] + i + 1 for b in range(B)]
        sli = torch.tensor(lens_i, dtype=torch.int32, device="cuda")
        tq.tq_decode_attention(gkc, gvc, kcc, vcc, B, Hq, Hkv, cap, sli, torch.from_numpy(Q[i]).cuda(), scale, outc,
                               wsc)
        torch.cuda.synchronize()
        assert torch.equal(outs[i], outc), i
        ref = estimate.attention(okc, ovc, kcode, vcode, Q[i].astype(np.float64), lens_i, Hkv, cap, scale)
        got = outs[i].cpu().numpy()
        for b in range(B):
            rowwise_ok(got[b], ref[b])


def packed_rows(gcb, buf, rows_total, ids, nb):
    """Records and norm entries of rows ``ids`` of a cache buffer, as bytes."""
    rb = tq.record_bytes(gcb)
    off = (rows_total * rb + 255) // 256 * 256
    ids = torch.from_numpy(np.asarray(ids, dtype=np.int64)).cuda()
    rec = buf[: rows_total * rb].view(rows_total, rb)[ids]
    nrm = buf[off: off + rows_total * nb].view(rows_total, nb)[ids]
    return torch.cat([rec, nrm], dim=1)


def test_paged_table_entry_outside_the_cache_is_flagged():
    """An entry naming a page past the pool is never dereferenced: the read
    goes to page 0, the append is skipped, and tq_check_device reports
    TQ_EINVAL (then the flag is clear again)."""
    B, Hq, Hkv, ps, max_pages, num_pages = 1, 4, 1, 16, 4, 4
    ocb, gcb = pair(3)
    table = np.array([[2, 0, num_pages + 5, 1]], dtype=np.int32)
    kc = torch.zeros(tq.cache_bytes(gcb, num_pages * Hkv * ps), dtype=torch.uint8, device="cuda")
    bt = torch.from_numpy(table).cuda()
    sl = torch.tensor([40], dtype=torch.int32, device="cuda")   # token 39 sits in the bad page
    x = torch.from_numpy(wl.queries((B, Hkv, 128), name="tiny_q")).cuda()
    tq.tq_append_paged(gcb, kc, num_pages, ps, bt, B, Hkv, sl, x, 128)
    torch.cuda.synchronize()
    with pytest.raises(tq.TqError) as e:
        tq.tq_check_device(gcb)
    assert e.value.status == tq.TQ_EINVAL
    assert torch.count_nonzero(kc) == 0
    ws = torch.empty(tq.tq_logits_workspace(gcb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    out = torch.zeros((B, Hq, max_pages * ps), device="cuda")
    tq.tq_logits_paged(gcb, kc, num_pages, ps, bt, B, Hq, Hkv, sl, x.new_zeros((B, Hq, 128)), out, ws)
    torch.cuda.synchronize()
    with pytest.raises(tq.TqError) as e:
        tq.tq_check_device(gcb)
    assert e.value.status == tq.TQ_EINVAL
    tq.tq_check_device(gcb)


def test_paged_invalid_arguments_return_status_without_launch():
    ocb, gcb = pair(3)
    ocp, gcp = pair(3, "mse", mode="polar")     # MSE-only keys are scored in scalar mode only
    kc = torch.zeros(tq.cache_bytes(gcb, 64), dtype=torch.uint8, device="cuda")
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    sl = torch.tensor([10], dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 4, 128), device="cuda")
    out = torch.zeros((1, 4, 64), device="cuda")
    ws = torch.empty(tq.tq_logits_workspace(gcb, 1, 4, 1), dtype=torch.uint8, device="cuda")
    for ps in (0, 8, 24, -16):
        with pytest.raises(tq.TqError) as e:
            tq.tq_logits_paged(gcb, kc, 4, ps, bt, 1, 4, 1, sl, q, out, ws)
        assert e.value.status == tq.TQ_EINVAL
    with pytest.raises(tq.TqError) as e:
        tq.tq_logits_paged(gcb, kc, 0, 16, bt, 1, 4, 1, sl, q, out, ws)
    assert e.value.status == tq.TQ_EINVAL
    with pytest.raises(tq.TqError) as e:
        tq.tq_logits_paged(gcp, kc, 4, 16, bt, 1, 4, 1, sl, q, out, ws)
    assert e.value.status == tq.TQ_EUNSUPPORTED
    torch.cuda.synchronize()
    tq.tq_check_device(gcb)
