"""Every output stays inside its buffer, and codebook setup survives a failed
device allocation.

Each output (cache, logits, attention output, search ids and scores, and
the workspaces) is the front of a larger byte buffer whose tail holds a
canary pattern; after the call the tail must be byte-for-byte unchanged.
The cases reach every quantize kernel (two-group tensor-core, tensor-memory
operand at d = 128 fp32 and d = 256, in scalar and polar mode; row-per-warp,
short-batch) and the scoring kernels.  The allocation hook makes the n-th device allocation of
tq_make_codebook fail: the call must return TQ_ENOMEM and leave a working
library behind.
"""
import math

import numpy as np
import pytest
import torch

from decode_attention_21_b300 import tq
from decode_attention_21_b300 import workloads as wl

pytestmark = pytest.mark.gpu

CANARY = 0xA5
TAIL = 4096


def guarded(nbytes):
    """(whole buffer, front view of nbytes) with a canary tail."""
    buf = torch.full((nbytes + TAIL,), CANARY, dtype=torch.uint8, device="cuda")
    return buf, buf[:nbytes]


def tail_intact(buf, nbytes):
    torch.cuda.synchronize()
    return bool(torch.all(buf[nbytes:] == CANARY))


@pytest.mark.parametrize("d,dtype,n,extra,mode", [(128, "bf16", 4096, 0, 0), (128, "bf16", 4096, 32, 0),
                                                  (128, "f32", 4096, 0, 0), (256, "f32", 4096, 0, 0),
                                                  (256, "bf16", 2048 + 5, 0, 0), (128, "bf16", 100, 0, 0),
                                                  (128, "f32", 20000, 32, 0), (128, "bf16", 4096 + 7, 0, 1),
                                                  (128, "f32", 4096, 0, 1), (256, "bf16", 2048 + 5, 0, 1)])
def test_quantize_writes_stay_inside_the_cache(d, dtype, n, extra, mode):
    cb = tq.Codebook(d, 3, tq.KIND_PROD, tq.MODE_POLAR if mode else tq.MODE_SCALAR, extra=extra)
    d_in = 200 if d == 256 else 128
    x = wl.search_rows(n, "db") if d == 256 else np.concatenate(
        [wl.llama_kv_slice(0, h, 0, 4096) for h in range(-(-n // 4096))])[:n]
    xt = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    if dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    nbytes = tq.cache_bytes(cb, n)
    buf, cache = guarded(nbytes)
    tq.tq_quantize(cb, cache, n, xt, n, d_in)
    tq.tq_check_device(cb)
    assert tail_intact(buf, nbytes)


def test_scoring_writes_stay_inside_outputs_and_workspaces():
    kcb = tq.Codebook(128, 3, tq.KIND_PROD)
    vcb = tq.Codebook(128, 3, tq.KIND_MSE)
    B, Hq, Hkv, cap = 2, 8, 2, 1024
    rows = B * Hkv * cap
    kc = torch.zeros(tq.cache_bytes(kcb, rows), dtype=torch.uint8, device="cuda")
    vc = torch.zeros(tq.cache_bytes(vcb, rows), dtype=torch.uint8, device="cuda")
    for u in range(B * Hkv):
        dst = torch.arange(u * cap, (u + 1) * cap, dtype=torch.int64, device="cuda")
        tq.tq_quantize(kcb, kc, rows, torch.from_numpy(wl.llama_kv_slice(2, u, 0, cap, which="keys")).cuda(), cap,
                       128, dst_rows=dst)
        tq.tq_quantize(vcb, vc, rows, torch.from_numpy(wl.llama_kv_slice(2, u, 0, cap, which="values")).cuda(), cap,
                       128, dst_rows=dst)
    q = torch.from_numpy(wl.queries((B, Hq, 128), seed=3)).cuda()
    seq = torch.tensor([cap, 700], dtype=torch.int32, device="cuda")
    # logits
    lb = B * Hq * cap * 4
    lbuf, lfront = guarded(lb)
    wsb = tq.tq_logits_workspace(kcb, B, Hq, Hkv)
    wbuf, wfront = guarded(wsb)
    tq.tq_logits(kcb, kc, B, Hq, Hkv, cap, seq, q, lfront.view(torch.float32).view(B, Hq, cap), wfront)
    tq.tq_check_device(kcb)
    assert tail_intact(lbuf, lb) and tail_intact(wbuf, wsb)
    # decode attention
    ob = B * Hq * 128 * 4
    obuf, ofront = guarded(ob)
    wsa = tq.tq_decode_attention_workspace(kcb, B, Hq, Hkv, cap)
    abuf, afront = guarded(wsa)
    tq.tq_decode_attention(kcb, vcb, kc, vc, B, Hq, Hkv, cap, seq, q, 1.0 / math.sqrt(128),
                           ofront.view(torch.float32).view(B, Hq, 128), afront)
    tq.tq_check_device(kcb)
    assert tail_intact(obuf, ob) and tail_intact(abuf, wsa)


@pytest.mark.parametrize("k", [10, 20])
def test_search_writes_stay_inside_outputs_and_workspace(k):
    # k = 10: tensor-core scan, re-ranking and certificate; k = 20: exact scan
    cb = tq.Codebook(256, 3, tq.KIND_PROD)
    n_db, nq = 20000, 300
    db = torch.zeros(tq.cache_bytes(cb, n_db), dtype=torch.uint8, device="cuda")
    tq.tq_quantize(cb, db, n_db, torch.from_numpy(wl.search_rows(n_db, "db")).cuda(), n_db, 200)
    q = torch.from_numpy(wl.search_rows(nq, "search_q")).cuda()
    ib, sb = nq * k * 4, nq * k * 4
    ibuf, ifront = guarded(ib)
    sbuf, sfront = guarded(sb)
    wsb = tq.tq_search_workspace(cb, n_db, nq, k)
    wbuf, wfront = guarded(wsb)
    tq.tq_search(cb, db, n_db, q, nq, 200, k, ifront.view(torch.int32).view(nq, k),
                 sfront.view(torch.float32).view(nq, k), wfront)
    tq.tq_check_device(cb)
    assert tail_intact(ibuf, ib) and tail_intact(sbuf, sb) and tail_intact(wbuf, wsb)


def test_codebook_allocation_failure_is_reported_and_recovered():
    failed = 0
    try:
        for nth in range(16):
            tq.tq_fail_allocation(nth)
            try:
                cb = tq.Codebook(128, 3, tq.KIND_PROD)
            except tq.TqError as e:
                assert e.status == tq.TQ_ENOMEM
                assert "injected" in tq.tq_last_error()
                failed += 1
            else:
                del cb
            tq.tq_fail_allocation(-1)
    finally:
        tq.tq_fail_allocation(-1)
    assert failed >= 4
    # the library still works after the failed setups
    cb = tq.Codebook(128, 3, tq.KIND_PROD)
    x = torch.from_numpy(wl.llama_kv_slice(0, 0, 0, 64)).cuda()
    cache = torch.zeros(tq.cache_bytes(cb, 64), dtype=torch.uint8, device="cuda")
    tq.tq_quantize(cb, cache, 64, x, 64, 128)
    tq.tq_check_device(cb)
    assert int(cache.sum()) > 0


@pytest.mark.parametrize("d,dtype,extra,mode", [(128, "bf16", 0, 0), (128, "f32", 0, 0), (256, "f32", 0, 0),
                                                (256, "bf16", 0, 0), (128, "bf16", 32, 0), (128, "bf16", 0, 1),
                                                (256, "f32", 0, 1)])
def test_quantize_destination_outside_the_cache_is_skipped_and_flagged(d, dtype, extra, mode):
    # a destination row past the cache is not written (the canary tail stays)
    # and tq_check_device reports TQ_EINVAL; every other row is written
    cb = tq.Codebook(d, 3, tq.KIND_PROD, tq.MODE_POLAR if mode else tq.MODE_SCALAR, extra=extra)
    n, rows = 4096, 5000
    d_in = 256 if d == 256 else 128
    x = np.random.default_rng(d).standard_normal((n, d_in)).astype(np.float32)
    xt = torch.from_numpy(x).cuda()
    if dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    dst = torch.arange(n, dtype=torch.int64, device="cuda") + 7
    dst[1234] = rows + 5
    nbytes = tq.cache_bytes(cb, rows)
    buf, cache = guarded(nbytes)
    tq.tq_quantize(cb, cache, rows, xt, n, d_in, dst_rows=dst)
    with pytest.raises(tq.TqError) as e:
        tq.tq_check_device(cb)
    assert e.value.status == tq.TQ_EINVAL
    assert tail_intact(buf, nbytes)
    ref = torch.zeros(tq.cache_bytes(cb, rows), dtype=torch.uint8, device="cuda")
    ok_dst = dst.clone()
    ok_dst[1234] = 3                                   # a row nobody else writes
    tq.tq_quantize(cb, ref, rows, xt, n, d_in, dst_rows=ok_dst)
    tq.tq_check_device(cb)
    W = tq.record_bytes(cb)
    recs, recs_ref = cache[: rows * W].view(rows, W), ref[: rows * W].view(rows, W)
    written = torch.cat([dst[:1234], dst[1235:]])     # rows both calls wrote
    assert torch.equal(recs[written], recs_ref[written])
