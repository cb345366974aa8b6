"""Bounded device-side waits give up cleanly.

Every wait of a kernel on its own bulk copies or tensor-core operations is
bounded.  tq_set_first_wait_limit(cb, 0) makes the first such wait of each
launch give up at once, which drives the timeout path without faulting or
hanging anything: the kernel records TQ_ETIMEOUT for tq_check_device, lets
the work it already issued finish, frees its tensor memory and returns.  The
next call with the default limit must then run normally and give the same
bytes as a call that never timed out.
"""
import math

import numpy as np
import pytest
import torch

from decode_attention_21_b300 import tq
from decode_attention_21_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def _expect_timeout(cb):
    with pytest.raises(tq.TqError) as e:
        tq.tq_check_device(cb)
    assert e.value.status == tq.TQ_ETIMEOUT


def test_tensor_core_quantize_gives_up_and_recovers():
    cb = tq.Codebook(128, 3, tq.KIND_PROD)
    n = 4096                                          # bf16, >= 2048 rows: the tcgen05 path
    x = torch.from_numpy(wl.llama_kv_slice(2, 0, 0, n, which="keys")).cuda().to(torch.bfloat16)
    ref = torch.zeros(tq.cache_bytes(cb, n), dtype=torch.uint8, device="cuda")
    tq.tq_quantize(cb, ref, n, x, n, 128)
    tq.tq_check_device(cb)
    cache = torch.zeros_like(ref)
    tq.tq_set_first_wait_limit(cb, 0)
    try:
        tq.tq_quantize(cb, cache, n, x, n, 128)
        _expect_timeout(cb)
    finally:
        tq.tq_set_first_wait_limit(cb, -1)
    tq.tq_quantize(cb, cache, n, x, n, 128)
    tq.tq_check_device(cb)
    assert torch.equal(cache, ref)


def _key_value_caches(kcb, vcb, B, Hkv, T):
    rows = B * Hkv * T
    kc = torch.zeros(tq.cache_bytes(kcb, rows), dtype=torch.uint8, device="cuda")
    vc = torch.zeros(tq.cache_bytes(vcb, rows), dtype=torch.uint8, device="cuda")
    for u in range(B * Hkv):
        dst = torch.arange(u * T, (u + 1) * T, dtype=torch.int64, device="cuda")
        k = torch.from_numpy(wl.llama_kv_slice(3, u, 0, T, which="keys")).cuda()
        v = torch.from_numpy(wl.llama_kv_slice(3, u, 0, T, which="values")).cuda()
        tq.tq_quantize(kcb, kc, rows, k, T, 128, dst_rows=dst)
        tq.tq_quantize(vcb, vc, rows, v, T, 128, dst_rows=dst)
    tq.tq_check_device(kcb)
    return kc, vc


def test_staged_logits_give_up_and_recover():
    kcb, vcb = tq.Codebook(128, 4, tq.KIND_PROD), tq.Codebook(128, 3, tq.KIND_MSE)
    B, Hq, Hkv, T = 2, 8, 2, 1024                     # capacity a multiple of 16: the staged kernel
    kc, _ = _key_value_caches(kcb, vcb, B, Hkv, T)
    q = torch.from_numpy(wl.queries((B, Hq, 128), seed=11)).cuda()
    seq = torch.tensor([T, 700], dtype=torch.int32, device="cuda")
    ws = torch.empty(tq.tq_logits_workspace(kcb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    ref = torch.zeros(B, Hq, T, device="cuda")
    tq.tq_logits(kcb, kc, B, Hq, Hkv, T, seq, q, ref, ws)
    out = torch.zeros(B, Hq, T, device="cuda")
    tq.tq_set_first_wait_limit(kcb, 0)
    try:
        tq.tq_logits(kcb, kc, B, Hq, Hkv, T, seq, q, out, ws)
        _expect_timeout(kcb)
    finally:
        tq.tq_set_first_wait_limit(kcb, -1)
    tq.tq_logits(kcb, kc, B, Hq, Hkv, T, seq, q, out, ws)
    tq.tq_check_device(kcb)
    assert torch.equal(out, ref)


def test_staged_attention_gives_up_and_recovers():
    kcb, vcb = tq.Codebook(128, 3, tq.KIND_PROD), tq.Codebook(128, 3, tq.KIND_MSE)
    B, Hq, Hkv, T = 2, 8, 2, 2048
    kc, vc = _key_value_caches(kcb, vcb, B, Hkv, T)
    q = torch.from_numpy(wl.queries((B, Hq, 128), seed=12)).cuda()
    seq = torch.tensor([T, 1500], dtype=torch.int32, device="cuda")
    ws = torch.empty(tq.tq_decode_attention_workspace(kcb, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(128)
    ref = torch.zeros(B, Hq, 128, device="cuda")
    tq.tq_decode_attention(kcb, vcb, kc, vc, B, Hq, Hkv, T, seq, q, scale, ref, ws)
    tq.tq_set_first_wait_limit(kcb, 0)
    try:
        tq.tq_decode_attention(kcb, vcb, kc, vc, B, Hq, Hkv, T, seq, q, scale, torch.zeros_like(ref), ws)
        _expect_timeout(kcb)
    finally:
        tq.tq_set_first_wait_limit(kcb, -1)
    out = torch.zeros_like(ref)
    tq.tq_decode_attention(kcb, vcb, kc, vc, B, Hq, Hkv, T, seq, q, scale, out, ws)
    tq.tq_check_device(kcb)
    assert torch.equal(out, ref)
    assert np.all(np.isfinite(out.cpu().numpy()))


def test_tensor_memory_operand_quantize_gives_up_and_recovers():
    # the d = 256 kernel (X and the residual in tensor memory, Pi and S
    # streamed through a TMA ring): a timeout on its first ring wait must
    # drain the loads already issued and free its tensor memory
    cb = tq.Codebook(256, 3, tq.KIND_PROD)
    n = 4096
    x = torch.from_numpy(wl.search_rows(n, "db")).cuda()
    ref = torch.zeros(tq.cache_bytes(cb, n), dtype=torch.uint8, device="cuda")
    tq.tq_quantize(cb, ref, n, x, n, 200)
    tq.tq_check_device(cb)
    cache = torch.zeros_like(ref)
    tq.tq_set_first_wait_limit(cb, 0)
    try:
        tq.tq_quantize(cb, cache, n, x, n, 200)
        _expect_timeout(cb)
    finally:
        tq.tq_set_first_wait_limit(cb, -1)
    tq.tq_quantize(cb, cache, n, x, n, 200)
    tq.tq_check_device(cb)
    assert torch.equal(cache, ref)
