"""tq_append_logits: a decode step's key append and logits in one call.

The fused path (scalar mode, d = 128, no extra-bit words: the append rides
in the query-prep launch) and the fallback (two launches as tq_quantize +
tq_logits) must both give the cache bytes and logits of the two separate
calls bit for bit; one case is also held to the oracle on the resulting
cache, and a destination outside the cache is skipped and flagged.
"""
import math

import numpy as np
import pytest
import torch

from decode_attention_21_b300 import tq
from decode_attention_21_b300 import workloads as wl
from oracle import estimate, layout, quant

pytestmark = pytest.mark.gpu


def filled_cache(cb, B, Hkv, cap, lens, seed):
    """A cache whose (b, kvh) rows 0..lens[b]-2 hold keys (the step appends row lens[b]-1)."""
    rows = B * Hkv * cap
    cache = torch.zeros(tq.cache_bytes(cb, rows), dtype=torch.uint8, device="cuda")
    for b in range(B):
        for h in range(Hkv):
            n = lens[b] - 1
            if n <= 0:
                continue
            x = torch.from_numpy(wl.llama_kv_slice(b, h, 0, n, seed=seed)).cuda()
            dst = torch.arange(n, dtype=torch.int64, device="cuda") + (b * Hkv + h) * cap
            tq.tq_quantize(cb, cache, rows, x, n, 128, dst_rows=dst)
    return cache


def step_inputs(B, Hq, Hkv, cap, lens, dtype, seed):
    rng = np.random.default_rng(seed)
    n = B * Hkv
    x = torch.from_numpy(rng.standard_normal((n, 128)).astype(np.float32) * 2.0).cuda()
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    dst = torch.tensor([(b * Hkv + h) * cap + lens[b] - 1 for b in range(B) for h in range(Hkv)], dtype=torch.int64,
                       device="cuda")
    q = torch.from_numpy(wl.queries((B, Hq, 128), seed=seed)).cuda()
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return x, dst, q, seq


def run_both(cb, B, Hq, Hkv, cap, lens, dtype, seed=5):
    x, dst, q, seq = step_inputs(B, Hq, Hkv, cap, lens, dtype, seed)
    base = filled_cache(cb, B, Hkv, cap, lens, seed)
    rows = B * Hkv * cap
    ws = torch.empty(tq.tq_logits_workspace(cb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    # separate calls
    c1 = base.clone()
    l1 = torch.full((B, Hq, cap), 7.0, device="cuda")
    tq.tq_quantize(cb, c1, rows, x, len(x), 128, dst_rows=dst)
    tq.tq_logits(cb, c1, B, Hq, Hkv, cap, seq, q, l1, ws)
    # one call
    c2 = base.clone()
    l2 = torch.full((B, Hq, cap), 7.0, device="cuda")
    tq.tq_append_logits(cb, c2, x, len(x), 128, dst, B, Hq, Hkv, cap, seq, q, l2, ws)
    tq.tq_check_device(cb)
    torch.cuda.synchronize()
    return c1, l1, c2, l2, x, q


@pytest.mark.parametrize("bits,kind", [(4, tq.KIND_PROD), (3, tq.KIND_PROD), (2, tq.KIND_PROD), (3, tq.KIND_MSE)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,Hq,Hkv,cap,lens", [(1, 32, 8, 4096, [4096]), (2, 8, 2, 1024, [1024, 333]),
                                              (3, 3, 3, 512, [1, 200, 512]), (1, 16, 2, 256, [100]),
                                              (2, 12, 1, 333, [333, 20]), (5, 4, 1, 64, [64, 1, 17, 33, 2])])
def test_fused_step_equals_separate_calls(bits, kind, dtype, B, Hq, Hkv, cap, lens):
    cb = tq.Codebook(128, bits, kind)
    c1, l1, c2, l2, _, _ = run_both(cb, B, Hq, Hkv, cap, lens, dtype)
    assert torch.equal(c1, c2)
    assert torch.equal(l1, l2)


@pytest.mark.parametrize("mode,extra", [(tq.MODE_POLAR, 0), (tq.MODE_SCALAR, 32)])
def test_unfused_codebooks_equal_separate_calls(mode, extra):
    cb = tq.Codebook(128, 3, tq.KIND_PROD, mode, extra=extra)
    c1, l1, c2, l2, _, _ = run_both(cb, 2, 8, 2, 512, [512, 77], "bf16")
    assert torch.equal(c1, c2)
    assert torch.equal(l1, l2)


def test_fused_step_against_the_oracle():
    """The prior keys come from the oracle's own packed cache; the step's new
    keys are appended by the fused call.  The oracle compresses every row
    itself (prior and new) and scores them: the GPU logits match within the
    parity bar, except at an appended row whose code the GPU took on the
    other side of a near-tie (at most 0.1% of that row's bits)."""
    B, Hq, Hkv, cap, lens = 2, 8, 2, 1024, [1024, 500]
    cb = tq.Codebook(128, 4, tq.KIND_PROD)
    ocb = quant.Codebook(128, 4, kind="prod")
    rows = B * Hkv * cap
    X = np.zeros((rows, 128))
    for b in range(B):
        for h in range(Hkv):
            r0 = (b * Hkv + h) * cap
            X[r0:r0 + lens[b] - 1] = wl.llama_kv_slice(b, h, 0, lens[b] - 1, seed=9)
    prior = quant.quantize(ocb, X)
    cache = torch.from_numpy(layout.write_cache(ocb, rows, prior)).cuda()
    x, dst, q, seq = step_inputs(B, Hq, Hkv, cap, lens, "f32", 9)
    ws = torch.empty(tq.tq_logits_workspace(cb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    got_l = torch.full((B, Hq, cap), 7.0, device="cuda")
    tq.tq_append_logits(cb, cache, x, len(x), 128, dst, B, Hq, Hkv, cap, seq, q, got_l, ws)
    tq.tq_check_device(cb)
    # the oracle: every row compressed and scored from the inputs
    dst_np = dst.cpu().numpy()
    X[dst_np] = x.cpu().numpy().astype(np.float64)
    full = quant.quantize(ocb, X)
    want = estimate.logits(ocb, full, q.cpu().numpy().astype(np.float64), np.array(lens), Hkv, cap)
    # the appended rows' codes (GPU output) against the oracle's
    got_code = layout.read_cache(ocb, rows, cache.cpu().numpy())
    differs = (got_code["idx"][dst_np] != full["idx"][dst_np]).any(axis=1) | \
              (got_code["sigma"][dst_np] != full["sigma"][dst_np]).any(axis=1)
    nbits = 128 * (ocb.b1 + 1)
    flips = (got_code["idx"][dst_np] != full["idx"][dst_np]).sum() + \
            (got_code["sigma"][dst_np] != full["sigma"][dst_np]).sum()
    assert flips <= max(1, 1e-3 * nbits * len(dst_np))
    got = got_l.cpu().numpy().astype(np.float64)
    for b in range(B):
        g, w = got[b, :, :lens[b]].copy(), want[b, :, :lens[b]].copy()
        for k, r in enumerate(dst_np):
            if differs[k] and r // (Hkv * cap) == b:
                t = r % cap
                h = (r // cap) % Hkv
                G = Hq // Hkv
                g[h * G:(h + 1) * G, t] = w[h * G:(h + 1) * G, t] = 0.0   # a near-tie code: not compared
        scale = np.max(np.abs(w), axis=-1, keepdims=True)
        assert np.all(np.abs(g - w) <= 1e-3 * scale + 1e-30)


def test_fused_destination_outside_the_cache_is_flagged():
    B, Hq, Hkv, cap = 1, 4, 1, 256
    cb = tq.Codebook(128, 4, tq.KIND_PROD)
    rows = B * Hkv * cap
    cache = torch.zeros(tq.cache_bytes(cb, rows), dtype=torch.uint8, device="cuda")
    x = torch.from_numpy(wl.llama_kv_slice(0, 0, 0, 2)).cuda()
    dst = torch.tensor([3, rows + 1], dtype=torch.int64, device="cuda")
    q = torch.from_numpy(wl.queries((B, Hq, 128), seed=1)).cuda()
    seq = torch.tensor([4], dtype=torch.int32, device="cuda")
    lg = torch.zeros((B, Hq, cap), device="cuda")
    ws = torch.empty(tq.tq_logits_workspace(cb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    tq.tq_append_logits(cb, cache, x, 2, 128, dst, B, Hq, Hkv, cap, seq, q, lg, ws)
    with pytest.raises(tq.TqError) as e:
        tq.tq_check_device(cb)
    assert e.value.status == tq.TQ_EINVAL
    W = tq.record_bytes(cb)
    assert int(cache[3 * W:4 * W].sum()) > 0           # the valid row was written
    tq.tq_check_device(cb)                             # the flag is cleared once read


def test_fused_step_in_a_cuda_graph():
    B, Hq, Hkv, cap, lens = 1, 32, 8, 2048, [2048]
    cb = tq.Codebook(128, 4, tq.KIND_PROD)
    c1, l1, _, _, _, _ = run_both(cb, B, Hq, Hkv, cap, lens, "bf16")
    x, dst, q, seq = step_inputs(B, Hq, Hkv, cap, lens, "bf16", 5)
    c3 = filled_cache(cb, B, Hkv, cap, lens, 5)
    l3 = torch.full((B, Hq, cap), 7.0, device="cuda")
    ws = torch.empty(tq.tq_logits_workspace(cb, B, Hq, Hkv), dtype=torch.uint8, device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        tq.tq_append_logits(cb, c3, x, len(x), 128, dst, B, Hq, Hkv, cap, seq, q, l3, ws)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    tq.tq_check_device(cb)
    assert torch.equal(c1, c3)
    assert torch.equal(l1, l3)
