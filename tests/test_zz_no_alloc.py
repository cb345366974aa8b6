"""The allocation-free decode-attention entry point.

tq_decode_attention_static is for callers that cannot allocate device memory
for this library (a plugin whose host framework owns all device memory, or a
loop that must not call cudaMalloc).  It must give the same result as
tq_decode_attention with a caller workspace, on consecutive calls that share
the built-in scratch array, and refuse work that does not fit the array.
This file is collected last so that a run stopping at its first failure has
already run every other test; it builds everything it needs itself, so it
also passes alone in a fresh process.
"""
import math

import numpy as np
import pytest
import torch

from decode_attention_21_b300 import tq
from decode_attention_21_b300 import workloads as wl
from oracle import estimate, layout, quant

pytestmark = pytest.mark.gpu


def _case(B, Hq, Hkv, cap, kb=3, vb=3):
    okc, ovc = quant.Codebook(128, kb, "prod"), quant.Codebook(128, vb, "mse")
    gkc, gvc = tq.Codebook(128, kb, tq.KIND_PROD), tq.Codebook(128, vb, tq.KIND_MSE)
    rows = B * Hkv * cap
    K = np.concatenate([wl.llama_kv_slice(1, h, 0, cap, which="keys") for h in range(B * Hkv)])
    V = np.concatenate([wl.llama_kv_slice(1, h, 0, cap, which="values") for h in range(B * Hkv)])
    kcode, vcode = quant.quantize(okc, K.astype(np.float64)), quant.quantize(ovc, V.astype(np.float64))
    kimg = torch.from_numpy(layout.write_cache(okc, rows, kcode)).cuda()
    vimg = torch.from_numpy(layout.write_cache(ovc, rows, vcode)).cuda()
    return (okc, ovc, kcode, vcode), gkc, gvc, kimg, vimg


def _close(got, ref, tol=1e-3):
    g = got.cpu().numpy().astype(np.float64)
    r = ref.cpu().numpy().astype(np.float64)
    scale = np.maximum(np.max(np.abs(r), axis=-1, keepdims=True), 1e-30)
    assert np.all(np.abs(g - r) <= tol * scale)


@pytest.mark.parametrize("B,Hq,Hkv,cap,lens0,lens1", [(2, 8, 2, 2048, [2048, 1500], [700, 2048]),
                                                       (3, 4, 1, 300, [300, 1, 0], [17, 0, 300])])
def test_static_matches_workspace_version_on_consecutive_calls(B, Hq, Hkv, cap, lens0, lens1):
    # Two calls in a row with different lengths, so the second call covers a
    # different set of split chunks than the first: a partial left in the
    # shared array by the first call and read by the second would show.  The
    # caller-workspace reference gets a workspace filled with NaN bytes before
    # each call, and both are held to the oracle on the same codes.
    (okc, ovc, kcode, vcode), gkc, gvc, kimg, vimg = _case(B, Hq, Hkv, cap)
    scale = 1.0 / math.sqrt(128)
    ws = torch.empty(tq.tq_decode_attention_workspace(gkc, B, Hq, Hkv, cap), dtype=torch.uint8, device="cuda")
    for call, lens in enumerate((lens0, lens1)):
        sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
        qn = wl.queries((B, Hq, 128), seed=7 + call)
        q = torch.from_numpy(qn).cuda()
        ws.fill_(0xFF)
        ref = torch.full((B, Hq, 128), float("nan"), device="cuda")
        tq.tq_decode_attention(gkc, gvc, kimg, vimg, B, Hq, Hkv, cap, sl, q, scale, ref, ws)
        out = torch.full((B, Hq, 128), float("nan"), device="cuda")
        tq.tq_decode_attention_static(gkc, gvc, kimg, vimg, B, Hq, Hkv, cap, sl, q, scale, out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        _close(out, ref)
        want = estimate.attention(okc, ovc, kcode, vcode, qn.astype(np.float64), lens, Hkv, cap, scale)
        _close(out, torch.from_numpy(want))


def test_static_rejects_work_beyond_its_array():
    gkc = tq.Codebook(128, 3, tq.KIND_PROD)
    gvc = tq.Codebook(128, 3, tq.KIND_MSE)
    B, Hq, Hkv, cap = 64, 32, 8, 1 << 20
    assert tq.tq_decode_attention_workspace(gkc, B, Hq, Hkv, cap) > (4 << 20)
    dummy = torch.zeros(256, dtype=torch.uint8, device="cuda")
    out = torch.full((4,), 123.0, device="cuda")
    with pytest.raises(tq.TqError) as e:
        tq.tq_decode_attention_static(gkc, gvc, dummy, dummy, B, Hq, Hkv, cap, dummy, dummy, 0.1, out)
    assert e.value.status == tq.TQ_EINVAL
    assert "scratch" in tq.tq_last_error()
    torch.cuda.synchronize()
    assert torch.all(out == 123.0)
