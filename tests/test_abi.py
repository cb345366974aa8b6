"""The C-ABI library without a GPU: it loads, exports every declared entry
point, validates arguments on the host, and its host-side setup mathematics
(independent C++: splitmix64, Householder QR, Gauss-Legendre Lloyd-Max)
agrees with the oracle's."""
import ctypes
import os
import re

import numpy as np
import pytest

from decode_attention_21_b300 import tq
from oracle import codebook as ocb
from oracle import polar as opolar
from oracle.rotation import haar_rotation, qjl_matrix

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    return sorted(set(re.findall(r"^\s*(?:tq_status|void|size_t|const char\*)\s+(tq_\w+)\(", text, re.M)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(tq.LIB_PATH):
        from decode_attention_21_b300 import build
        build.build()
    return tq.lib()


def test_every_declared_symbol_is_exported(L):
    syms = declared_symbols()
    assert len(syms) >= 15
    for s in syms:
        assert hasattr(L, s), s
    assert sorted(tq.EXPORTS) == syms


def test_descriptor_validation_on_host(L):
    for d, bits, kind, mode, extra in [(64, 3, 0, 0, 0), (128, 5, 0, 0, 0), (128, 1, 0, 0, 0), (128, 5, 1, 0, 0),
                                       (128, 3, 2, 0, 0), (128, 3, 0, 2, 0), (128, 3, 0, 0, 16), (128, 3, 0, 1, 32),
                                       (128, 4, 1, 0, 32)]:
        desc = tq.Desc(d, bits, d, mode, kind, extra, 1, 2, None, None)
        h = ctypes.c_void_p()
        assert L.tq_make_codebook(ctypes.byref(desc), ctypes.byref(h)) == tq.TQ_EINVAL
        assert L.tq_last_error()
        assert L.tq_host_tables(ctypes.byref(desc), 1, None, None, None, None) == tq.TQ_EINVAL
    # m must equal d for keys
    desc = tq.Desc(128, 3, 64, 0, 0, 0, 1, 2, None, None)
    assert L.tq_host_tables(ctypes.byref(desc), 1, None, None, None, None) == tq.TQ_EINVAL
    assert L.tq_cache_bytes(None, 10) == 0 and L.tq_record_bytes(None) == 0
    assert L.tq_quantize(None, None, 0, None, 0, 0, 0, None, None) == tq.TQ_EINVAL
    assert L.tq_logits(None, None, 1, 1, 1, 1, None, None, None, None, 0, None) == tq.TQ_EINVAL
    assert L.tq_append_logits(None, None, None, 0, 1, 128, None, 1, 1, 1, 1, None, None, None, None, 0,
                              None) == tq.TQ_EINVAL
    assert L.tq_decode_attention(None, None, None, None, 1, 1, 1, 1, None, None, 1.0, None, None, 0, None) == tq.TQ_EINVAL


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("b1", [1, 2, 3, 4])
def test_scalar_tables_match_oracle_bit_for_bit(L, d, b1):
    c, t, _, _ = tq.host_tables(d, b1, kind=tq.KIND_MSE)
    oc, ot = ocb.scalar_codebook(d, b1)
    assert np.array_equal(c, oc) and np.array_equal(t, ot)


@pytest.mark.parametrize("level", [1, 2, 3, 7])
@pytest.mark.parametrize("b1", [1, 2, 3])
def test_polar_tables_match_oracle(L, level, b1):
    c, t, _, _ = tq.host_tables(128, b1, kind=tq.KIND_MSE, mode=tq.MODE_POLAR, level=level)
    tab = opolar.PolarTables(128, b1)
    assert np.array_equal(c, tab.cent32[level])
    assert np.array_equal(t, tab.bound32[level])


@pytest.mark.parametrize("d,seed", [(128, 1), (256, 7)])
def test_rotation_and_sketch_match_oracle(L, d, seed):
    _, _, pi, s = tq.host_tables(d, 3, seed_pi=seed, seed_s=seed + 1)
    P = haar_rotation(d, seed)
    assert np.max(np.abs(pi - P)) < 1e-12
    assert np.array_equal(s.astype(np.float64), qjl_matrix(d, d, seed + 1))


@pytest.mark.parametrize("E,bits", [(32, 2), (64, 3), (32, 4)])
def test_split_tables_match_oracle(L, E, bits):
    # outlier-channel split: the library's d x d rotation and block-diagonal
    # sketch, built from the two groups' own seeds and the channel list, and
    # group B's stage-1 tables, against the oracle's two instances
    from oracle import split
    out = np.random.default_rng(E + bits).choice(128, size=E, replace=False)
    c, t, pi, s = tq.host_tables(128, bits, seed_pi=5, seed_s=9, outliers=out)
    scb = split.SplitCodebook(128, bits, out, seed_pi=5, seed_s=9)
    assert np.max(np.abs(pi - scb.full_rotation())) < 1e-12
    assert np.array_equal(s.astype(np.float64), scb.full_sketch())
    assert np.array_equal(c, scb.groups[1].c) and np.array_equal(t, scb.groups[1].t)


def test_split_descriptor_checks(L):
    out = np.arange(32, dtype=np.int32)
    for d, kind, mode, extra, chans in [(256, tq.KIND_PROD, tq.MODE_SCALAR, 32, out),
                                        (128, tq.KIND_MSE, tq.MODE_SCALAR, 32, out),
                                        (128, tq.KIND_PROD, tq.MODE_POLAR, 32, out),
                                        (128, tq.KIND_PROD, tq.MODE_SCALAR, 32, np.r_[out[:31], 0].astype(np.int32)),
                                        (128, tq.KIND_PROD, tq.MODE_SCALAR, 32, np.r_[out[:31], 128].astype(np.int32))]:
        desc = tq.Desc(d, 3, d, mode, kind, extra, 1, 2, None, None, None)
        desc.outliers = chans.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        assert L.tq_host_tables(ctypes.byref(desc), 1, None, None, None, None) == tq.TQ_EINVAL
