"""ctypes binding of ``libtq.so`` with the C-ABI names of ``include/tq.h``.

Argument marshalling only: tensors are passed as raw device pointers and every
step runs in the library's CUDA kernels.  If the library is missing the first
call raises; there is no fallback path.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtq.so")

TQ_OK, TQ_EINVAL, TQ_ENOMEM, TQ_ECUDA, TQ_ETIMEOUT, TQ_EUNSUPPORTED = range(6)
MODE_SCALAR, MODE_POLAR = 0, 1
KIND_PROD, KIND_MSE = 0, 1
F32, BF16 = 0, 1

EXPORTS = ["tq_make_codebook", "tq_free_codebook", "tq_codebook_tables", "tq_host_tables", "tq_record_bytes", "tq_cache_bytes",
           "tq_quantize", "tq_quantize_rotated", "tq_logits_workspace", "tq_logits", "tq_append_logits", "tq_logits_dense",
           "tq_decode_attention_workspace", "tq_decode_attention", "tq_decode_attention_static",
           "tq_search_workspace", "tq_search", "tq_search_fallbacks", "tq_set_first_wait_limit", "tq_fail_allocation",
           "tq_append_paged", "tq_logits_paged", "tq_decode_attention_paged", "tq_advance_lengths",
           "tq_check_device", "tq_last_error"]


class TqError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"tq status {status}: {msg}")
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("bits", ctypes.c_int32), ("m", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("kind", ctypes.c_int32), ("extra", ctypes.c_int32), ("seed_pi", ctypes.c_uint64),
                ("seed_s", ctypes.c_uint64), ("pi", ctypes.POINTER(ctypes.c_double)),
                ("s", ctypes.POINTER(ctypes.c_float)), ("outliers", ctypes.POINTER(ctypes.c_int32))]


_lib = None


def lib():
    """The loaded library; raises if ``libtq.so`` has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m decode_attention_21_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        L.tq_make_codebook.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(vp)]
        L.tq_free_codebook.argtypes = [vp]
        L.tq_free_codebook.restype = None
        L.tq_codebook_tables.argtypes = [vp, vp, vp, vp, vp]
        L.tq_host_tables.argtypes = [ctypes.POINTER(Desc), i32, vp, vp, vp, vp]
        L.tq_record_bytes.argtypes = [vp]
        L.tq_record_bytes.restype = sz
        L.tq_cache_bytes.argtypes = [vp, i64]
        L.tq_cache_bytes.restype = sz
        L.tq_quantize.argtypes = [vp, vp, i64, vp, i32, i64, i32, vp, vp]
        L.tq_quantize_rotated.argtypes = [vp, vp, i64, vp, vp, i64, vp, vp]
        L.tq_logits_workspace.argtypes = [vp, i32, i32, i32]
        L.tq_logits_workspace.restype = sz
        L.tq_logits.argtypes = [vp, vp, i32, i32, i32, i64, vp, vp, vp, vp, sz, vp]
        L.tq_append_logits.argtypes = [vp, vp, vp, i32, i64, i32, vp, i32, i32, i32, i64, vp, vp, vp, vp, sz, vp]
        L.tq_logits_dense.argtypes = [vp, i32, i32, i32, i32, i32, i64, vp, vp, vp, vp]
        L.tq_decode_attention_workspace.argtypes = [vp, i32, i32, i32, i64]
        L.tq_decode_attention_workspace.restype = sz
        L.tq_decode_attention.argtypes = [vp, vp, vp, vp, i32, i32, i32, i64, vp, vp, ctypes.c_float, vp, vp, sz, vp]
        L.tq_decode_attention_static.argtypes = [vp, vp, vp, vp, i32, i32, i32, i64, vp, vp, ctypes.c_float, vp,
                                                 vp]
        L.tq_search_workspace.argtypes = [vp, i64, i32, i32]
        L.tq_search_workspace.restype = sz
        L.tq_search.argtypes = [vp, vp, i64, vp, i32, i32, i32, vp, vp, vp, sz, vp]
        L.tq_search_fallbacks.argtypes = [vp, vp, i32, ctypes.POINTER(i32)]
        L.tq_set_first_wait_limit.argtypes = [vp, i64]
        L.tq_fail_allocation.argtypes = [i32]
        L.tq_append_paged.argtypes = [vp, vp, i32, i32, vp, i32, i32, i32, vp, vp, i32, i32, vp]
        L.tq_logits_paged.argtypes = [vp, vp, i32, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
        L.tq_decode_attention_paged.argtypes = [vp, vp, vp, vp, i32, i32, vp, i32, i32, i32, i32, vp, vp,
                                                ctypes.c_float, vp, vp, sz, vp]
        L.tq_advance_lengths.argtypes = [vp, i32, i32, vp]
        L.tq_check_device.argtypes = [vp]
        L.tq_last_error.argtypes = []
        L.tq_last_error.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name not in ("tq_free_codebook", "tq_record_bytes", "tq_cache_bytes", "tq_logits_workspace",
                            "tq_decode_attention_workspace", "tq_search_workspace", "tq_last_error"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(st):
    if st != TQ_OK:
        raise TqError(st, lib().tq_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return stream


class Codebook:
    """Owner of a ``tq_codebook*`` built on the current CUDA device."""

    def __init__(self, d=128, bits=3, kind=KIND_PROD, mode=MODE_SCALAR, seed_pi=1, seed_s=2, m=None, extra=0,
                 pi=None, s=None, outliers=None):
        import numpy as np
        if outliers is not None:
            extra = len(outliers)
        desc = Desc(d, bits, m if m is not None else d, mode, kind, extra, seed_pi, seed_s, None, None, None)
        self._keep = []
        if outliers is not None:
            a = np.ascontiguousarray(outliers, dtype=np.int32)
            self._keep.append(a)
            desc.outliers = a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        if pi is not None:
            a = np.ascontiguousarray(pi, dtype=np.float64)
            self._keep.append(a)
            desc.pi = a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
        if s is not None:
            a = np.ascontiguousarray(s, dtype=np.float32)
            self._keep.append(a)
            desc.s = a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
        h = ctypes.c_void_p()
        _check(lib().tq_make_codebook(ctypes.byref(desc), ctypes.byref(h)))
        self.handle = h.value
        self.d, self.bits, self.kind, self.mode, self.extra = d, bits, kind, mode, extra
        self.split = outliers is not None
        self.b1 = bits - 1 if kind == KIND_PROD else bits

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.tq_free_codebook(self.handle)
            self.handle = None

    @property
    def _as_parameter_(self):
        return self.handle


def codebook_tables(cb):
    import numpy as np
    L = 1 << cb.b1
    c = np.zeros(L, dtype=np.float32)
    t = np.zeros(L - 1, dtype=np.float32)
    pi = np.zeros((cb.d, cb.d), dtype=np.float64)
    s = np.zeros((cb.d, cb.d), dtype=np.float32)
    _check(lib().tq_codebook_tables(cb.handle, c.ctypes.data, t.ctypes.data, pi.ctypes.data, s.ctypes.data))
    return c, t, pi, (s if cb.kind == KIND_PROD else None)


def host_tables(d, bits, kind=KIND_PROD, mode=MODE_SCALAR, seed_pi=1, seed_s=2, level=2, outliers=None):
    """(centroids, boundaries, pi, s) the library would build, computed on the host
    (for an outlier-channel split: group B's tables, the d x d rotation and sketch)."""
    import numpy as np
    desc = Desc(d, bits, d, mode, kind, 0, seed_pi, seed_s, None, None, None)
    if outliers is not None:
        keep = np.ascontiguousarray(outliers, dtype=np.int32)
        desc.extra = len(keep)
        desc.outliers = keep.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    b1 = bits - 1 if kind == KIND_PROD else bits
    L = 1 << b1
    c = np.zeros(L, dtype=np.float32)
    t = np.zeros(max(L - 1, 1), dtype=np.float32)
    pi = np.zeros((d, d), dtype=np.float64)
    s = np.zeros((d, d), dtype=np.float32)
    _check(lib().tq_host_tables(ctypes.byref(desc), level, c.ctypes.data, t.ctypes.data, pi.ctypes.data,
                                s.ctypes.data))
    return c, t[:L - 1], pi, (s if kind == KIND_PROD else None)


def record_bytes(cb):
    return lib().tq_record_bytes(cb.handle)


def cache_bytes(cb, rows):
    return lib().tq_cache_bytes(cb.handle, rows)


def tq_quantize(cb, cache, cache_rows, x, n, d_in, dst_rows=None, stream=None):
    dt = BF16 if x.dtype == torch.bfloat16 else F32
    _check(lib().tq_quantize(cb.handle, _ptr(cache), cache_rows, _ptr(x), dt, n, d_in, _ptr(dst_rows),
                             _stream(stream)))


def tq_quantize_rotated(cb, cache, cache_rows, y, norms, n, dst_rows=None, stream=None):
    _check(lib().tq_quantize_rotated(cb.handle, _ptr(cache), cache_rows, _ptr(y), _ptr(norms), n, _ptr(dst_rows),
                                     _stream(stream)))


def tq_logits_workspace(kcb, B, Hq, Hkv):
    return lib().tq_logits_workspace(kcb.handle, B, Hq, Hkv)


def tq_logits(kcb, kcache, B, Hq, Hkv, capacity, seq_lens, q, logits, workspace, stream=None):
    _check(lib().tq_logits(kcb.handle, _ptr(kcache), B, Hq, Hkv, capacity, _ptr(seq_lens), _ptr(q), _ptr(logits),
                           _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_append_logits(kcb, kcache, x, n, d_in, dst_rows, B, Hq, Hkv, capacity, seq_lens, q, logits, workspace,
                     stream=None):
    """tq_quantize of the step's new keys x into kcache, then tq_logits (one
    call; the append rides in the query-prep launch where it can)."""
    dt = BF16 if x.dtype == torch.bfloat16 else F32
    _check(lib().tq_append_logits(kcb.handle, _ptr(kcache), _ptr(x), dt, n, d_in, _ptr(dst_rows), B, Hq, Hkv,
                                  capacity, _ptr(seq_lens), _ptr(q), _ptr(logits), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_logits_dense(keys, B, Hq, Hkv, capacity, seq_lens, q, logits, stream=None):
    """Unquantized comparator: keys [B, Hkv, capacity, 128] fp32 or bf16."""
    dt = {torch.float32: F32, torch.bfloat16: BF16}[keys.dtype]
    _check(lib().tq_logits_dense(_ptr(keys), dt, keys.shape[-1], B, Hq, Hkv, capacity, _ptr(seq_lens), _ptr(q),
                                 _ptr(logits), _stream(stream)))


def tq_decode_attention_workspace(kcb, B, Hq, Hkv, capacity):
    return lib().tq_decode_attention_workspace(kcb.handle, B, Hq, Hkv, capacity)


def tq_decode_attention(kcb, vcb, kcache, vcache, B, Hq, Hkv, capacity, seq_lens, q, scale, out, workspace,
                        stream=None):
    _check(lib().tq_decode_attention(kcb.handle, vcb.handle, _ptr(kcache), _ptr(vcache), B, Hq, Hkv, capacity,
                                     _ptr(seq_lens), _ptr(q), float(scale), _ptr(out), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_decode_attention_static(kcb, vcb, kcache, vcache, B, Hq, Hkv, capacity, seq_lens, q, scale, out,
                               stream=None):
    """Decode attention with the library's built-in scratch array (no workspace
    argument, no allocation); see include/tq.h for its limit and sharing rules."""
    _check(lib().tq_decode_attention_static(kcb.handle, vcb.handle, _ptr(kcache), _ptr(vcache), B, Hq, Hkv, capacity,
                                            _ptr(seq_lens), _ptr(q), float(scale), _ptr(out), _stream(stream)))


def tq_search_workspace(cb, n_db, nq, k):
    return lib().tq_search_workspace(cb.handle, n_db, nq, k)


def tq_search(cb, db_cache, n_db, q, nq, d_in, k, ids, scores, workspace, stream=None):
    _check(lib().tq_search(cb.handle, _ptr(db_cache), n_db, _ptr(q), nq, d_in, k, _ptr(ids), _ptr(scores),
                           _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_search_fallbacks(cb, workspace, k):
    """Queries of the last tq_search on ``workspace`` that the exact scan re-ran
    (-1: that call used the exact scan only).  Synchronises the device."""
    n = ctypes.c_int32()
    _check(lib().tq_search_fallbacks(cb.handle, _ptr(workspace), k, ctypes.byref(n)))
    return n.value


def tq_append_paged(cb, cache, num_pages, page_size, block_table, B, Hkv, seq_lens, x, d_in, stream=None):
    """Append x [B, Hkv, d_in] at token seq_lens[b] - 1 of each sequence of a
    paged cache; block_table is int32 [B, max_pages]."""
    dt = BF16 if x.dtype == torch.bfloat16 else F32
    _check(lib().tq_append_paged(cb.handle, _ptr(cache), num_pages, page_size, _ptr(block_table),
                                 block_table.shape[1], B, Hkv, _ptr(seq_lens), _ptr(x), dt, d_in, _stream(stream)))


def tq_logits_paged(kcb, kcache, num_pages, page_size, block_table, B, Hq, Hkv, seq_lens, q, logits, workspace,
                    stream=None):
    _check(lib().tq_logits_paged(kcb.handle, _ptr(kcache), num_pages, page_size, _ptr(block_table),
                                 block_table.shape[1], B, Hq, Hkv, _ptr(seq_lens), _ptr(q), _ptr(logits),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_decode_attention_paged(kcb, vcb, kcache, vcache, num_pages, page_size, block_table, B, Hq, Hkv, seq_lens, q,
                              scale, out, workspace, stream=None):
    _check(lib().tq_decode_attention_paged(kcb.handle, vcb.handle, _ptr(kcache), _ptr(vcache), num_pages, page_size,
                                           _ptr(block_table), block_table.shape[1], B, Hq, Hkv, _ptr(seq_lens),
                                           _ptr(q), float(scale), _ptr(out), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_advance_lengths(seq_lens, B, delta=1, stream=None):
    _check(lib().tq_advance_lengths(_ptr(seq_lens), B, delta, _stream(stream)))


def tq_fail_allocation(nth):
    """Test hook: the nth device allocation of tq_make_codebook from now on fails (-1: off)."""
    _check(lib().tq_fail_allocation(nth))


def tq_set_first_wait_limit(cb, polls):
    """Test use: polls of the first bounded device-side wait of each launch
    with this codebook (0: give up at once, -1: the default)."""
    _check(lib().tq_set_first_wait_limit(cb.handle, polls))


def tq_check_device(cb):
    _check(lib().tq_check_device(cb.handle))


def tq_last_error():
    return lib().tq_last_error().decode()
