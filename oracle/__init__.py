"""ctypes wrapper around the plain CPU oracle (liblsc_oracle.so).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke() and
bench.py's CPU-baseline leg import this package.  The arithmetic lives in
oracle/lsc_oracle.c; this module only marshals numpy arrays.

Pool memory on the oracle side is a dict {layer index: numpy uint8 array of one
GDN layer's region (num_slots pages)}.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

F32, BF16, F16 = 0, 1, 2
ATTENTION, GDN = 0, 1
OK, SOFT_COLD = 0, 1
REJECT_ARG, REJECT_RANGE, REJECT_DUP_DST, REJECT_SRC_IS_DST, REJECT_LAYOUT = -1, -2, -3, -4, -5
NOOP, HIT, MISS = 0, 1, 2

_ESIZE = {F32: 4, BF16: 2, F16: 2}


class _Pool(C.Structure):
    _fields_ = [
        ("num_layers", C.c_int), ("layer_kind", C.POINTER(C.c_int)), ("num_slots", C.c_int),
        ("conv_dim", C.c_int), ("conv_width", C.c_int), ("conv_dtype", C.c_int),
        ("num_v_heads", C.c_int), ("head_v_dim", C.c_int), ("head_k_dim", C.c_int),
        ("ssm_dtype", C.c_int), ("page_bytes", C.c_longlong),
    ]


class _Layout(C.Structure):
    _fields_ = [(n, C.c_longlong) for n in (
        "conv_elems", "conv_bytes", "ssm_elems", "ssm_bytes", "ssm_offset", "payload", "page",
        "conv_stride_elems", "ssm_stride_elems", "region_bytes")] + [("num_gdn", C.c_int)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = C.CDLL(path)
        P = C.c_void_p
        _lib.orc_layout.argtypes = [C.POINTER(_Pool), C.POINTER(_Layout)]
        _lib.orc_classify.argtypes = [C.POINTER(_Pool), P, P, C.c_int, P, C.c_int, P, P]
        _lib.orc_restore.argtypes = [C.POINTER(_Pool), P, P, P, C.c_int, P, C.c_int, P, P]
        _lib.orc_gather.argtypes = [C.POINTER(_Pool), P, P, P, C.c_int, P, P]
        _lib.orc_scatter.argtypes = [C.POINTER(_Pool), P, P, C.c_int, P, P]
        _lib.orc_gdn_decode.argtypes = [C.POINTER(_Pool), P, C.c_int, P, P, P, P, C.c_int, P, P, P]
        _lib.orc_gdn_recurrent.argtypes = [C.POINTER(_Pool), P, C.c_int, P, P, P, C.c_int,
                                           P, P, P, P, P, P]
        _lib.orc_gdn_prefill_conv.argtypes = [C.POINTER(_Pool), P, C.c_int, P, P, P, C.c_int,
                                               P, P, P, P, P]
        _lib.orc_kv_layout.argtypes = [C.POINTER(_KvPool), C.POINTER(_KvLayout)]
        _lib.orc_copy_prefix.argtypes = [C.POINTER(_KvPool), P, P, P, P, C.c_int]
        _lib.orc_bf16_bits.argtypes = [C.c_float]
        _lib.orc_bf16_bits.restype = C.c_ushort
        _lib.orc_num_threads.restype = C.c_int
    return _lib


class _KvPool(C.Structure):
    _fields_ = [("num_layers", C.c_int), ("num_blocks", C.c_int), ("block_tokens", C.c_int),
                ("num_kv_heads", C.c_int), ("head_dim", C.c_int), ("dtype", C.c_int), ("page_bytes", C.c_longlong)]


class _KvLayout(C.Structure):
    _fields_ = [(n, C.c_longlong) for n in ("row_bytes", "payload", "page", "block_stride_elems",
                                             "lane_stride_elems", "region_bytes")]


class KvPool:
    """Oracle-side description of an attention K/V pool."""

    def __init__(self, num_layers, num_blocks, block_tokens, num_kv_heads, head_dim, dtype, page_bytes):
        self.s = _KvPool(num_layers, num_blocks, block_tokens, num_kv_heads, head_dim, dtype, page_bytes)

    def __getattr__(self, name):
        s = self.__dict__.get("s")
        if s is not None and name in dict(_KvPool._fields_):
            return getattr(s, name)
        raise AttributeError(name)


def kv_layout(pool):
    """Returns (rc, dict of _KvLayout fields)."""
    L = _KvLayout()
    rc = lib().orc_kv_layout(C.byref(pool.s), C.byref(L))
    return rc, {n: getattr(L, n) for n, _ in _KvLayout._fields_}


def copy_prefix(pool, regions, src, dst, n_tokens):
    """regions: list of uint8 arrays, one per attention layer (2 lanes each)."""
    src, dst, nt = _c(src, np.int32), _c(dst, np.int32), _c(n_tokens, np.int32)
    ptrs = (C.c_void_p * max(pool.num_layers, 1))()
    for l in range(pool.num_layers):
        r = regions[l]
        assert r.dtype == np.uint8 and r.flags.c_contiguous
        ptrs[l] = r.ctypes.data
    return lib().orc_copy_prefix(C.byref(pool.s), ptrs, _ptr(src), _ptr(dst), _ptr(nt), len(src))


class Pool:
    """Oracle-side description of a state pool (shapes, dtypes, page stride)."""

    def __init__(self, layer_kinds, num_slots, conv_dim, conv_width, conv_dtype,
                 num_v_heads, head_v_dim, head_k_dim, ssm_dtype, page_bytes):
        self.layer_kinds = list(layer_kinds)
        self._kinds = (C.c_int * len(self.layer_kinds))(*self.layer_kinds)
        self.s = _Pool(len(self.layer_kinds), self._kinds, num_slots, conv_dim, conv_width,
                       conv_dtype, num_v_heads, head_v_dim, head_k_dim, ssm_dtype, page_bytes)

    def __getattr__(self, name):
        s = self.__dict__.get("s")
        if s is not None and name in dict(_Pool._fields_):
            return getattr(s, name)
        raise AttributeError(name)

    @property
    def gdn_layers(self):
        return [l for l, k in enumerate(self.layer_kinds) if k == GDN]


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def layout(pool):
    out = _Layout()
    rc = lib().orc_layout(C.byref(pool.s), C.byref(out))
    if rc != OK:
        return rc, None
    return rc, {n: getattr(out, n) for n, _ in _Layout._fields_}


def classify(pool, live, src, nkv, block_size, initialized):
    live, src, nkv = _c(live, np.int32), _c(src, np.int32), _c(nkv, np.int32)
    init = _c(initialized, np.uint8)
    act = np.zeros(len(live), np.int8)
    rc = lib().orc_classify(C.byref(pool.s), _ptr(live), _ptr(src), len(live), _ptr(nkv),
                            block_size, _ptr(init), _ptr(act))
    return rc, act


def restore(pool, regions, live, src, nkv, block_size, initialized, has_initial_state):
    """regions: {layer: uint8 array}; has_initial_state: uint8 array, updated in place."""
    live, src, nkv = _c(live, np.int32), _c(src, np.int32), _c(nkv, np.int32)
    init = _c(initialized, np.uint8)
    assert has_initial_state.dtype == np.uint8 and has_initial_state.flags.c_contiguous
    ptrs = (C.c_void_p * pool.num_layers)()
    for l in range(pool.num_layers):
        r = regions.get(l)
        if r is not None:
            assert r.dtype == np.uint8 and r.flags.c_contiguous
            ptrs[l] = r.ctypes.data
    return lib().orc_restore(C.byref(pool.s), ptrs, _ptr(live), _ptr(src), len(live), _ptr(nkv),
                             block_size, _ptr(init), _ptr(has_initial_state))


def gather(pool, region, idx, has_init=None):
    """Returns (rc, conv_dense uint8 [n, conv_bytes], ssm_dense uint8 [n, ssm_bytes])."""
    _, L = layout(pool)
    idx = _c(idx, np.int32)
    hs = _c(has_init, np.uint8)
    n = len(idx)
    conv = np.full((n, L["conv_bytes"]), 0x5A, np.uint8)
    ssm = np.full((n, L["ssm_bytes"]), 0x5A, np.uint8)
    rc = lib().orc_gather(C.byref(pool.s), _ptr(region), _ptr(idx), _ptr(hs), n, _ptr(conv), _ptr(ssm))
    return rc, conv, ssm


def scatter(pool, region, idx, conv_dense, ssm_dense):
    idx = _c(idx, np.int32)
    conv = _c(conv_dense, np.uint8)
    ssm = _c(ssm_dense, np.uint8)
    return lib().orc_scatter(C.byref(pool.s), _ptr(region), _ptr(idx), len(idx), _ptr(conv), _ptr(ssm))


def gdn_decode(pool, region, idx, has_init, x_raw, conv_w_raw, num_k_heads, alpha, beta):
    """x_raw / conv_w_raw: uint8 or typed arrays holding the conv dtype's bytes.
    Returns (rc, out float32 [n, Hv, dv]); region is updated in place."""
    idx = _c(idx, np.int32)
    hs = _c(has_init, np.uint8)
    x = np.ascontiguousarray(x_raw)
    w = np.ascontiguousarray(conv_w_raw)
    a = _c(alpha, np.float32)
    b = _c(beta, np.float32)
    n = len(idx)
    out = np.full((n, pool.num_v_heads, pool.head_v_dim), np.nan, np.float32)
    rc = lib().orc_gdn_decode(C.byref(pool.s), _ptr(region), n, _ptr(idx), _ptr(hs), _ptr(x),
                              _ptr(w), num_k_heads, _ptr(a), _ptr(b), _ptr(out))
    return rc, out


def gdn_recurrent(pool, region, idx, has_init, cu_seqlens, num_k_heads, q, k, v, alpha, beta):
    """Returns (rc, out float32 [T, Hv, dv]); region is updated in place."""
    idx = _c(idx, np.int32)
    hs = _c(has_init, np.uint8)
    cu = _c(cu_seqlens, np.int32)
    q, k, v = _c(q, np.float32), _c(k, np.float32), _c(v, np.float32)
    a, b = _c(alpha, np.float32), _c(beta, np.float32)
    T = int(cu[-1]) if len(cu) else 0
    out = np.full((T, pool.num_v_heads, pool.head_v_dim), np.nan, np.float32)
    rc = lib().orc_gdn_recurrent(C.byref(pool.s), _ptr(region), len(idx), _ptr(idx), _ptr(hs),
                                 _ptr(cu), num_k_heads, _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                 _ptr(b), _ptr(out))
    return rc, out


def gdn_prefill_conv(pool, region, idx, has_init, cu_seqlens, num_k_heads, x_raw, conv_w_raw):
    """x_raw [T, conv_dim] / conv_w_raw [conv_dim, W]: arrays holding the conv
    dtype's bytes.  Returns (rc, q, k [T, Hk, dk], v [T, Hv, dv] float32); the
    slots' conv states are updated in place."""
    idx = _c(idx, np.int32)
    hs = _c(has_init, np.uint8)
    cu = _c(cu_seqlens, np.int32)
    x = np.ascontiguousarray(x_raw)
    w = np.ascontiguousarray(conv_w_raw)
    T = int(cu[-1]) if len(cu) else 0
    q = np.full((T, num_k_heads, pool.head_k_dim), np.nan, np.float32)
    k = np.full((T, num_k_heads, pool.head_k_dim), np.nan, np.float32)
    v = np.full((T, pool.num_v_heads, pool.head_v_dim), np.nan, np.float32)
    rc = lib().orc_gdn_prefill_conv(C.byref(pool.s), _ptr(region), len(idx), _ptr(idx), _ptr(hs),
                                    _ptr(cu), num_k_heads, _ptr(x), _ptr(w), _ptr(q), _ptr(k), _ptr(v))
    return rc, q, k, v


def bf16_bits(f):
    return lib().orc_bf16_bits(float(f))


def num_threads():
    return lib().orc_num_threads()


def esize(dtype):
    return _ESIZE[dtype]
