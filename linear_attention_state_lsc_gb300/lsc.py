"""ctypes binding of liblsc (include/lsc.h, include/lsc_prefix_cache.h,
include/lsc_kv.h, include/lsc_store.h), same names as the C ABI.

Argument marshalling only: every step of the hot path runs in the CUDA kernels
of liblsc.so.  Pointers are plain integers; torch tensors, numpy arrays and
None (NULL) are accepted wherever a pointer is expected.  Loading fails loudly
when liblsc.so has not been built -- there is no fallback.
"""
import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblsc.so")

# return codes (include/lsc.h)
LSC_OK = 0
LSC_SOFT_COLD = 1
LSC_ERR_INVALID_ARG = -1
LSC_ERR_OUT_OF_RANGE = -2
LSC_ERR_DUP_DST = -3
LSC_ERR_SRC_IS_DST = -4
LSC_ERR_MISALIGNED = -5
LSC_ERR_STATELESS_LAYER = -6
LSC_ERR_UNSUPPORTED = -7
LSC_ERR_CUDA = -8
LSC_ERR_DEV_TIMEOUT = -9
LSC_ERR_NO_MEMORY = -10
LSC_ERR_LAYOUT = -11
LSC_ERR_WRONG_DEVICE = -12
LSC_ERR_NO_SLOT = -13
LSC_ERR_ORDER = -14
LSC_ERR_NO_SPACE = -15
LSC_ERR_CORRUPT = -16
LSC_ERR_NOT_FOUND = -17
LSC_ERR_IO = -18

# prefix-cache slot states (include/lsc_prefix_cache.h)
LSC_SLOT_FREE, LSC_SLOT_LIVE, LSC_SLOT_CHECKPOINT, LSC_SLOT_RESERVED = 0, 1, 2, 3

LSC_LAYER_ATTENTION, LSC_LAYER_GDN = 0, 1
LSC_RECURRENT_AUTO, LSC_RECURRENT_TOKEN, LSC_RECURRENT_CHUNKED = 0, 1, 2
LSC_DECODE_EARLY_STATE = 1
LSC_F32, LSC_BF16, LSC_F16 = 0, 1, 2


class LscError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {lsc_error_string(code)} ({code})")


class LinearStateCacheOp(C.Structure):
    _fields_ = [("linear_state_id", C.c_int32), ("restore_src_slot_id", C.c_int32),
                ("restore_prefix_hash", C.c_uint64), ("save_prefix_hash", C.c_uint64),
                ("save_dst_slot_id", C.c_int32), ("reserved", C.c_int32)]


# numpy view of an array of LinearStateCacheOp (same layout, 32 bytes)
OP_DTYPE = np.dtype([("linear_state_id", "<i4"), ("restore_src_slot_id", "<i4"),
                     ("restore_prefix_hash", "<u8"), ("save_prefix_hash", "<u8"),
                     ("save_dst_slot_id", "<i4"), ("reserved", "<i4")], align=True)


class lsc_pool_desc(C.Structure):
    _fields_ = [("num_layers", C.c_int32), ("layer_kinds", C.POINTER(C.c_int32)),
                ("num_slots", C.c_int32), ("conv_dim", C.c_int32), ("conv_width", C.c_int32),
                ("conv_dtype", C.c_int32), ("num_v_heads", C.c_int32), ("head_v_dim", C.c_int32),
                ("head_k_dim", C.c_int32), ("ssm_dtype", C.c_int32), ("page_bytes", C.c_int64)]


class lsc_layer_view(C.Structure):
    _fields_ = [("region", C.c_void_p), ("region_bytes", C.c_int64), ("gdn_index", C.c_int32),
                ("conv_dtype", C.c_int32), ("ssm_dtype", C.c_int32),
                ("conv", C.c_void_p), ("conv_shape", C.c_int64 * 3), ("conv_strides", C.c_int64 * 3),
                ("conv_storage_offset", C.c_int64),
                ("ssm", C.c_void_p), ("ssm_shape", C.c_int64 * 4), ("ssm_strides", C.c_int64 * 4),
                ("ssm_storage_offset", C.c_int64),
                ("page_bytes", C.c_int64), ("payload_bytes", C.c_int64), ("conv_bytes", C.c_int64),
                ("ssm_offset_bytes", C.c_int64), ("ssm_bytes", C.c_int64)]


class lsc_restore_report(C.Structure):
    _fields_ = [("n_hit", C.c_int32), ("n_miss", C.c_int32), ("n_noop", C.c_int32),
                ("soft_cold", C.c_int32), ("launches", C.c_int32), ("reserved", C.c_int32),
                ("bytes_copied", C.c_int64)]


class lsc_gdn_decode_args(C.Structure):
    _fields_ = [("n", C.c_int32), ("num_k_heads", C.c_int32), ("idx", C.c_void_p),
                ("has_init", C.c_void_p), ("x", C.c_void_p), ("conv_weight", C.c_void_p),
                ("alpha", C.c_void_p), ("beta", C.c_void_p), ("out", C.c_void_p), ("flags", C.c_uint32)]


class lsc_gdn_recurrent_args(C.Structure):
    _fields_ = [("n_seq", C.c_int32), ("num_k_heads", C.c_int32), ("total_tokens", C.c_int32),
                ("algorithm", C.c_int32), ("idx", C.c_void_p), ("has_init", C.c_void_p),
                ("cu_seqlens", C.c_void_p), ("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p),
                ("alpha", C.c_void_p), ("beta", C.c_void_p), ("out", C.c_void_p),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t)]


class lsc_pc_row(C.Structure):
    _fields_ = [("seq_id", C.c_int64), ("restore_prefix_hash", C.c_uint64),
                ("save_prefix_hash", C.c_uint64), ("tokens_after_step", C.c_int64)]


class lsc_pc_report(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("restore_hit", "restore_miss", "save", "skip_duplicate",
                                          "skip_cached", "skip_unaligned", "skip_no_slot", "reserved")]


class lsc_gdn_prefill_conv_args(C.Structure):
    _fields_ = [("n_seq", C.c_int32), ("num_k_heads", C.c_int32), ("total_tokens", C.c_int32),
                ("reserved", C.c_int32), ("idx", C.c_void_p), ("has_init", C.c_void_p),
                ("cu_seqlens", C.c_void_p), ("x", C.c_void_p), ("conv_weight", C.c_void_p),
                ("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p)]


class lsc_kv_pool_desc(C.Structure):
    _fields_ = [("num_layers", C.c_int32), ("num_blocks", C.c_int32), ("block_tokens", C.c_int32),
                ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("dtype", C.c_int32),
                ("page_bytes", C.c_int64)]


class lsc_kv_layer_view(C.Structure):
    _fields_ = [("region", C.c_void_p), ("region_bytes", C.c_int64), ("k", C.c_void_p), ("v", C.c_void_p),
                ("shape", C.c_int64 * 4), ("strides", C.c_int64 * 4), ("lane_stride", C.c_int64),
                ("page_bytes", C.c_int64), ("payload_bytes", C.c_int64), ("row_bytes", C.c_int64),
                ("dtype", C.c_int32), ("reserved", C.c_int32)]


# numpy view of an array of lsc_kv_copy_op
KV_OP_DTYPE = np.dtype([("src_block", "<i4"), ("dst_block", "<i4"), ("n_tokens", "<i4"), ("reserved", "<i4")])


_lib = None


def load():
    """Load liblsc.so (built by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"liblsc.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = C.CDLL(LIB_PATH)
    P, I32, I64 = C.c_void_p, C.c_int32, C.c_int64
    sig = {
        "lsc_pool_required_bytes": ([C.POINTER(lsc_pool_desc), C.POINTER(C.c_size_t)], C.c_int),
        "lsc_pool_create": ([C.POINTER(lsc_pool_desc), P, C.c_size_t, C.POINTER(P)], C.c_int),
        "lsc_pool_destroy": ([P], C.c_int),
        "lsc_pool_layer_view": ([P, I32, C.POINTER(lsc_layer_view)], C.c_int),
        "lsc_pool_num_slots": ([P], I32),
        "lsc_pool_status": ([P, P, C.POINTER(I32)], C.c_int),
        "lsc_restore_classify": ([P, P, I32, P, I32, P, P, C.POINTER(lsc_restore_report)], C.c_int),
        "lsc_restore": ([P, P, I32, P, I32, P, P, P, P, C.POINTER(lsc_restore_report)], C.c_int),
        "lsc_gather": ([P, I32, P, P, I32, P, P, P], C.c_int),
        "lsc_scatter": ([P, I32, P, I32, P, P, P], C.c_int),
        "lsc_gdn_decode": ([P, I32, C.POINTER(lsc_gdn_decode_args), P], C.c_int),
        "lsc_gdn_recurrent": ([P, I32, C.POINTER(lsc_gdn_recurrent_args), P], C.c_int),
        "lsc_gdn_recurrent_workspace_bytes": ([P, C.POINTER(lsc_gdn_recurrent_args), C.POINTER(C.c_size_t)],
                                              C.c_int),
        "lsc_gdn_recurrent_noalloc": ([P, I32, C.POINTER(lsc_gdn_recurrent_args), P], C.c_int),
        "lsc_gdn_prefill_conv": ([P, I32, C.POINTER(lsc_gdn_prefill_conv_args), P], C.c_int),
        "lsc_kv_pool_required_bytes": ([C.POINTER(lsc_kv_pool_desc), C.POINTER(C.c_size_t)], C.c_int),
        "lsc_kv_pool_create": ([C.POINTER(lsc_kv_pool_desc), P, C.c_size_t, C.POINTER(P)], C.c_int),
        "lsc_kv_pool_destroy": ([P], C.c_int),
        "lsc_kv_pool_layer_view": ([P, I32, C.POINTER(lsc_kv_layer_view)], C.c_int),
        "lsc_copy_prefix": ([P, P, I32, P, P, C.POINTER(I64)], C.c_int),
        "lsc_pc_create": ([I32, I32, C.POINTER(P)], C.c_int),
        "lsc_pc_destroy": ([P], C.c_int),
        "lsc_pc_allocate_live_slot": ([P, I64, C.POINTER(I32)], C.c_int),
        "lsc_pc_release_sequence": ([P, I64], C.c_int),
        "lsc_pc_match": ([P, C.c_uint64, C.POINTER(I32)], C.c_int),
        "lsc_pc_unpin": ([P, I32], C.c_int),
        "lsc_pc_resolve": ([P, P, I32, P, P, C.POINTER(lsc_pc_report)], C.c_int),
        "lsc_pc_commit": ([P], C.c_int),
        "lsc_pc_slot": ([P, I32, C.POINTER(I32), C.POINTER(I32), C.POINTER(C.c_uint64)], C.c_int),
        "lsc_pc_sequence": ([P, I64, C.POINTER(I32), C.POINTER(I32)], C.c_int),
        "lsc_pc_counts": ([P, C.POINTER(I32), C.POINTER(I32), C.POINTER(I32), C.POINTER(I32)], C.c_int),
        "lsc_error_string": ([C.c_int], C.c_char_p),
        "lsc_build_info": ([], C.c_char_p),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def ptr(x):
    """Integer address of a tensor / array / int; None -> 0 (NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    if hasattr(x, "data_ptr"):
        return x.data_ptr() or None
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(type(x))


def _stream(s):
    if s is None or isinstance(s, int):
        return s or None
    return s.cuda_stream or None  # torch.cuda.Stream


def _event(e):
    if e is None or isinstance(e, int):
        return e or None
    return e.cuda_event or None  # torch.cuda.Event (must have been created/recorded once)


def lsc_error_string(code):
    return load().lsc_error_string(int(code)).decode()


def lsc_build_info():
    return load().lsc_build_info().decode()


def make_pool_desc(layer_kinds, num_slots, conv_dim, conv_width, conv_dtype, num_v_heads,
                   head_v_dim, head_k_dim, ssm_dtype, page_bytes):
    kinds = (C.c_int32 * len(layer_kinds))(*layer_kinds)
    d = lsc_pool_desc(len(layer_kinds), kinds, num_slots, conv_dim, conv_width, conv_dtype,
                      num_v_heads, head_v_dim, head_k_dim, ssm_dtype, page_bytes)
    d._keep = kinds
    return d


def lsc_pool_required_bytes(desc):
    n = C.c_size_t(0)
    rc = load().lsc_pool_required_bytes(C.byref(desc), C.byref(n))
    if rc < 0:
        raise LscError(rc, "lsc_pool_required_bytes")
    return n.value


def lsc_pool_create(desc, device_base=None, base_bytes=0):
    """Returns (rc, pool handle or None)."""
    h = C.c_void_p()
    rc = load().lsc_pool_create(C.byref(desc), ptr(device_base), base_bytes, C.byref(h))
    return rc, (h.value if rc == LSC_OK else None)


def lsc_pool_destroy(pool):
    return load().lsc_pool_destroy(pool)


def lsc_pool_layer_view(pool, layer):
    v = lsc_layer_view()
    rc = load().lsc_pool_layer_view(pool, layer, C.byref(v))
    return rc, v


def lsc_pool_num_slots(pool):
    return load().lsc_pool_num_slots(pool)


def lsc_pool_status(pool, stream=None):
    s = C.c_int32(0)
    rc = load().lsc_pool_status(pool, _stream(stream), C.byref(s))
    if rc < 0:
        raise LscError(rc, "lsc_pool_status")
    return s.value


def ops_array(live, src, restore_hash=None, save_hash=None, save_slot=None):
    """numpy array of LinearStateCacheOp records."""
    n = len(live)
    a = np.zeros(n, OP_DTYPE)
    a["linear_state_id"] = live
    a["restore_src_slot_id"] = src
    a["restore_prefix_hash"] = 0 if restore_hash is None else restore_hash
    a["save_prefix_hash"] = 0 if save_hash is None else save_hash
    a["save_dst_slot_id"] = -1 if save_slot is None else save_slot
    return a


def _host(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def lsc_restore_classify(pool, ops, n_kv_cache_tokens, block_size, linear_state_initialized):
    """Returns (rc, actions int8 [n] (0 no-op, 1 hit, 2 miss), lsc_restore_report)."""
    assert ops.dtype == OP_DTYPE
    nkv = _host(n_kv_cache_tokens, np.int32)
    init = _host(linear_state_initialized, np.uint8)
    act = np.zeros(len(ops), np.int8)
    rep = lsc_restore_report()
    rc = load().lsc_restore_classify(pool, ops.ctypes.data, len(ops), nkv.ctypes.data, block_size,
                                     init.ctypes.data, act.ctypes.data, C.byref(rep))
    return rc, act, rep


def lsc_restore(pool, ops, n_kv_cache_tokens, block_size, linear_state_initialized,
                has_initial_state, prepare_stream=None, done_event=None):
    """ops / n_kv / initialized on the host; has_initial_state a device uint8
    tensor (pre-filled).  Returns (rc, lsc_restore_report)."""
    assert ops.dtype == OP_DTYPE
    ops = np.ascontiguousarray(ops)
    nkv = _host(n_kv_cache_tokens, np.int32)
    init = _host(linear_state_initialized, np.uint8)
    rep = lsc_restore_report()
    rc = load().lsc_restore(pool, ops.ctypes.data, len(ops), nkv.ctypes.data, block_size,
                            init.ctypes.data, ptr(has_initial_state), _stream(prepare_stream),
                            _event(done_event), C.byref(rep))
    return rc, rep


def lsc_gather(pool, layer, idx, has_init, n, conv_dense, ssm_dense, stream=None):
    return load().lsc_gather(pool, layer, ptr(idx), ptr(has_init), n, ptr(conv_dense),
                             ptr(ssm_dense), _stream(stream))


def lsc_scatter(pool, layer, idx, n, conv_dense, ssm_dense, stream=None):
    return load().lsc_scatter(pool, layer, ptr(idx), n, ptr(conv_dense), ptr(ssm_dense),
                              _stream(stream))


def decode_args(n, num_k_heads, idx, has_init, x, conv_weight, alpha, beta, out, flags=0):
    return lsc_gdn_decode_args(n, num_k_heads, ptr(idx), ptr(has_init), ptr(x), ptr(conv_weight),
                               ptr(alpha), ptr(beta), ptr(out), flags)


def lsc_gdn_decode(pool, layer, args, stream=None):
    return load().lsc_gdn_decode(pool, layer, C.byref(args), _stream(stream))


def recurrent_args(n_seq, num_k_heads, total_tokens, idx, has_init, cu_seqlens, q, k, v, alpha,
                   beta, out, algorithm=0, workspace=None, workspace_bytes=0):
    return lsc_gdn_recurrent_args(n_seq, num_k_heads, total_tokens, algorithm, ptr(idx), ptr(has_init),
                                  ptr(cu_seqlens), ptr(q), ptr(k), ptr(v), ptr(alpha), ptr(beta),
                                  ptr(out), ptr(workspace), workspace_bytes)


def lsc_gdn_recurrent_noalloc(pool, layer, args, stream=None):
    return load().lsc_gdn_recurrent_noalloc(pool, layer, C.byref(args), _stream(stream))


def lsc_gdn_recurrent_workspace_bytes(pool, args):
    n = C.c_size_t(0)
    rc = load().lsc_gdn_recurrent_workspace_bytes(pool, C.byref(args), C.byref(n))
    return rc, n.value


def lsc_gdn_recurrent(pool, layer, args, stream=None):
    return load().lsc_gdn_recurrent(pool, layer, C.byref(args), _stream(stream))


def prefill_conv_args(n_seq, num_k_heads, total_tokens, idx, has_init, cu_seqlens, x, conv_weight, q, k, v):
    return lsc_gdn_prefill_conv_args(n_seq, num_k_heads, total_tokens, 0, ptr(idx), ptr(has_init),
                                     ptr(cu_seqlens), ptr(x), ptr(conv_weight), ptr(q), ptr(k), ptr(v))


def lsc_gdn_prefill_conv(pool, layer, args, stream=None):
    return load().lsc_gdn_prefill_conv(pool, layer, C.byref(args), _stream(stream))


# ---- scheduler-side prefix cache (include/lsc_prefix_cache.h) ---------------

PC_ROW_DTYPE = np.dtype([("seq_id", "<i8"), ("restore_prefix_hash", "<u8"),
                         ("save_prefix_hash", "<u8"), ("tokens_after_step", "<i8")])


def lsc_pc_create(num_slots, block_size):
    """Returns (rc, cache handle)."""
    h = C.c_void_p()
    rc = load().lsc_pc_create(num_slots, block_size, C.byref(h))
    return rc, h.value


def lsc_pc_destroy(pc):
    return load().lsc_pc_destroy(pc)


def lsc_pc_allocate_live_slot(pc, seq_id):
    """Returns (rc, slot)."""
    s = C.c_int32(-1)
    rc = load().lsc_pc_allocate_live_slot(pc, seq_id, C.byref(s))
    return rc, s.value


def lsc_pc_release_sequence(pc, seq_id):
    return load().lsc_pc_release_sequence(pc, seq_id)


def lsc_pc_match(pc, prefix_hash):
    """Returns (rc, slot or -1)."""
    s = C.c_int32(-1)
    rc = load().lsc_pc_match(pc, prefix_hash, C.byref(s))
    return rc, s.value


def lsc_pc_unpin(pc, slot):
    return load().lsc_pc_unpin(pc, slot)


def pc_rows(seq_ids, restore_hashes, save_hashes, tokens_after_step):
    rows = np.zeros(len(seq_ids), PC_ROW_DTYPE)
    rows["seq_id"] = seq_ids
    rows["restore_prefix_hash"] = restore_hashes
    rows["save_prefix_hash"] = save_hashes
    rows["tokens_after_step"] = tokens_after_step
    return rows


def lsc_pc_resolve(pc, rows):
    """rows: a PC_ROW_DTYPE array.  Returns (rc, ops OP_DTYPE [n],
    linear_state_initialized uint8 [n], lsc_pc_report)."""
    assert rows.dtype == PC_ROW_DTYPE
    rows = np.ascontiguousarray(rows)
    ops = np.zeros(len(rows), OP_DTYPE)
    init = np.zeros(len(rows), np.uint8)
    rep = lsc_pc_report()
    rc = load().lsc_pc_resolve(pc, rows.ctypes.data, len(rows), ops.ctypes.data, init.ctypes.data,
                               C.byref(rep))
    return rc, ops, init, rep


def lsc_pc_commit(pc):
    return load().lsc_pc_commit(pc)


def lsc_pc_slot(pc, slot):
    """Returns (rc, state, pins, hash)."""
    st, pins, h = C.c_int32(), C.c_int32(), C.c_uint64()
    rc = load().lsc_pc_slot(pc, slot, C.byref(st), C.byref(pins), C.byref(h))
    return rc, st.value, pins.value, h.value


def lsc_pc_sequence(pc, seq_id):
    """Returns (rc, live slot, linear_state_initialized)."""
    s, i = C.c_int32(-1), C.c_int32(0)
    rc = load().lsc_pc_sequence(pc, seq_id, C.byref(s), C.byref(i))
    return rc, s.value, i.value


def lsc_pc_counts(pc):
    """Returns (rc, (free, live, checkpoint, reserved))."""
    c = [C.c_int32() for _ in range(4)]
    rc = load().lsc_pc_counts(pc, *[C.byref(x) for x in c])
    return rc, tuple(x.value for x in c)


# ---- attention K/V block pool (include/lsc_kv.h) ------------------------------

def lsc_kv_pool_required_bytes(desc):
    n = C.c_size_t(0)
    rc = load().lsc_kv_pool_required_bytes(C.byref(desc), C.byref(n))
    if rc != LSC_OK:
        raise LscError(rc, "lsc_kv_pool_required_bytes")
    return n.value


def lsc_kv_pool_create(desc, device_base=None, base_bytes=0):
    """Returns (rc, pool handle)."""
    h = C.c_void_p()
    rc = load().lsc_kv_pool_create(C.byref(desc), ptr(device_base), base_bytes, C.byref(h))
    return rc, h.value


def lsc_kv_pool_destroy(pool):
    return load().lsc_kv_pool_destroy(pool)


def lsc_kv_pool_layer_view(pool, layer):
    v = lsc_kv_layer_view()
    rc = load().lsc_kv_pool_layer_view(pool, layer, C.byref(v))
    return rc, v


def kv_ops(src_blocks, dst_blocks, n_tokens):
    ops = np.zeros(len(src_blocks), KV_OP_DTYPE)
    ops["src_block"] = src_blocks
    ops["dst_block"] = dst_blocks
    ops["n_tokens"] = n_tokens
    return ops


def lsc_copy_prefix(pool, ops, stream=None, done_event=None):
    """ops: a KV_OP_DTYPE array on the host.  Returns (rc, bytes_copied)."""
    assert ops.dtype == KV_OP_DTYPE
    ops = np.ascontiguousarray(ops)
    b = C.c_int64(0)
    rc = load().lsc_copy_prefix(pool, ops.ctypes.data, len(ops), _stream(stream), _event(done_event), C.byref(b))
    return rc, b.value


# ---- snapshot store (include/lsc_store.h) -------------------------------------

class lsc_store_stats(C.Structure):
    _fields_ = [("used_bytes", C.c_int64), ("quota_bytes", C.c_int64), ("n_blobs", C.c_int32),
                ("n_entries", C.c_int32), ("n_unreferenced", C.c_int32), ("n_pinned", C.c_int32)]


_STORE_SIG = {
    "lsc_store_open": ([C.c_char_p, C.c_uint64, C.c_int64, C.POINTER(C.c_void_p)], C.c_int),
    "lsc_store_close": ([C.c_void_p], C.c_int),
    "lsc_store_put_blob": ([C.c_void_p, C.c_uint64, C.c_int32, C.c_void_p, C.c_int64], C.c_int),
    "lsc_store_get_blob": ([C.c_void_p, C.c_uint64, C.c_void_p, C.c_int64, C.POINTER(C.c_int64),
                            C.POINTER(C.c_int32)], C.c_int),
    "lsc_store_blob_size": ([C.c_void_p, C.c_uint64, C.POINTER(C.c_int64)], C.c_int),
    "lsc_store_put_entry": ([C.c_void_p, C.c_uint64, C.c_void_p, C.c_int32], C.c_int),
    "lsc_store_get_entry": ([C.c_void_p, C.c_uint64, C.c_void_p, C.c_int32, C.POINTER(C.c_int32)], C.c_int),
    "lsc_store_drop_entry": ([C.c_void_p, C.c_uint64], C.c_int),
    "lsc_store_pin": ([C.c_void_p, C.c_uint64], C.c_int),
    "lsc_store_unpin": ([C.c_void_p, C.c_uint64], C.c_int),
    "lsc_store_stats_get": ([C.c_void_p, C.POINTER(lsc_store_stats)], C.c_int),
    "lsc_store_save_state": ([C.c_void_p, C.c_uint64, C.c_void_p, C.c_int32, C.c_void_p], C.c_int),
    "lsc_store_load_state": ([C.c_void_p, C.c_uint64, C.c_void_p, C.c_int32, C.c_void_p], C.c_int),
}


def _store_fn(name):
    lib = load()
    f = getattr(lib, name)
    if name in _STORE_SIG and f.argtypes is None:
        f.argtypes, f.restype = _STORE_SIG[name]
    return f


def lsc_store_open(directory, namespace_digest, quota_bytes):
    """Returns (rc, store handle)."""
    h = C.c_void_p()
    rc = _store_fn("lsc_store_open")(os.fsencode(directory), namespace_digest, quota_bytes, C.byref(h))
    return rc, h.value


def lsc_store_close(store):
    return _store_fn("lsc_store_close")(store)


def lsc_store_put_blob(store, key, kind, data):
    """data: a bytes-like object or numpy array (host)."""
    a = np.frombuffer(bytes(data), np.uint8) if not isinstance(data, np.ndarray) else np.ascontiguousarray(data)
    return _store_fn("lsc_store_put_blob")(store, key, kind, a.ctypes.data if a.size else None, a.nbytes)


def lsc_store_get_blob(store, key):
    """Returns (rc, kind, payload bytes or None)."""
    n = C.c_int64(0)
    rc = _store_fn("lsc_store_blob_size")(store, key, C.byref(n))
    if rc != LSC_OK:
        return rc, None, None
    buf = np.zeros(max(n.value, 1), np.uint8)
    kind = C.c_int32(-1)
    rc = _store_fn("lsc_store_get_blob")(store, key, buf.ctypes.data, buf.nbytes, C.byref(n), C.byref(kind))
    return rc, kind.value, (bytes(buf[:n.value]) if rc == LSC_OK else None)


def lsc_store_put_entry(store, key, blob_keys):
    a = np.ascontiguousarray(blob_keys, dtype=np.uint64)
    return _store_fn("lsc_store_put_entry")(store, key, a.ctypes.data if a.size else None, len(a))


def lsc_store_get_entry(store, key):
    """Returns (rc, list of blob keys)."""
    n = C.c_int32(0)
    buf = np.zeros(4096, np.uint64)
    rc = _store_fn("lsc_store_get_entry")(store, key, buf.ctypes.data, len(buf), C.byref(n))
    return rc, [int(x) for x in buf[:n.value]] if rc == LSC_OK else []


def lsc_store_drop_entry(store, key):
    return _store_fn("lsc_store_drop_entry")(store, key)


def lsc_store_pin(store, key):
    return _store_fn("lsc_store_pin")(store, key)


def lsc_store_unpin(store, key):
    return _store_fn("lsc_store_unpin")(store, key)


def lsc_store_stats_get(store):
    st = lsc_store_stats()
    rc = _store_fn("lsc_store_stats_get")(store, C.byref(st))
    return rc, st


def lsc_store_save_state(store, key, pool, slot, stream=None):
    return _store_fn("lsc_store_save_state")(store, key, pool, slot, _stream(stream))


def lsc_store_load_state(store, key, pool, slot, stream=None):
    return _store_fn("lsc_store_load_state")(store, key, pool, slot, _stream(stream))
