"""C-ABI checks that need no GPU: the library loads and exports every symbol the
header declares, the struct layouts agree, and the host logic (layout, views,
row classification, validation, error codes, the layout log) matches the
oracle.  No call here enqueues device work."""
import ctypes
import os
import re
import subprocess
import sys

import numpy as np
import pytest

import oracle
from linear_attention_state_lsc_gb300 import lsc as L
from linear_attention_state_lsc_gb300 import workloads as W

from _util import gpu_present, lib_desc, oracle_layout, oracle_pool, ops_of

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]
FAKE_BASE = 1 << 40  # 256 B aligned, never dereferenced: host-only pools


def declared_functions():
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(lsc_[a-z_]+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol(lsc):
    names = declared_functions()
    assert len(names) >= 25 and "lsc_pc_resolve" in names
    lib = ctypes.CDLL(L.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (lsc_\w+)", out))
    assert set(names) <= exported


def test_struct_layouts(lsc):
    assert ctypes.sizeof(L.LinearStateCacheOp) == 32 == L.OP_DTYPE.itemsize
    assert L.OP_DTYPE.fields["save_dst_slot_id"][1] == ctypes.sizeof(ctypes.c_int32) * 2 + 16
    assert ctypes.sizeof(L.lsc_restore_report) == 32
    assert "sm_103a" in L.lsc_build_info()


def test_error_strings(lsc):
    for code in range(-18, 2):
        s = L.lsc_error_string(code)
        assert s and s != "unknown error", code
    assert L.lsc_error_string(-99) == "unknown error"


def host_pool(w, layers=None):
    rc, pool = L.lsc_pool_create(lib_desc(w, layers), FAKE_BASE, 1 << 44)
    assert rc == L.LSC_OK, L.lsc_error_string(rc)
    return pool


@pytest.mark.parametrize("name", ["c0", "c0p", "c1", "c2", "c3", "s1", "s2", "s3", "s4"])
def test_layer_views_match_oracle_layout(lsc, name):
    w = W.get(name) if name.startswith("c") else W.small(name)
    Lo = oracle_layout(w)
    pool = host_pool(w)
    esc, ess = W.ESIZE[w.conv_dtype], W.ESIZE[w.ssm_dtype]
    assert L.lsc_pool_required_bytes(lib_desc(w)) == Lo["num_gdn"] * Lo["region_bytes"]
    g = 0
    for l, kind in enumerate(w.layers):
        rc, v = L.lsc_pool_layer_view(pool, l)
        if kind == W.ATTN:
            assert rc == L.LSC_ERR_STATELESS_LAYER
            continue
        assert rc == L.LSC_OK
        assert v.gdn_index == g
        assert v.region == FAKE_BASE + g * Lo["region_bytes"]
        assert v.region_bytes == Lo["region_bytes"]
        assert list(v.conv_shape) == [w.num_slots, w.conv_dim, w.conv_width - 1]
        assert list(v.conv_strides) == [Lo["conv_stride_elems"], w.conv_width - 1, 1]
        assert list(v.ssm_shape) == [w.num_slots, w.num_v_heads, w.head_v_dim, w.head_k_dim]
        assert list(v.ssm_strides) == [Lo["ssm_stride_elems"], w.head_v_dim * w.head_k_dim, w.head_k_dim, 1]
        assert v.ssm - v.region == Lo["ssm_offset"] and v.ssm_storage_offset * ess == Lo["ssm_offset"]
        assert v.conv == v.region and v.conv_storage_offset == 0
        assert v.payload_bytes == Lo["payload"] and v.conv_bytes == Lo["conv_bytes"]
        assert v.ssm_bytes == Lo["ssm_bytes"]
        g += 1
    assert L.lsc_pool_layer_view(pool, len(w.layers))[0] == L.LSC_ERR_OUT_OF_RANGE
    assert L.lsc_pool_num_slots(pool) == w.num_slots
    assert L.lsc_pool_destroy(pool) == L.LSC_OK


def test_worked_block_stride_example_through_the_library(lsc):
    """vLLM-Ascend "非连续 KV Cache" §3.4: a 48-element fp16 view in a 128 B page
    has a slot stride of 64 elements."""
    d = L.make_pool_desc([L.LSC_LAYER_GDN], 4, 16, 4, L.LSC_F16, 1, 2, 2, L.LSC_F32, 128)
    rc, pool = L.lsc_pool_create(d, FAKE_BASE, 4 * 128)
    assert rc == L.LSC_OK
    rc, v = L.lsc_pool_layer_view(pool, 0)
    assert rc == L.LSC_OK
    assert v.conv_strides[0] == 64 and v.conv_shape[1] * v.conv_shape[2] == 48
    assert v.ssm_strides[0] == 32
    L.lsc_pool_destroy(pool)


@pytest.mark.parametrize("page,code", [(100, L.LSC_ERR_LAYOUT), (130, L.LSC_ERR_LAYOUT), (136, L.LSC_ERR_MISALIGNED)])
def test_pool_rejects_bad_pages(lsc, page, code):
    d = L.make_pool_desc([L.LSC_LAYER_GDN], 4, 16, 4, L.LSC_F16, 1, 2, 2, L.LSC_F32, page)
    assert L.lsc_pool_create(d, FAKE_BASE, 1 << 20)[0] == code


def test_pool_rejects_bad_base_and_args(lsc):
    w = W.get("c0")
    assert L.lsc_pool_create(lib_desc(w), FAKE_BASE + 8, 1 << 20)[0] == L.LSC_ERR_MISALIGNED
    assert L.lsc_pool_create(lib_desc(w), FAKE_BASE, 100)[0] == L.LSC_ERR_NO_MEMORY
    bad = lib_desc(w)
    bad.conv_width = 1
    assert L.lsc_pool_create(bad, FAKE_BASE, 1 << 20)[0] == L.LSC_ERR_INVALID_ARG
    bad = lib_desc(w)
    bad.ssm_dtype = 7
    assert L.lsc_pool_create(bad, FAKE_BASE, 1 << 20)[0] == L.LSC_ERR_INVALID_ARG


def _classify_both(w, rows, layers=None):
    pool = host_pool(w, layers)
    rc_l, act_l, rep = L.lsc_restore_classify(pool, ops_of(rows), rows.nkv, rows.block_size, rows.initialized)
    rc_o, act_o = oracle.classify(oracle_pool(w, layers), rows.live, rows.src, rows.nkv, rows.block_size,
                                  rows.initialized)
    L.lsc_pool_destroy(pool)
    return rc_l, act_l, rep, rc_o, act_o


@pytest.mark.parametrize("case", ["combos", "c0", "c1", "c3"])
def test_classification_matches_oracle(lsc, case):
    if case == "combos":
        w = W.get("c0")
        w.num_slots = 40
        rows = W.combo_rows(40, 16, seed=9)
    else:
        w = W.get(case)
        rows = W.restore_rows(case)
    rc_l, act_l, rep, rc_o, act_o = _classify_both(w, rows)
    assert rc_l == L.LSC_OK and rc_o == oracle.OK
    np.testing.assert_array_equal(act_l, act_o)  # both use 0 no-op, 1 hit, 2 miss
    assert rep.n_hit == (act_o == oracle.HIT).sum() and rep.n_miss == (act_o == oracle.MISS).sum()
    assert rep.n_noop == (act_o == oracle.NOOP).sum()
    Lo = oracle_layout(w)
    assert rep.bytes_copied == rep.n_hit * Lo["num_gdn"] * (Lo["conv_bytes"] + Lo["ssm_bytes"])
    if case == "c3":
        assert (rep.n_hit, rep.n_miss, rep.n_noop) == (205, 154, 153)
    if case == "c1":
        assert rep.n_hit == 64


ERRMAP = {oracle.REJECT_RANGE: L.LSC_ERR_OUT_OF_RANGE, oracle.REJECT_DUP_DST: L.LSC_ERR_DUP_DST,
          oracle.REJECT_SRC_IS_DST: L.LSC_ERR_SRC_IS_DST, oracle.REJECT_ARG: L.LSC_ERR_INVALID_ARG}


@pytest.mark.parametrize("case", ["range_dst", "range_src", "neg_dst", "dup_dst", "src_is_dst", "src_is_other_dst",
                                  "dup_src_ok", "noop_out_of_range_ok"])
def test_validation_matches_oracle(lsc, case):
    w = W.get("c0")
    live = np.array([1, 2, 3], np.int32)
    src = np.array([10, 11, 12], np.int32)
    nkv = np.array([16, 16, 16], np.int32)
    init = np.zeros(3, np.uint8)
    if case == "range_dst":
        live[1] = 16
    elif case == "range_src":
        src[2] = 99
    elif case == "neg_dst":
        live[0] = -1
    elif case == "dup_dst":
        live[2] = live[0]
    elif case == "src_is_dst":
        src[1] = live[1]
    elif case == "src_is_other_dst":
        src[0] = live[2]
    elif case == "dup_src_ok":
        src[:] = 10
    elif case == "noop_out_of_range_ok":
        live[1], nkv[1] = 77, 17
    rows = W._rows(live, src, nkv, init, 16, np.random.default_rng(0))
    rc_l, _, _, rc_o, _ = _classify_both(w, rows)
    assert rc_l == ERRMAP.get(rc_o, rc_o)
    if case.endswith("_ok"):
        assert rc_l == L.LSC_OK


def test_restore_rejects_before_touching_the_device(lsc):
    """On a host-only pool a valid call fails with LSC_ERR_CUDA (it would have to
    enqueue), an invalid one with its validation error: validation runs first.
    (The valid call is made only where no GPU is visible.)"""
    w = W.get("c0")
    pool = host_pool(w)
    rows = W.restore_rows("c0")
    ops = ops_of(rows)
    if not gpu_present():
        rc, _ = L.lsc_restore(pool, ops, rows.nkv, 16, rows.initialized, FAKE_BASE)
        assert rc == L.LSC_ERR_CUDA
    ops2 = ops.copy()
    ops2["linear_state_id"][3] = ops2["linear_state_id"][0]
    assert L.lsc_restore(pool, ops2, rows.nkv, 16, rows.initialized, FAKE_BASE)[0] == L.LSC_ERR_DUP_DST
    assert L.lsc_restore(pool, ops, rows.nkv, 0, rows.initialized, FAKE_BASE)[0] == L.LSC_ERR_INVALID_ARG
    assert L.lsc_restore(pool, ops, rows.nkv, 16, rows.initialized, None)[0] == L.LSC_ERR_INVALID_ARG
    assert L.lsc_gather(pool, 1, FAKE_BASE, None, 4, FAKE_BASE, FAKE_BASE) == L.LSC_ERR_STATELESS_LAYER
    assert L.lsc_scatter(pool, 5, FAKE_BASE, 4, FAKE_BASE, FAKE_BASE) == L.LSC_ERR_OUT_OF_RANGE
    L.lsc_pool_destroy(pool)


def test_soft_cold_classification_without_gdn_layers(lsc):
    w = W.get("c0")
    w.num_slots = 40
    rows = W.combo_rows(40, 16, seed=1)
    pool = host_pool(w, [W.ATTN, W.ATTN, W.ATTN])
    rc, act, rep = L.lsc_restore_classify(pool, ops_of(rows), rows.nkv, 16, rows.initialized)
    assert rc == L.LSC_OK and rep.soft_cold == 1 and rep.bytes_copied == 0 and rep.n_hit > 0
    assert L.lsc_pool_required_bytes(lib_desc(w, [W.ATTN] * 3)) == 0
    L.lsc_pool_destroy(pool)


def test_alloc_fault_injection_and_layout_log():
    """LSC_FAULT=alloc makes pool creation fail cleanly; LSC_LOG=1 prints one
    [lsc-pool] line per GDN layer with page size, shapes, strides, offsets and
    contiguity (vLLM-Ascend "非连续 KV Cache" §7)."""
    code = (
        "import sys; sys.path.insert(0, %r); sys.path.insert(0, %r)\n"
        "from linear_attention_state_lsc_gb300 import lsc as L, workloads as W\n"
        "from _util import lib_desc\n"
        "rc, p = L.lsc_pool_create(lib_desc(W.get('c0p')), 1 << 40, 1 << 30)\n"
        "print('RC', rc)\n"
    ) % (ROOT, os.path.join(ROOT, "tests"))
    env = dict(os.environ, LSC_FAULT="alloc")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True)
    assert "RC %d" % L.LSC_ERR_NO_MEMORY in r.stdout, r.stderr
    env = dict(os.environ, LSC_LOG="1")
    env.pop("LSC_FAULT", None)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True)
    assert "RC 0" in r.stdout, r.stderr
    lines = [l for l in r.stderr.splitlines() if l.startswith("[lsc-pool]")]
    assert len(lines) == 2
    assert "page_bytes=3072" in lines[0] and "conv shape=[16,64,3] stride=[768,3,1]" in lines[0]
    assert "ssm shape=[16,2,16,16] stride=[768,256,16,1]" in lines[0] and "padding=256" in lines[0]
    assert "contiguous=0" in lines[0] and "layer=2 gdn=1" in lines[1]


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "lsc.h"
#include "lsc_kv.h"
#include "lsc_prefix_cache.h"
#include "lsc_store.h"

int main(void) {
  /* the worked example of a padded page: a [16, 3] bf16 conv view (96 B) and a
     [1, 2, 2] f32 ssm view (16 B) in a 128 B page: one GDN layer, 4 slots */
  int32_t kinds[2] = {LSC_LAYER_GDN, LSC_LAYER_ATTENTION};
  lsc_pool_desc d;
  size_t n = 0;
  lsc_prefix_cache *pc = NULL;
  int32_t slot = -1;
  memset(&d, 0, sizeof d);
  d.num_layers = 2;
  d.layer_kinds = kinds;
  d.num_slots = 4;
  d.conv_dim = 16;
  d.conv_width = 4;
  d.conv_dtype = LSC_BF16;
  d.num_v_heads = 1;
  d.head_v_dim = 2;
  d.head_k_dim = 2;
  d.ssm_dtype = LSC_F32;
  d.page_bytes = 128;
  if (lsc_pool_required_bytes(&d, &n) != LSC_OK) return 1;
  if (strcmp(lsc_error_string(LSC_ERR_ORDER), lsc_error_string(LSC_OK)) == 0) return 2;
  if (lsc_pc_create(8, 16, &pc) != LSC_OK) return 3;
  if (lsc_pc_allocate_live_slot(pc, 42, &slot) != LSC_OK || slot != 0) return 4;
  if (lsc_pc_destroy(pc) != LSC_OK) return 5;
  printf("%zu\n", n);
  return 0;
}
"""


def test_headers_compile_as_c_and_link(tmp_path):
    """The four public headers are plain C99 (compiled with -pedantic, no
    warnings), and a C program links against liblsc.so and calls host-only
    entry points of each area."""
    L.load()
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    lib_dir = os.path.dirname(L.LIB_PATH)
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                         os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", lib_dir, "-llsc",
                         "-Wl,-rpath," + lib_dir], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stderr)
    # 1 GDN layer x 4 slots x 128 B, as the library reports it through Python too
    desc = L.make_pool_desc([L.LSC_LAYER_GDN, L.LSC_LAYER_ATTENTION], 4, 16, 4, L.LSC_BF16, 1, 2, 2, L.LSC_F32, 128)
    assert int(run.stdout) == L.lsc_pool_required_bytes(desc)


def test_algorithmic_bytes_of_the_bench(lsc):
    """The byte counts bench.py divides by (roofline 'achieved') against the
    per-unit figures derived from the workload shapes: c1 restore = 2 payloads
    per (hit row, GDN layer) = 2 x 2 146 304 B; a decode row = state read and
    written + x + alpha, beta + out + idx + has_init, plus the conv weights once
    per launch (c2: 2 228 485 B per row, 65 536 B of weights)."""
    sys.path.insert(0, ROOT)
    import bench
    views = {}
    for name in ("c1", "c2"):
        w = W.get(name)
        rc, pool = L.lsc_pool_create(lib_desc(w), FAKE_BASE, 1 << 44)
        assert rc == L.LSC_OK
        views[name] = (w, L.lsc_pool_layer_view(pool, w.gdn_layers[0])[1])
        L.lsc_pool_destroy(pool)
    w1, v1 = views["c1"]
    assert bench.restore_bytes(v1, 64, 36, 64) == 64 * 36 * 4_292_608 + 64          # 9.890 GB per serving-step restore
    assert bench.decode_bytes(v1, w1, 64) == 64 * 4_325_637 + 65_536               # 276.9 MB per serving-step decode
    w2, v2 = views["c2"]
    assert bench.decode_bytes(v2, w2, 256) == 256 * 2_228_485 + 65_536              # 570.56 MB per c2 decode launch


def test_binding_structs_and_constants_match_the_headers(tmp_path):
    """Every ctypes structure of the binding has the size and field offsets of
    the C struct of the same name, and every LSC_ constant the binding defines
    has the value of the header's macro, as a C compiler sees them."""
    structs = [getattr(L, n) for n in dir(L)
               if isinstance(getattr(L, n), type) and issubclass(getattr(L, n), ctypes.Structure)]
    assert len(structs) >= 12
    consts = {n: getattr(L, n) for n in dir(L) if n.startswith("LSC_") and isinstance(getattr(L, n), int)}
    lines = []
    for s in structs:
        lines.append(f'  printf("%s %zu\\n", "{s.__name__}", sizeof({s.__name__}));')
        for f in s._fields_:
            lines.append(f'  printf("%s %zu\\n", "{s.__name__}.{f[0]}", offsetof({s.__name__}, {f[0]}));')
    for n in consts:
        lines.append(f'  printf("%s %lld\\n", "{n}", (long long)({n}));')
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"lsc.h\"\n#include \"lsc_kv.h\"\n"
                   "#include \"lsc_prefix_cache.h\"\n#include \"lsc_store.h\"\nint main(void) {\n"
                   + "\n".join(lines) + "\n  return 0;\n}\n")
    exe = tmp_path / "layout"
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                         "-o", str(exe)], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    got = dict(l.rsplit(" ", 1) for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                         check=True).stdout.splitlines())
    for s in structs:
        assert int(got[s.__name__]) == ctypes.sizeof(s), s.__name__
        for f in s._fields_:
            assert int(got[f"{s.__name__}.{f[0]}"]) == getattr(s, f[0]).offset, (s.__name__, f[0])
    for n, v in consts.items():
        assert int(got[n]) == v, n


def test_recurrent_workspace_query_host_only():
    """The chunked order's scratch is one record of (2 * 64 * 64 + 64 + 64 + 16)
    floats per (chunk slot, v head), with (T + 63) / 64 + n_seq chunk slots
    (sequence i's chunks start at slot floor(cu_i / 64) + i); the token order,
    and AUTO below head_k_dim 128, need none.  The query needs no GPU."""
    L.load()
    rec = (2 * 64 * 64 + 64 + 64 + 16) * 4
    assert rec == 33344
    for name, dk, n_seq, T in (("c4", 128, 64, 60840), ("c4", 128, 1, 1), ("c4", 128, 3, 0), ("s1", 32, 5, 300)):
        w = W.get(name) if name.startswith("c") else W.small(name)
        pool = host_pool(w)
        try:
            for algo in (L.LSC_RECURRENT_AUTO, L.LSC_RECURRENT_TOKEN, L.LSC_RECURRENT_CHUNKED):
                args = L.recurrent_args(n_seq, w.num_k_heads, T, None, None, None, None, None, None, None, None,
                                        None, algorithm=algo)
                rc, n = L.lsc_gdn_recurrent_workspace_bytes(pool, args)
                assert rc == L.LSC_OK
                chunked = algo == L.LSC_RECURRENT_CHUNKED or (algo == L.LSC_RECURRENT_AUTO and dk == 128)
                slots = (T + 63) // 64 + n_seq
                assert n == (slots * w.num_v_heads * rec if chunked else 0), (name, algo, n)
            bad = L.recurrent_args(-1, w.num_k_heads, T, None, None, None, None, None, None, None, None, None)
            assert L.lsc_gdn_recurrent_workspace_bytes(pool, bad)[0] == L.LSC_ERR_INVALID_ARG
        finally:
            L.lsc_pool_destroy(pool)


def test_decode_flags_validated_before_any_device_work():
    """lsc_gdn_decode refuses flag bits it does not define with INVALID_ARG,
    checked on the host before the device is touched (the stand-in pointers
    are never dereferenced)."""
    L.load()
    w = W.get("c0")
    pool = host_pool(w)
    try:
        l = w.gdn_layers[0]
        for bad in (2, 0x80000000, L.LSC_DECODE_EARLY_STATE | 8):
            args = L.decode_args(2, 1, 256, 256, 256, 256, 256, 256, 256, bad)
            assert L.lsc_gdn_decode(pool, l, args) == L.LSC_ERR_INVALID_ARG
    finally:
        L.lsc_pool_destroy(pool)
