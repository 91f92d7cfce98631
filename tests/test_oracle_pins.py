"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- a value a page prints (tests/golden/), a hand-derived truth table,
an invariant, a closed form, or a brute force written in another formulation
(np.convolve, a tanh form of SiLU, the delta rule as a dense matrix product).

Every test here runs on the CPU only.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_lsc_gb300 import workloads as W

from _util import (golden_kv, host_regions, oracle_layout, oracle_pool, payload_mask,
                   read_golden, views)


# ---------------------------------------------------------------- layout

def test_block_stride_worked_example():
    """vLLM-Ascend "非连续 KV Cache" §3.4: 48 fp16 elements (96 B) in a 128 B page
    advance by 64 elements, leaving a 16-element gap outside the view."""
    g = golden_kv("block_stride_example.txt")
    assert g["logical_elements"] * g["element_bytes"] == g["logical_payload_bytes"]
    # conv view [16, 3] at fp16 = 48 elements; a tiny fp32 ssm view [1, 2, 2] = 16 B
    p = oracle.Pool([oracle.GDN], 4, 16, 4, oracle.F16, 1, 2, 2, oracle.F32, g["page_bytes"])
    rc, L = oracle.layout(p)
    assert rc == oracle.OK
    assert L["conv_elems"] == g["logical_elements"]
    assert L["conv_bytes"] == g["logical_payload_bytes"]
    assert L["conv_stride_elems"] == g["block_stride_elements"]
    assert L["conv_stride_elems"] - L["conv_elems"] == g["gap_elements"]
    assert L["ssm_stride_elems"] == g["page_bytes"] // 4
    assert L["region_bytes"] == 4 * g["page_bytes"]


def test_layout_rejects_bad_pages():
    ok = oracle.Pool([oracle.GDN], 4, 16, 4, oracle.F16, 1, 2, 2, oracle.F32, 128)
    assert oracle.layout(ok)[0] == oracle.OK
    small = oracle.Pool([oracle.GDN], 4, 16, 4, oracle.F16, 1, 2, 2, oracle.F32, 100)
    assert oracle.layout(small)[0] == oracle.REJECT_LAYOUT          # page < payload
    odd = oracle.Pool([oracle.GDN], 4, 16, 4, oracle.F16, 1, 2, 2, oracle.F32, 130)
    assert oracle.layout(odd)[0] == oracle.REJECT_LAYOUT            # 130 % 4 != 0


def test_layout_serving_shapes():
    """Sizes the workload table states in words: conv [8192, 3] bf16 and ssm
    [32, 128, 128] fp32 are 48 KiB and 2 MiB; the 4 KiB-rounded page holds both."""
    L = oracle_layout(W.get("c1"))
    assert L["conv_bytes"] == 48 * 1024 and L["ssm_bytes"] == 2 * 1024 * 1024
    assert L["page"] % 4096 == 0 and L["page"] >= L["payload"] and L["page"] - L["payload"] < 4096
    assert L["num_gdn"] == 36
    L2 = oracle_layout(W.get("c2"))
    assert L2["ssm_bytes"] == 1024 * 1024 and L2["page"] - L2["payload"] == 512
    L0 = oracle_layout(W.get("c0"))
    assert L0["page"] % 256 == 0 and L0["page"] - L0["payload"] < 256


# ---------------------------------------------------------------- restore

def _tiny(slots=40, layers=(W.GDN, W.ATTN, W.GDN), pad=0xA5):
    w = W.get("c0p")
    w.num_slots = slots
    w.layers = list(layers)
    w.pad_byte = pad
    return w


def _snapshot(regions):
    return {l: r.copy() for l, r in regions.items()}


def test_restore_truth_table():
    """All 16 combinations of n_kv x initialized x source against the hand-derived
    table (tests/golden/restore_truth_table.txt)."""
    table = read_golden("restore_truth_table.txt")
    w = _tiny()
    rows = W.combo_rows(w.num_slots, 16, seed=3)
    pool = oracle_pool(w)
    regions = host_regions(w, seed=1)
    by_key = {(int(a), int(b), int(c)): (d, int(e)) for a, b, c, d, e in table}
    rc, act = oracle.classify(pool, rows.live, rows.src, rows.nkv, 16, rows.initialized)
    assert rc == oracle.OK
    hs = rows.hs_prefill.copy()
    assert oracle.restore(pool, regions, rows.live, rows.src, rows.nkv, 16, rows.initialized, hs) == oracle.OK
    names = {oracle.NOOP: "noop", oracle.HIT: "hit", oracle.MISS: "miss"}
    assert len(rows.live) == 16
    for r in range(16):
        key = (int(rows.nkv[r]), int(rows.initialized[r]), int(rows.src[r] >= 0))
        want_action, want_hs = by_key[key]
        assert names[int(act[r])] == want_action, (r, key)
        assert hs[r] == want_hs, (r, key)


def test_restore_c0_rows():
    table = read_golden("c0_restore_rows.txt")
    w = W.get("c0")
    rows = W.restore_rows("c0")
    pool = oracle_pool(w)
    regions = host_regions(w)
    hs = rows.hs_prefill.copy()
    rc, act = oracle.classify(pool, rows.live, rows.src, rows.nkv, rows.block_size, rows.initialized)
    assert rc == oracle.OK
    assert oracle.restore(pool, regions, rows.live, rows.src, rows.nkv, rows.block_size,
                          rows.initialized, hs) == oracle.OK
    names = {oracle.NOOP: "noop", oracle.HIT: "hit", oracle.MISS: "miss"}
    for r, (nkv, init, has_src, action, hs_after) in enumerate(table):
        assert int(rows.nkv[r]) == int(nkv) and int(rows.initialized[r]) == int(init)
        assert int(rows.src[r] >= 0) == int(has_src)
        assert names[int(act[r])] == action
        assert hs[r] == int(hs_after)
    assert rows.src[0] == rows.src[3]  # the duplicate-source row


@pytest.mark.parametrize("name", ["c0", "c0p", "s4"])
def test_restore_copies_payload_and_nothing_else(name):
    """Invariants: each hit's destination views equal the source's pre-image in
    every GDN layer (one history position, Kapitsa 源码拆解 05); every other byte,
    including random padding and the inter-view gap, is unchanged."""
    w = W.get(name) if name.startswith("c") else W.small(name)
    w.num_slots = max(w.num_slots, 24)
    L = oracle_layout(w)
    rows = W.combo_rows(w.num_slots, w.block_size, seed=11)
    pool = oracle_pool(w)
    regions = host_regions(w, seed=2, random_padding=True)
    pre = _snapshot(regions)
    hs = rows.hs_prefill.copy()
    assert oracle.restore(pool, regions, rows.live, rows.src, rows.nkv, w.block_size, rows.initialized, hs) == oracle.OK
    _, act = oracle.classify(pool, rows.live, rows.src, rows.nkv, w.block_size, rows.initialized)
    mask = payload_mask(w, L)
    for l in w.gdn_layers:
        before = pre[l].reshape(w.num_slots, w.page_bytes)
        after = regions[l].reshape(w.num_slots, w.page_bytes)
        expect = before.copy()
        for r in np.nonzero(act == oracle.HIT)[0]:
            expect[rows.live[r], mask] = before[rows.src[r], mask]
        np.testing.assert_array_equal(after, expect)
    assert (act == oracle.HIT).sum() >= 2


def test_restore_soft_fail_without_linear_layers():
    """xLLM notes §4.3: no layer copied -> soft fail to a cold start, no crash."""
    w = _tiny(layers=(W.ATTN, W.ATTN, W.ATTN))
    pool = oracle_pool(w)
    rows = W.combo_rows(w.num_slots, 16, seed=5)
    hs = rows.hs_prefill.copy()
    rc = oracle.restore(pool, {}, rows.live, rows.src, rows.nkv, 16, rows.initialized, hs)
    assert rc == oracle.SOFT_COLD
    _, act = oracle.classify(pool, rows.live, rows.src, rows.nkv, 16, rows.initialized)
    assert (hs[act == oracle.HIT] == 0).all() and (act == oracle.HIT).any()
    assert (hs[act == oracle.MISS] == 0).all()
    np.testing.assert_array_equal(hs[act == oracle.NOOP], rows.hs_prefill[act == oracle.NOOP])


@pytest.mark.parametrize("case", ["range_dst", "range_src", "dup_dst", "src_is_dst", "src_is_other_dst", "block0"])
def test_restore_rejects_and_changes_nothing(case):
    w = _tiny()
    pool = oracle_pool(w)
    regions = host_regions(w, seed=4)
    pre = _snapshot(regions)
    live = np.array([1, 2, 3], np.int32)
    src = np.array([10, 11, 12], np.int32)
    nkv = np.array([16, 16, 16], np.int32)
    init = np.zeros(3, np.uint8)
    bs, want = 16, None
    if case == "range_dst":
        live[1], want = w.num_slots, oracle.REJECT_RANGE
    elif case == "range_src":
        src[2], want = w.num_slots + 5, oracle.REJECT_RANGE
    elif case == "dup_dst":
        live[2], want = live[0], oracle.REJECT_DUP_DST
    elif case == "src_is_dst":
        src[1], want = live[1], oracle.REJECT_SRC_IS_DST
    elif case == "src_is_other_dst":
        src[0], want = live[2], oracle.REJECT_SRC_IS_DST
    elif case == "block0":
        bs, want = 0, oracle.REJECT_ARG
    hs = np.array([7, 7, 7], np.uint8)
    assert oracle.restore(pool, regions, live, src, nkv, bs, init, hs) == want
    assert (hs == 7).all()
    for l in regions:
        np.testing.assert_array_equal(regions[l], pre[l])


def test_restore_ignores_rows_that_copy_nothing():
    """A no-op or miss row with an out-of-range live slot is not an error: only
    rows that copy are checked (the worker addresses slots only to copy)."""
    w = _tiny()
    pool = oracle_pool(w)
    regions = host_regions(w, seed=4)
    live = np.array([-1, w.num_slots + 3], np.int32)
    src = np.array([-1, 5], np.int32)
    nkv = np.array([16, 17], np.int32)  # miss, no-op
    hs = np.array([1, 1], np.uint8)
    assert oracle.restore(pool, regions, live, src, nkv, 16, np.zeros(2, np.uint8), hs) == oracle.OK
    assert list(hs) == [0, 1]


# ---------------------------------------------------------------- gather / scatter

@pytest.mark.parametrize("name", ["c0p", "s4"])
def test_gather_scatter_roundtrip_and_padding(name):
    """vLLM-Ascend §5: gather keeps the index mapping and the has_initial_state mask;
    scatter writes rows back in place and leaves padding as it was."""
    w = W.get(name) if name.startswith("c") else W.small(name)
    L = oracle_layout(w)
    pool = oracle_pool(w)
    regions = host_regions(w, seed=6, random_padding=True)
    l = w.gdn_layers[-1]
    reg = regions[l]
    pre = reg.copy()
    rng = np.random.default_rng(0)
    idx = rng.permutation(w.num_slots)[:7].astype(np.int32)
    idx[3] = -1
    hs = np.array([1, 1, 0, 1, 1, 0, 1], np.uint8)
    rc, conv, ssm = oracle.gather(pool, reg, idx, hs)
    assert rc == oracle.OK
    pages = pre.reshape(w.num_slots, w.page_bytes)
    for i in range(len(idx)):
        if idx[i] >= 0 and hs[i]:
            np.testing.assert_array_equal(conv[i], pages[idx[i], :L["conv_bytes"]])
            np.testing.assert_array_equal(ssm[i], pages[idx[i], L["ssm_offset"]:L["ssm_offset"] + L["ssm_bytes"]])
        else:
            assert not conv[i].any() and not ssm[i].any()
    # all warm, no negative index: scatter(gather(P)) == P byte for byte
    idx2 = np.abs(idx[[0, 1, 2, 4, 5, 6]]).astype(np.int32)
    rc, conv, ssm = oracle.gather(pool, reg, idx2, None)
    assert oracle.scatter(pool, reg, idx2, conv, ssm) == oracle.OK
    np.testing.assert_array_equal(reg, pre)
    # scatter new content: only the selected slots' views change
    conv2 = rng.integers(0, 256, size=conv.shape, dtype=np.uint8)
    ssm2 = rng.integers(0, 256, size=ssm.shape, dtype=np.uint8)
    assert oracle.scatter(pool, reg, idx2, conv2, ssm2) == oracle.OK
    expect = pre.reshape(w.num_slots, w.page_bytes).copy()
    for i, s in enumerate(idx2):
        expect[s, :L["conv_bytes"]] = conv2[i]
        expect[s, L["ssm_offset"]:L["ssm_offset"] + L["ssm_bytes"]] = ssm2[i]
    np.testing.assert_array_equal(reg.reshape(w.num_slots, w.page_bytes), expect)


def test_gather_scatter_reject():
    w = W.get("c0")
    pool = oracle_pool(w)
    reg = host_regions(w)[0]
    pre = reg.copy()
    assert oracle.gather(pool, reg, np.array([0, 16], np.int32))[0] == oracle.REJECT_RANGE
    _, L = oracle.layout(pool)
    conv = np.zeros((2, L["conv_bytes"]), np.uint8)
    ssm = np.zeros((2, L["ssm_bytes"]), np.uint8)
    assert oracle.scatter(pool, reg, np.array([3, 3], np.int32), conv, ssm) == oracle.REJECT_DUP_DST
    assert oracle.scatter(pool, reg, np.array([3, 99], np.int32), conv, ssm) == oracle.REJECT_RANGE
    np.testing.assert_array_equal(reg, pre)


# ---------------------------------------------------------------- decode math

def np_silu(z):
    # z * sigmoid(z) written through tanh: sigmoid(z) = (1 + tanh(z / 2)) / 2
    return 0.5 * z * (1.0 + np.tanh(0.5 * z))


def np_conv(state, x, wt):
    """Depthwise causal conv over the window [state, x] via np.convolve."""
    seq = np.concatenate([state, x[:, None]], axis=1)
    y = np.array([np.convolve(seq[c], wt[c][::-1], mode="valid")[0] for c in range(seq.shape[0])])
    return y, seq[:, 1:]


def np_unit(x):
    return x / np.sqrt(np.linalg.norm(x) ** 2 + 1e-6)


def np_delta(S, q, k, v, a, b):
    """S' = a S (I - b k k^T) + b v k^T as a dense matrix product; o = S' q."""
    dk = len(k)
    S2 = S @ (a * (np.eye(dk) - b * np.outer(k, k))) + b * np.outer(v, k)
    return S2, S2 @ q


def _decode_setup(w, seed=0, n=4, cold=(1,)):
    L = oracle_layout(w)
    pool = oracle_pool(w)
    regions = host_regions(w, seed=seed)
    l = w.gdn_layers[0]
    rng = np.random.default_rng(seed + 100)
    idx = rng.permutation(w.num_slots)[:n].astype(np.int32)
    hs = np.ones(n, np.uint8)
    for c in cold:
        hs[c] = 0
    x, cw, alpha, beta = W.decode_inputs(w, n, seed=seed, layer=l)
    xr = W.to_dtype_bytes(x, w.conv_dtype)
    cwr = W.to_dtype_bytes(cw, w.conv_dtype)
    return L, pool, regions[l], idx, hs, xr, cwr, alpha, beta


def _states(w, L, reg, slot):
    page = reg.reshape(w.num_slots, w.page_bytes)[slot]
    conv = W.from_dtype_bytes(page[:L["conv_bytes"]], w.conv_dtype).astype(np.float64)
    ssm = W.from_dtype_bytes(page[L["ssm_offset"]:L["ssm_offset"] + L["ssm_bytes"]], w.ssm_dtype).astype(np.float64)
    return conv.reshape(w.conv_dim, w.conv_width - 1), ssm.reshape(w.num_v_heads, w.head_v_dim, w.head_k_dim)


def _brute_decode(w, conv_state, ssm, x, cw, a, b, warm):
    Hk, Hv, dk, dv = w.num_k_heads, w.num_v_heads, w.head_k_dim, w.head_v_dim
    if not warm:
        conv_state = np.zeros_like(conv_state)
        ssm = np.zeros_like(ssm)
    z, new_conv = np_conv(conv_state, x, cw)
    y = np_silu(z)
    q = y[:Hk * dk].reshape(Hk, dk)
    k = y[Hk * dk:2 * Hk * dk].reshape(Hk, dk)
    v = y[2 * Hk * dk:].reshape(Hv, dv)
    new_ssm = np.empty_like(ssm)
    o = np.empty((Hv, dv))
    for h in range(Hv):
        g = h // (Hv // Hk)
        new_ssm[h], o[h] = np_delta(ssm[h], np_unit(q[g]), np_unit(k[g]), v[h], a[h], b[h])
    return new_conv, new_ssm, o


@pytest.mark.parametrize("name", ["c0", "s4", "s1"])
def test_decode_brute_force(name):
    """Oracle decode vs. a brute force in another formulation (np.convolve, tanh
    SiLU, dense-matrix delta rule); warm and cold rows; bytes outside the touched
    rows' views unchanged."""
    w = W.get(name) if name.startswith("c") else W.small(name)
    L, pool, reg, idx, hs, xr, cwr, alpha, beta = _decode_setup(w, seed=1)
    pre = reg.copy()
    rc, out = oracle.gdn_decode(pool, reg, idx, hs, xr, cwr, w.num_k_heads, alpha, beta)
    assert rc == oracle.OK
    x = W.from_dtype_bytes(xr, w.conv_dtype).reshape(len(idx), w.conv_dim).astype(np.float64)
    cw = W.from_dtype_bytes(cwr, w.conv_dtype).reshape(w.conv_dim, w.conv_width).astype(np.float64)
    for i, s in enumerate(idx):
        c0, s0 = _states(w, L, pre, s)
        nc, ns, o = _brute_decode(w, c0, s0, x[i], cw, alpha[i].astype(np.float64), beta[i].astype(np.float64), hs[i])
        c1, s1 = _states(w, L, reg, s)
        np.testing.assert_array_equal(c1, nc)   # the shift is exact at any dtype
        if w.ssm_dtype == W.F32:
            np.testing.assert_allclose(s1, ns, rtol=1e-6, atol=1e-7)
        else:  # one bf16 step of rounding
            np.testing.assert_allclose(s1, ns, rtol=2 ** -7, atol=1e-30)
        np.testing.assert_allclose(out[i], o, rtol=1e-5, atol=1e-6)
    touched = np.zeros((w.num_slots, w.page_bytes), bool)
    touched[idx] = payload_mask(w, L)
    np.testing.assert_array_equal(reg.reshape(w.num_slots, -1)[~touched], pre.reshape(w.num_slots, -1)[~touched])


def _decode_with(w, alpha_val, beta_val, seed=2):
    L, pool, reg, idx, hs, xr, cwr, alpha, beta = _decode_setup(w, seed=seed, cold=())
    alpha = np.full_like(alpha, alpha_val)
    beta = np.full_like(beta, beta_val)
    pre = reg.copy()
    rc, out = oracle.gdn_decode(pool, reg, idx, hs, xr, cwr, w.num_k_heads, alpha, beta)
    assert rc == oracle.OK
    x = W.from_dtype_bytes(xr, w.conv_dtype).reshape(len(idx), w.conv_dim).astype(np.float64)
    cw = W.from_dtype_bytes(cwr, w.conv_dtype).reshape(w.conv_dim, w.conv_width).astype(np.float64)
    res = []
    for i, s in enumerate(idx):
        c0, s0 = _states(w, L, pre, s)
        _, s1 = _states(w, L, reg, s)
        y = np_silu(np_conv(c0, x[i], cw)[0])
        Hk, dk, dv = w.num_k_heads, w.head_k_dim, w.head_v_dim
        q = np.stack([np_unit(v) for v in y[:Hk * dk].reshape(Hk, dk)])
        k = np.stack([np_unit(v) for v in y[Hk * dk:2 * Hk * dk].reshape(Hk, dk)])
        v = y[2 * Hk * dk:].reshape(w.num_v_heads, dv)
        res.append((s0, s1, q, k, v, out[i]))
    return res


@pytest.mark.parametrize("name", ["c0", "s4"])
def test_decode_beta0_alpha1_leaves_state_bit_exact(name):
    """Closed form from the benchmark spec: beta = 0, alpha = 1 leaves S unchanged
    bit for bit, and o = S q (a textbook matvec)."""
    w = W.get(name) if name.startswith("c") else W.small(name)
    G = w.num_v_heads // w.num_k_heads
    for s0, s1, q, k, v, o in _decode_with(w, 1.0, 0.0):
        np.testing.assert_array_equal(s1, s0)
        for h in range(w.num_v_heads):
            np.testing.assert_allclose(o[h], s0[h] @ q[h // G], rtol=1e-5, atol=1e-6)


def test_decode_beta0_scales_state():
    w = W.get("c0")
    for s0, s1, q, k, v, o in _decode_with(w, 0.625, 0.0):
        np.testing.assert_array_equal(s1, (0.625 * s0).astype(np.float32))


def test_decode_alpha0_is_rank_one():
    w = W.get("c0")
    G = w.num_v_heads // w.num_k_heads
    for s0, s1, q, k, v, o in _decode_with(w, 0.0, 0.75):
        for h in range(w.num_v_heads):
            np.testing.assert_allclose(s1[h], 0.75 * np.outer(v[h], k[h // G]), rtol=1e-6, atol=1e-7)
            assert np.linalg.matrix_rank(s1[h], tol=1e-5) == 1


def test_decode_delta_rule_fixed_point():
    """alpha = beta = 1: S' k = v + (1 - |k|^2)(S k - v); with |k| = 1 up to the
    epsilon, the updated state maps k onto v (the delta rule's correction)."""
    w = W.get("c0")
    G = w.num_v_heads // w.num_k_heads
    for s0, s1, q, k, v, o in _decode_with(w, 1.0, 1.0):
        for h in range(w.num_v_heads):
            kh = k[h // G]
            rho = kh @ kh
            np.testing.assert_allclose(s1[h] @ kh, v[h] + (1 - rho) * (s0[h] @ kh - v[h]), rtol=1e-5, atol=1e-5)
            assert abs(1 - rho) < 1e-4


def test_conv_weight_orientation_and_channel_split():
    """With the weight on the newest tap only and a cold state, y = SiLU(x): the
    outputs then follow from x alone, which pins the [q | k | v] split, the head
    sharing and the tap order.  With the weight on the oldest tap, y = SiLU(oldest
    state)."""
    w = W.get("c0")
    L, pool, reg, idx, hs, xr, cwr, alpha, beta = _decode_setup(w, seed=3, cold=(0, 1, 2, 3))
    cw = np.zeros((w.conv_dim, w.conv_width), np.float32)
    cw[:, -1] = 1.0
    alpha[:] = 0.0
    beta[:] = 1.0
    rc, out = oracle.gdn_decode(pool, reg, idx, hs, xr, W.to_dtype_bytes(cw, w.conv_dtype),
                                w.num_k_heads, alpha, beta)
    assert rc == oracle.OK
    x = W.from_dtype_bytes(xr, w.conv_dtype).reshape(len(idx), w.conv_dim).astype(np.float64)
    Hk, dk, dv, Hv = w.num_k_heads, w.head_k_dim, w.head_v_dim, w.num_v_heads
    for i in range(len(idx)):
        y = np_silu(x[i])
        q, k, v = np_unit(y[:dk]), np_unit(y[dk:2 * dk]), y[2 * dk:].reshape(Hv, dv)
        np.testing.assert_allclose(out[i], v * (k @ q), rtol=1e-5, atol=1e-6)
    # oldest tap: warm rows, y = SiLU(state[:, 0])
    L, pool, reg, idx, hs, xr, cwr, alpha, beta = _decode_setup(w, seed=4, cold=())
    pre = reg.copy()
    cw = np.zeros((w.conv_dim, w.conv_width), np.float32)
    cw[:, 0] = 1.0
    alpha[:] = 0.0
    beta[:] = 1.0
    rc, out = oracle.gdn_decode(pool, reg, idx, hs, xr, W.to_dtype_bytes(cw, w.conv_dtype),
                                w.num_k_heads, alpha, beta)
    for i, s in enumerate(idx):
        c0, _ = _states(w, L, pre, s)
        y = np_silu(c0[:, 0])
        q, k, v = np_unit(y[:dk]), np_unit(y[dk:2 * dk]), y[2 * dk:].reshape(Hv, dv)
        np.testing.assert_allclose(out[i], v * (k @ q), rtol=1e-5, atol=1e-6)


def test_decode_negative_index_and_reject():
    w = W.get("c0")
    L, pool, reg, idx, hs, xr, cwr, alpha, beta = _decode_setup(w)
    pre = reg.copy()
    idx = np.array([-1, -1, -1, -1], np.int32)
    rc, out = oracle.gdn_decode(pool, reg, idx, hs, xr, cwr, w.num_k_heads, alpha, beta)
    assert rc == oracle.OK and not out.any()
    np.testing.assert_array_equal(reg, pre)
    rc, _ = oracle.gdn_decode(pool, reg, np.array([1, 1, 2, 3], np.int32), hs, xr, cwr, 1, alpha, beta)
    assert rc == oracle.REJECT_DUP_DST
    rc, _ = oracle.gdn_decode(pool, reg, np.array([1, 2, 3, 16], np.int32), hs, xr, cwr, 1, alpha, beta)
    assert rc == oracle.REJECT_RANGE
    np.testing.assert_array_equal(reg, pre)


def test_bf16_rounding_matches_torch():
    """The oracle's bf16 store rounds to nearest even like torch's CPU cast,
    including exact ties and values near the overflow edge."""
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -1 - 2 ** -8, 3.3895314e38, 0.0, -0.0, 1e-40], np.float32),
    ]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_bits(float(v)) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, want)


# ---------------------------------------------------------------- recurrence

def _rec_setup(w, lengths, seed=0, warm=(1, 0, 1)):
    L = oracle_layout(w)
    pool = oracle_pool(w)
    regions = host_regions(w, seed=seed)
    l = w.gdn_layers[0]
    rng = np.random.default_rng(seed + 55)
    idx = rng.permutation(w.num_slots)[:len(lengths)].astype(np.int32)
    hs = np.array([warm[i % len(warm)] for i in range(len(lengths))], np.uint8)
    cu, q, k, v, a, b = W.recurrent_inputs(w, lengths, seed=seed, layer=l)
    return L, pool, regions[l], idx, hs, cu, q, k, v, a, b


@pytest.mark.parametrize("name", ["c0", "s4"])
def test_recurrence_matches_sequential_matrix_form(name):
    """T tokens of the recurrence equal T sequential dense-matrix delta-rule
    steps from the slot state (zero when cold); zero-length sequences leave the
    state alone."""
    w = W.get(name) if name.startswith("c") else W.small(name)
    lengths = [5, 0, 13, 1]
    L, pool, reg, idx, hs, cu, q, k, v, a, b = _rec_setup(w, lengths, seed=2)
    pre = reg.copy()
    rc, out = oracle.gdn_recurrent(pool, reg, idx, hs, cu, w.num_k_heads, q, k, v, a, b)
    assert rc == oracle.OK
    G = w.num_v_heads // w.num_k_heads
    for i, s in enumerate(idx):
        c0, s0 = _states(w, L, pre, s)
        c1, s1 = _states(w, L, reg, s)
        np.testing.assert_array_equal(c1, c0)  # no conv stage
        S = s0.copy() if hs[i] else np.zeros_like(s0)
        for t in range(cu[i], cu[i + 1]):
            for h in range(w.num_v_heads):
                g = h // G
                S[h], o = np_delta(S[h], q[t, g].astype(np.float64), k[t, g].astype(np.float64),
                                   v[t, h].astype(np.float64), float(a[t, h]), float(b[t, h]))
                np.testing.assert_allclose(out[t, h], o, rtol=1e-5, atol=1e-6)
        if cu[i + 1] == cu[i]:
            if hs[i]:
                np.testing.assert_array_equal(s1, s0)
            continue
        tol = dict(rtol=1e-6, atol=1e-7) if w.ssm_dtype == W.F32 else dict(rtol=2 ** -7, atol=1e-30)
        np.testing.assert_allclose(s1, S, **tol)


def test_recurrence_identity_gate():
    """alpha = 1, beta = 0 at every token: S unchanged bit for bit, o_t = S q_t."""
    w = W.get("c0")
    L, pool, reg, idx, hs, cu, q, k, v, a, b = _rec_setup(w, [7, 3], seed=3, warm=(1,))
    a[:] = 1.0
    b[:] = 0.0
    pre = reg.copy()
    rc, out = oracle.gdn_recurrent(pool, reg, idx, hs, cu, w.num_k_heads, q, k, v, a, b)
    assert rc == oracle.OK
    np.testing.assert_array_equal(reg, pre)
    for i, s in enumerate(idx):
        _, s0 = _states(w, L, pre, s)
        for t in range(cu[i], cu[i + 1]):
            for h in range(w.num_v_heads):
                np.testing.assert_allclose(out[t, h], s0[h] @ q[t, 0], rtol=1e-5, atol=1e-6)


def test_recurrence_negative_index():
    w = W.get("c0")
    L, pool, reg, idx, hs, cu, q, k, v, a, b = _rec_setup(w, [4, 6], seed=4)
    idx[1] = -1
    pre = reg.copy()
    rc, out = oracle.gdn_recurrent(pool, reg, idx, hs, cu, w.num_k_heads, q, k, v, a, b)
    assert rc == oracle.OK
    assert not out[cu[1]:cu[2]].any()
    page = pre.reshape(w.num_slots, -1)
    after = reg.reshape(w.num_slots, -1)
    others = [s for s in range(w.num_slots) if s != idx[0]]
    np.testing.assert_array_equal(after[others], page[others])
