"""Pins for the oracle's prefill conv (causal_conv1d over a sequence from the
slot's conv state, then the q | k | v split and the per-head L2 norm of q, k):
a brute force in another formulation (np.convolve over [state, x], SiLU through
tanh), cold and padding rows, sequences shorter than the conv window, the
equivalence of one call and two calls that carry the state through the slot,
and a one-token prefill against the decode's conv state update.

Sources: vLLM-Ascend "非连续 KV Cache" §6 (causal_conv1d_fn beside
causal_conv1d_update); Kapitsa "相同前缀不一定能全部复用" (the prefill continues
from the restored state).  CPU only.
"""
import numpy as np
import pytest

import oracle
from linear_attention_state_lsc_gb300 import workloads as W

from _util import host_regions, oracle_layout, oracle_pool


def np_silu(z):
    return 0.5 * z * (1.0 + np.tanh(0.5 * z))


def np_unit_rows(a):
    return a / np.sqrt((a * a).sum(axis=-1, keepdims=True) + 1e-6)


def conv_state(w, L, reg, slot):
    page = reg.reshape(w.num_slots, w.page_bytes)[slot]
    raw = page[:L["conv_bytes"]]
    return W.from_dtype_bytes(raw, w.conv_dtype).astype(np.float64).reshape(w.conv_dim, w.conv_width - 1)


def brute(w, state, x, cw):
    """[T, C] outputs and the final state for one sequence, via np.convolve."""
    seq = np.concatenate([state, x.T], axis=1)                 # [C, W-1+T]
    z = np.stack([np.convolve(seq[c], cw[c][::-1], mode="valid") for c in range(w.conv_dim)], axis=1)
    y = np_silu(z)                                             # [T, C]
    Hk, dk = w.num_k_heads, w.head_k_dim
    T = x.shape[0]
    q = np_unit_rows(y[:, :Hk * dk].reshape(T, Hk, dk))
    k = np_unit_rows(y[:, Hk * dk:2 * Hk * dk].reshape(T, Hk, dk))
    v = y[:, 2 * Hk * dk:].reshape(T, w.num_v_heads, w.head_v_dim)
    return q, k, v, seq[:, -(w.conv_width - 1):]


def setup(w, lengths, seed=0, layer=None):
    layer = w.gdn_layers[0] if layer is None else layer
    cu, x, cw = W.prefill_inputs(w, lengths, seed=seed, layer=layer)
    xr = W.to_dtype_bytes(x, w.conv_dtype).reshape(len(x), -1)
    cwr = W.to_dtype_bytes(cw, w.conv_dtype)
    x = W.from_dtype_bytes(xr.reshape(-1), w.conv_dtype).reshape(x.shape).astype(np.float64)
    cw = W.from_dtype_bytes(cwr, w.conv_dtype).reshape(cw.shape).astype(np.float64)
    return cu, xr, cwr, x, cw


@pytest.mark.parametrize("name", ["c0", "s1", "s4"])
def test_prefill_conv_brute_force(name):
    w = W.get(name) if name.startswith("c") else W.small(name)
    L = oracle_layout(w)
    pool = oracle_pool(w)
    reg = host_regions(w, seed=2)[w.gdn_layers[0]]
    pre = reg.copy()
    lengths = [5, 1, 2, 9]                     # includes sequences shorter than W - 1
    cu, xr, cwr, x, cw = setup(w, lengths, seed=3)
    rng = np.random.default_rng(4)
    idx = rng.permutation(w.num_slots)[:len(lengths)].astype(np.int32)
    hs = np.array([1, 1, 0, 1], np.uint8)
    rc, q, k, v = oracle.gdn_prefill_conv(pool, reg, idx, hs, cu, w.num_k_heads, xr, cwr)
    assert rc == oracle.OK
    for i, s in enumerate(idx):
        t0, t1 = cu[i], cu[i + 1]
        st = conv_state(w, L, pre, s) if hs[i] else np.zeros((w.conv_dim, w.conv_width - 1))
        bq, bk, bv, bst = brute(w, st, x[t0:t1], cw)
        np.testing.assert_allclose(q[t0:t1], bq, rtol=1e-6, atol=1e-7)
        np.testing.assert_allclose(k[t0:t1], bk, rtol=1e-6, atol=1e-7)
        np.testing.assert_allclose(v[t0:t1], bv, rtol=1e-6, atol=1e-7)
        np.testing.assert_array_equal(conv_state(w, L, reg, s), bst)   # inputs moved, not recomputed
    # nothing but the rows' conv views changed
    touched = np.zeros((w.num_slots, w.page_bytes), bool)
    touched[idx, :L["conv_bytes"]] = True
    np.testing.assert_array_equal(reg.reshape(w.num_slots, -1)[~touched], pre.reshape(w.num_slots, -1)[~touched])


def test_prefill_conv_padding_row_and_errors():
    w = W.small("s1")
    pool = oracle_pool(w)
    reg = host_regions(w, seed=1)[w.gdn_layers[0]]
    pre = reg.copy()
    cu, xr, cwr, x, cw = setup(w, [3, 4])
    rc, q, k, v = oracle.gdn_prefill_conv(pool, reg, np.array([-1, 2], np.int32), None, cu, w.num_k_heads, xr, cwr)
    assert rc == oracle.OK
    assert not q[:3].any() and not k[:3].any() and not v[:3].any()
    page = w.page_bytes
    np.testing.assert_array_equal(reg[:2 * page], pre[:2 * page])
    bad = reg.copy()
    assert oracle.gdn_prefill_conv(pool, bad, np.array([2, 2], np.int32), None, cu, w.num_k_heads, xr, cwr)[0] \
        == oracle.REJECT_DUP_DST
    assert oracle.gdn_prefill_conv(pool, bad, np.array([2, w.num_slots], np.int32), None, cu, w.num_k_heads, xr,
                                   cwr)[0] == oracle.REJECT_RANGE
    np.testing.assert_array_equal(bad, reg)


@pytest.mark.parametrize("split", [1, 2, 5])
def test_prefill_conv_split_carries_state(split):
    """Tokens [0, T) in one call equal [0, split) then [split, T) in two calls:
    the conv state written back after the first call is exactly what the second
    call's first tokens need."""
    w = W.small("s1")
    pool = oracle_pool(w)
    reg1 = host_regions(w, seed=5)[w.gdn_layers[0]]
    reg2 = reg1.copy()
    T = 9
    cu, xr, cwr, x, cw = setup(w, [T], seed=6)
    idx = np.array([3], np.int32)
    _, q, k, v = oracle.gdn_prefill_conv(pool, reg1, idx, None, cu, w.num_k_heads, xr, cwr)
    _, qa, ka, va = oracle.gdn_prefill_conv(pool, reg2, idx, None, np.array([0, split], np.int32), w.num_k_heads,
                                            xr[:split], cwr)
    _, qb, kb, vb = oracle.gdn_prefill_conv(pool, reg2, idx, None, np.array([0, T - split], np.int32),
                                            w.num_k_heads, xr[split:], cwr)
    np.testing.assert_array_equal(np.concatenate([qa, qb]), q)
    np.testing.assert_array_equal(np.concatenate([ka, kb]), k)
    np.testing.assert_array_equal(np.concatenate([va, vb]), v)
    np.testing.assert_array_equal(reg2, reg1)


@pytest.mark.parametrize("name", ["c0", "s4"])
def test_one_token_prefill_matches_decode_conv_state(name):
    """A one-token prefill leaves the same conv state as the decode's
    causal_conv1d_update on the same x (two independent code paths)."""
    w = W.get(name) if name.startswith("c") else W.small(name)
    L = oracle_layout(w)
    pool = oracle_pool(w)
    reg1 = host_regions(w, seed=7)[w.gdn_layers[0]]
    reg2 = reg1.copy()
    cu, xr, cwr, x, cw = setup(w, [1, 1], seed=8)
    idx = np.array([1, 4], np.int32)
    hs = np.array([1, 0], np.uint8)
    assert oracle.gdn_prefill_conv(pool, reg1, idx, hs, cu, w.num_k_heads, xr, cwr)[0] == oracle.OK
    a = np.full((2, w.num_v_heads), 0.9, np.float32)
    b = np.full((2, w.num_v_heads), 0.5, np.float32)
    assert oracle.gdn_decode(pool, reg2, idx, hs, xr, cwr, w.num_k_heads, a, b)[0] == oracle.OK
    for s in idx:
        np.testing.assert_array_equal(conv_state(w, L, reg1, s), conv_state(w, L, reg2, s))
