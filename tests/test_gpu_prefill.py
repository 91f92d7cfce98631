"""GPU parity of lsc_gdn_prefill_conv against the oracle: q, k, v within the
fp32 bound, the conv state bit-exact, everything else in the page untouched.
Both paths (the fused 8-channel path and the two-pass path) on several shapes,
sequence lengths around the conv window and the token tile, cold and padding
rows, inconsistent cu_seqlens, and the c4 shapes at full size on sampled
sequences.

Sources: vLLM-Ascend "非连续 KV Cache" §6 (causal_conv1d_fn); Kapitsa
"相同前缀不一定能全部复用".
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_lsc_gb300 import lsc as L
from linear_attention_state_lsc_gb300 import workloads as W

from _gpu import DevPool, dev, tol
from _util import oracle_layout, oracle_pool

pytestmark = pytest.mark.gpu


def shape(name, **kw):
    w = W.get(name) if name.startswith("c") else W.small(name)
    w = dataclasses.replace(w, layers=list(w.layers), extra=dict(w.extra))
    for k, v in kw.items():
        setattr(w, k, v)
    return w


def inputs(w, lengths, seed, pad=True):
    rng = np.random.default_rng(seed)
    idx = rng.permutation(w.num_slots)[:len(lengths)].astype(np.int32)
    if pad:
        idx[-1] = -1
    has = (rng.random(len(lengths)) < 0.6).astype(np.uint8)
    cu, x, cw = W.prefill_inputs(w, lengths, seed=seed, layer=0)
    xr = W.to_dtype_bytes(x, w.conv_dtype).reshape(len(x), -1)
    cwr = W.to_dtype_bytes(cw, w.conv_dtype).reshape(w.conv_dim, -1)
    return idx, has, cu, xr, cwr


def run(P, l, w, idx, has, cu, xr, cwr, x_offset=0):
    T = int(cu[-1])
    Hk, dk = w.num_k_heads, w.head_k_dim
    q = torch.full((max(T, 1), Hk, dk), float("nan"), device="cuda")
    k = torch.full_like(q, float("nan"))
    v = torch.full((max(T, 1), w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
    xbuf = torch.zeros(xr.size + x_offset, dtype=torch.uint8, device="cuda")
    xbuf[x_offset:] = dev(xr.reshape(-1))
    xd = xbuf[x_offset:]
    t = [dev(z) for z in (idx, has, cu)]
    args = L.prefill_conv_args(len(idx), Hk, T, *t, xd, dev(cwr.reshape(-1)), q, k, v)
    rc = L.lsc_gdn_prefill_conv(P.pool, l, args, torch.cuda.current_stream())
    torch.cuda.synchronize()
    return rc, q.cpu().numpy()[:T], k.cpu().numpy()[:T], v.cpu().numpy()[:T]


def check(w, P, l, pre, idx, has, cu, xr, cwr, q, k, v):
    reg = pre.copy()
    rc, qo, ko, vo = oracle.gdn_prefill_conv(oracle_pool(w), reg, idx, has, cu, w.num_k_heads, xr, cwr)
    assert rc == oracle.OK
    t = tol(W.F32)
    np.testing.assert_allclose(q, qo, **t)
    np.testing.assert_allclose(k, ko, **t)
    np.testing.assert_allclose(v, vo, **t)
    np.testing.assert_array_equal(P.download(l), reg)   # conv state bit-exact, the rest untouched


CASES = [("c0", {}), ("s1", {}), ("s2", {}), ("s3", {}), ("s4", {}),
         ("c1", {"num_slots": 6, "layers": [W.GDN]})]


@pytest.mark.parametrize("name,kw", CASES, ids=[n for n, _ in CASES])
@pytest.mark.parametrize("x_offset", [0, 1], ids=["aligned", "x-off-16B"])
def test_prefill_conv_matches_oracle(lsc, name, kw, x_offset):
    """x_offset 1: x starts one element past a 16-byte boundary (the two-pass path)."""
    w = shape(name, **kw)
    x_offset *= W.ESIZE[w.conv_dtype]
    lengths = [0, 1, 2, 3, 64, 65, 130, 7][:w.num_slots]
    with DevPool(w, seed=21, random_padding=True) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, xr, cwr = inputs(w, lengths, seed=4)
        rc, q, k, v = run(P, l, w, idx, has, cu, xr, cwr, x_offset)
        assert rc == L.LSC_OK, L.lsc_error_string(rc)
        check(w, P, l, pre, idx, has, cu, xr, cwr, q, k, v)
        assert P.status() == L.LSC_OK


def with_width(name, width):
    """A shape with another conv width; the page grows to hold the wider conv state."""
    w = shape(name)
    w.conv_width = width
    conv_bytes = w.conv_dim * (width - 1) * W.ESIZE[w.conv_dtype]
    ssm_bytes = w.num_v_heads * w.head_v_dim * w.head_k_dim * W.ESIZE[w.ssm_dtype]
    w.page_bytes = (conv_bytes + 15) // 16 * 16 + ssm_bytes + 256
    return w


@pytest.mark.parametrize("name", ["c0", "s3"], ids=["f32-conv", "bf16-conv"])
@pytest.mark.parametrize("width", [2, 3, 5, 8])
@pytest.mark.parametrize("x_offset", [0, 1], ids=["aligned", "x-off-16B"])
def test_prefill_conv_other_widths(lsc, name, width, x_offset):
    """Conv widths other than 4: the run-time-width fast path (aligned x) and
    the two-pass path (x one element off a 16-byte boundary)."""
    w = with_width(name, width)
    x_offset *= W.ESIZE[w.conv_dtype]
    lengths = [0, 1, width - 1, width, 70, 9][:w.num_slots]
    with DevPool(w, seed=22, random_padding=True) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, xr, cwr = inputs(w, lengths, seed=5)
        rc, q, k, v = run(P, l, w, idx, has, cu, xr, cwr, x_offset)
        assert rc == L.LSC_OK, L.lsc_error_string(rc)
        check(w, P, l, pre, idx, has, cu, xr, cwr, q, k, v)
        assert P.status() == L.LSC_OK


@pytest.mark.parametrize("x_offset", [0, 1], ids=["aligned", "x-off-16B"])
def test_prefill_null_has_init_means_all_warm(lsc, x_offset):
    """has_init = NULL: every sequence's window starts from its slot's conv state."""
    w = shape("s3")
    x_offset *= W.ESIZE[w.conv_dtype]
    lengths = [1, 2, 70, 5]
    with DevPool(w, seed=23, random_padding=True) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, xr, cwr = inputs(w, lengths, seed=6, pad=False)
        T = int(cu[-1])
        q = torch.full((T, w.num_k_heads, w.head_k_dim), float("nan"), device="cuda")
        k = torch.full_like(q, float("nan"))
        v = torch.full((T, w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
        xbuf = torch.zeros(xr.size + x_offset, dtype=torch.uint8, device="cuda")
        xbuf[x_offset:] = dev(xr.reshape(-1))
        args = L.prefill_conv_args(len(idx), w.num_k_heads, T, dev(idx), None, dev(cu), xbuf[x_offset:],
                                   dev(cwr.reshape(-1)), q, k, v)
        assert L.lsc_gdn_prefill_conv(P.pool, l, args, torch.cuda.current_stream()) == L.LSC_OK
        torch.cuda.synchronize()
        has[:] = 1
        check(w, P, l, pre, idx, has, cu, xr, cwr, q.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy())
        assert P.status() == L.LSC_OK


def test_prefill_then_decode_continues(lsc):
    """After a prefill the slot's conv state is the one a decode continues from:
    prefill of T tokens then one decode token equals the oracle doing the same."""
    w = shape("c0")
    with DevPool(w, seed=22) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, xr, cwr = inputs(w, [20, 5], seed=5, pad=False)
        rc, *_ = run(P, l, w, idx, has, cu, xr, cwr)
        assert rc == L.LSC_OK
        reg = pre.copy()
        assert oracle.gdn_prefill_conv(oracle_pool(w), reg, idx, has, cu, w.num_k_heads, xr, cwr)[0] == oracle.OK
        x, _, a, b = W.decode_inputs(w, 2, seed=6, layer=l)
        xd = W.to_dtype_bytes(x, w.conv_dtype)
        out = torch.empty((2, w.num_v_heads, w.head_v_dim), device="cuda")
        hs1 = np.ones(2, np.uint8)
        da = L.decode_args(2, w.num_k_heads, dev(idx), dev(hs1), dev(xd), dev(cwr.reshape(-1)), dev(a), dev(b), out)
        assert L.lsc_gdn_decode(P.pool, l, da, torch.cuda.current_stream()) == L.LSC_OK
        rc, out_o = oracle.gdn_decode(oracle_pool(w), reg, idx, hs1, xd, cwr, w.num_k_heads, a, b)
        assert rc == oracle.OK
        np.testing.assert_allclose(out.cpu().numpy(), out_o, **tol(w.ssm_dtype))


def test_prefill_inconsistent_cu_seqlens(lsc):
    w = shape("s1")
    with DevPool(w, seed=23) as P:
        l = P.gdn_layers[0]
        idx, has, cu, xr, cwr = inputs(w, [4, 6, 5], seed=7, pad=False)
        bad = cu.copy()
        bad[1], bad[2] = 8, 3          # decreasing
        rc, q, k, v = run(P, l, w, idx, has, bad, xr, cwr)
        assert rc == L.LSC_OK
        assert P.status() == L.LSC_ERR_INVALID_ARG
        assert P.status() == L.LSC_OK  # reading the status clears it
        # sequences with consistent bounds still ran
        idx2 = idx.copy()
        rc, q2, k2, v2 = run(P, l, w, idx2, has, cu, xr, cwr)
        assert rc == L.LSC_OK and P.status() == L.LSC_OK


def test_prefill_rejects_misaligned_arrays(lsc):
    """Arrays not aligned to their element size are refused on the host; no
    kernel runs on them."""
    w = shape("c0")   # f32 conv: x needs 4-byte alignment
    with DevPool(w) as P:
        l = P.gdn_layers[0]
        buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
        z = torch.zeros(16, dtype=torch.int32, device="cuda")
        ok = dict(n_seq=1, num_k_heads=w.num_k_heads, total_tokens=1, idx=z, has_init=None, cu_seqlens=z,
                  x=buf, conv_weight=buf, q=buf, k=buf, v=buf)
        for name in ("x", "conv_weight", "q", "v"):
            a = L.prefill_conv_args(**{**ok, name: buf.data_ptr() + 2})
            assert L.lsc_gdn_prefill_conv(P.pool, l, a, None) == L.LSC_ERR_MISALIGNED, name
        a = L.prefill_conv_args(**{**ok, "idx": z.data_ptr() + 1})
        assert L.lsc_gdn_prefill_conv(P.pool, l, a, None) == L.LSC_ERR_MISALIGNED


def test_prefill_argument_errors(lsc):
    w = shape("s1")
    with DevPool(w) as P:
        l = P.gdn_layers[0]
        z = torch.zeros(16, dtype=torch.int32, device="cuda")
        base = dict(n_seq=1, num_k_heads=w.num_k_heads, total_tokens=1, idx=z, has_init=None, cu_seqlens=z,
                    x=z, conv_weight=z, q=z, k=z, v=z)
        for bad in (dict(n_seq=-1), dict(num_k_heads=0), dict(cu_seqlens=None), dict(x=None),
                    dict(n_seq=0, total_tokens=3)):
            a = L.prefill_conv_args(**{**base, **bad})
            assert L.lsc_gdn_prefill_conv(P.pool, l, a, None) == L.LSC_ERR_INVALID_ARG, bad
        attn = [i for i, kind in enumerate(w.layers) if kind == W.ATTN]
        if attn:
            assert L.lsc_gdn_prefill_conv(P.pool, attn[0], L.prefill_conv_args(**base), None) == \
                L.LSC_ERR_STATELESS_LAYER


@pytest.mark.big
def test_prefill_c4_full_size_sampled(lsc):
    """The c4 token mix (64 sequences, 64..2048 tokens, about 61 k in all) on c1's
    pool shapes; the oracle checks three sequences (the first, a long one, the
    last) and every slot's conv state."""
    w = shape("c4", num_slots=72, layers=[W.GDN])
    lengths = W.seq_lengths(64, 64, 2048, seed=0)
    with DevPool(w, seed=24, device_fill=True) as P:
        l = P.gdn_layers[0]
        pre = P.download(l)
        idx, has, cu, xr, cwr = inputs(w, lengths, seed=8, pad=False)
        rc, q, k, v = run(P, l, w, idx, has, cu, xr, cwr)
        assert rc == L.LSC_OK and P.status() == L.LSC_OK
        got = P.download(l)
        Lo = oracle_layout(w)
        t = tol(W.F32)
        for i in (0, int(np.argmax(lengths)), 63):
            reg = pre.copy()
            sub_cu = np.array([0, lengths[i]], np.int32)
            rc, qo, ko, vo = oracle.gdn_prefill_conv(oracle_pool(w), reg, idx[i:i + 1], has[i:i + 1], sub_cu,
                                                     w.num_k_heads, xr[cu[i]:cu[i + 1]], cwr)
            assert rc == oracle.OK
            np.testing.assert_allclose(q[cu[i]:cu[i + 1]], qo, **t)
            np.testing.assert_allclose(k[cu[i]:cu[i + 1]], ko, **t)
            np.testing.assert_allclose(v[cu[i]:cu[i + 1]], vo, **t)
            page = slice(idx[i] * w.page_bytes, (idx[i] + 1) * w.page_bytes)
            np.testing.assert_array_equal(got[page], reg[page])
        # every sequence's new conv state is the last W-1 rows of its x (all longer than W-1)
        assert w.conv_dtype == W.BF16
        xe = xr.view(np.uint16)                                   # [T, C] bf16 bits
        for i in range(64):
            st = got[idx[i] * w.page_bytes: idx[i] * w.page_bytes + Lo["conv_bytes"]].view(np.uint16)
            want = xe[cu[i + 1] - (w.conv_width - 1):cu[i + 1]].T     # [C, W-1], oldest first
            np.testing.assert_array_equal(st.reshape(w.conv_dim, w.conv_width - 1), want)
