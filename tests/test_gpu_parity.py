"""GPU parity: every kernel of liblsc, called through the C ABI, against the CPU
oracle on the same seeded inputs, element by element.  Restore, gather and
scatter must be bit-exact (whole layer regions compared, padding included);
the GDN math must fall within the tolerance of tests/_gpu.tol.  Sizes span
several work units and ragged tails, and the edge cases of each call.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_lsc_gb300 import lsc as L
from linear_attention_state_lsc_gb300 import workloads as W

from _gpu import DevPool, conv_bytes_dev, dev, tol
from _util import oracle_layout, oracle_pool, ops_of, payload_mask

pytestmark = pytest.mark.gpu


def workload(name, **kw):
    w = W.get(name) if name.startswith("c") else W.small(name)
    w = dataclasses.replace(w, layers=list(w.layers), extra=dict(w.extra))
    for k, v in kw.items():
        setattr(w, k, v)
    if "page_bytes" not in kw:
        # keep the workload's padding, growing the page when a shape change needs it
        pad = w.page_bytes - _payload(W.get(name) if name.startswith("c") else W.small(name))
        w.page_bytes = (_payload(w) + pad + 15) // 16 * 16
    return w


def _payload(w):
    w = dataclasses.replace(w, page_bytes=1 << 40)  # any page that holds the payload
    return oracle_layout(w)["payload"]


def event():
    e = torch.cuda.Event()
    e.record(torch.cuda.current_stream())
    torch.cuda.synchronize()
    return e


def run_restore(P, rows, block_size):
    hs = dev(rows.hs_prefill)
    prep = torch.cuda.Stream()
    prep.wait_stream(torch.cuda.current_stream())
    ev = event()
    rc, rep = L.lsc_restore(P.pool, ops_of(rows), rows.nkv, block_size, rows.initialized, hs, prep, ev)
    torch.cuda.current_stream().wait_event(ev)
    torch.cuda.synchronize()
    return rc, rep, hs.cpu().numpy()


def oracle_restore(w, P, pre, rows, block_size, layers=None):
    regions = {l: pre[l].copy() for l in pre}
    hs = rows.hs_prefill.copy()
    rc = oracle.restore(oracle_pool(w, layers), regions, rows.live, rows.src, rows.nkv, block_size,
                        rows.initialized, hs)
    return rc, regions, hs


# ---------------------------------------------------------------- restore

@pytest.mark.parametrize("name", ["c0", "c0p", "s1", "s2", "s3", "s4"])
def test_restore_matches_oracle(lsc, name):
    w = workload(name, num_slots=max(W.get(name).num_slots if name.startswith("c") else 0, 24))
    rows = W.combo_rows(w.num_slots, w.block_size, seed=21)
    with DevPool(w, seed=3, random_padding=True) as P:
        pre = {l: P.host[l].copy() for l in P.gdn_layers}
        rc, rep, hs = run_restore(P, rows, w.block_size)
        assert rc == L.LSC_OK and rep.launches == 1
        rc_o, regions, hs_o = oracle_restore(w, P, pre, rows, w.block_size)
        assert rc_o == oracle.OK
        np.testing.assert_array_equal(hs, hs_o)
        for l in P.gdn_layers:
            np.testing.assert_array_equal(P.download(l), regions[l])
        assert P.status() == L.LSC_OK


def test_restore_c0_four_rows(lsc):
    """The tiny workload's rows: one hit, one miss, one no-op, one duplicate source."""
    w = W.get("c0")
    rows = W.restore_rows("c0")
    with DevPool(w, seed=0) as P:
        pre = {l: P.host[l].copy() for l in P.gdn_layers}
        rc, rep, hs = run_restore(P, rows, 16)
        assert rc == L.LSC_OK and (rep.n_hit, rep.n_miss, rep.n_noop) == (2, 1, 1)
        _, regions, hs_o = oracle_restore(w, P, pre, rows, 16)
        np.testing.assert_array_equal(hs, hs_o)
        assert list(hs) == [1, 0, 1, 1]
        for l in P.gdn_layers:
            np.testing.assert_array_equal(P.download(l), regions[l])


def test_restore_many_rows_several_launches(lsc):
    """More hit rows and has_initial_state writes than one launch's plan holds."""
    w = workload("s4", num_slots=12000)
    rng = np.random.default_rng(5)
    perm = rng.permutation(w.num_slots)
    n = 8000
    live, spare = perm[:n], perm[n:]
    src = np.where(rng.random(n) < 0.6, spare[rng.integers(0, len(spare), n)], -1)
    nkv = 8 * rng.integers(0, 5, n)
    nkv[rng.random(n) < 0.1] += 3
    init = (rng.random(n) < 0.05).astype(np.uint8)
    rows = W._rows(live, src, nkv, init, 8, rng)
    with DevPool(w, seed=4) as P:
        pre = {l: P.host[l].copy() for l in P.gdn_layers}
        rc, rep, hs = run_restore(P, rows, 8)
        assert rc == L.LSC_OK and rep.launches >= 2 and rep.n_hit > 2048
        _, regions, hs_o = oracle_restore(w, P, pre, rows, 8)
        np.testing.assert_array_equal(hs, hs_o)
        for l in P.gdn_layers:
            np.testing.assert_array_equal(P.download(l), regions[l])


def test_restore_soft_cold_on_device(lsc):
    """No GDN layer: hits go cold, misses cold, no-ops unchanged, LSC_SOFT_COLD."""
    w = workload("c0", num_slots=40)
    layers = [W.ATTN] * 3
    rows = W.combo_rows(40, 16, seed=8)
    with DevPool(w, layers=layers) as P:
        rc, rep, hs = run_restore(P, rows, 16)
        assert rc == L.LSC_SOFT_COLD and rep.soft_cold == 1
        hs_o = rows.hs_prefill.copy()
        assert oracle.restore(oracle_pool(w, layers), {}, rows.live, rows.src, rows.nkv, 16, rows.initialized,
                              hs_o) == oracle.SOFT_COLD
        np.testing.assert_array_equal(hs, hs_o)


def test_restore_empty_and_noop_only(lsc):
    w = W.get("c0")
    with DevPool(w) as P:
        pre = {l: P.host[l].copy() for l in P.gdn_layers}
        empty = W._rows([], [], [], [], 16, np.random.default_rng(0))
        rc, rep, hs = run_restore(P, empty, 16)
        assert rc == L.LSC_OK and rep.launches == 0
        noop = W._rows([1, 2], [3, 4], [20, 0], [0, 0], 16, np.random.default_rng(0))
        rc, rep, hs = run_restore(P, noop, 16)
        assert rc == L.LSC_OK and rep.launches == 0 and list(hs) == [1, 0]
        for l in P.gdn_layers:
            np.testing.assert_array_equal(P.download(l), pre[l])


# ---------------------------------------------------------------- gather / scatter

@pytest.mark.parametrize("name", ["c0p", "s1", "s3", "s4"])
def test_gather_scatter_match_oracle(lsc, name):
    w = workload(name)
    Lo = oracle_layout(w)
    rng = np.random.default_rng(6)
    n = min(w.num_slots, 11)
    idx = rng.permutation(w.num_slots)[:n].astype(np.int32)
    idx[2] = -1
    has = (rng.random(n) < 0.7).astype(np.uint8)
    with DevPool(w, seed=5, random_padding=True) as P:
        l = P.gdn_layers[-1]
        pre = P.host[l].copy()
        conv = torch.full((n, Lo["conv_bytes"]), 0x77, dtype=torch.uint8, device="cuda")
        ssm = torch.full((n, Lo["ssm_bytes"]), 0x77, dtype=torch.uint8, device="cuda")
        di, dh = dev(idx), dev(has)
        assert L.lsc_gather(P.pool, l, di, dh, n, conv, ssm, torch.cuda.current_stream()) == L.LSC_OK
        rc, conv_o, ssm_o = oracle.gather(oracle_pool(w), pre, idx, has)
        assert rc == oracle.OK
        np.testing.assert_array_equal(conv.cpu().numpy(), conv_o)
        np.testing.assert_array_equal(ssm.cpu().numpy(), ssm_o)
        # scatter fresh content back: only the named views change
        new_conv = torch.from_numpy(rng.integers(0, 256, conv_o.shape, dtype=np.uint8)).cuda()
        new_ssm = torch.from_numpy(rng.integers(0, 256, ssm_o.shape, dtype=np.uint8)).cuda()
        assert L.lsc_scatter(P.pool, l, di, n, new_conv, new_ssm, torch.cuda.current_stream()) == L.LSC_OK
        reg_o = pre.copy()
        assert oracle.scatter(oracle_pool(w), reg_o, idx, new_conv.cpu().numpy(), new_ssm.cpu().numpy()) == oracle.OK
        np.testing.assert_array_equal(P.download(l), reg_o)
        # gather with no mask (all warm) then scatter: the region is unchanged
        idx2 = np.abs(idx).astype(np.int32)
        d2 = dev(idx2)
        before = P.download(l)
        assert L.lsc_gather(P.pool, l, d2, None, n, conv, ssm, None) == L.LSC_OK
        assert L.lsc_scatter(P.pool, l, d2, n, conv, ssm, None) == L.LSC_OK
        np.testing.assert_array_equal(P.download(l), before)
        assert P.status() == L.LSC_OK


def test_gather_scatter_out_of_range_index_sets_status(lsc):
    w = workload("c0p")
    Lo = oracle_layout(w)
    with DevPool(w, seed=1) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx = np.array([3, w.num_slots, 5], np.int32)
        conv = torch.full((3, Lo["conv_bytes"]), 0x77, dtype=torch.uint8, device="cuda")
        ssm = torch.full((3, Lo["ssm_bytes"]), 0x77, dtype=torch.uint8, device="cuda")
        assert L.lsc_gather(P.pool, l, dev(idx), None, 3, conv, ssm, None) == L.LSC_OK
        assert P.status() == L.LSC_ERR_OUT_OF_RANGE
        assert P.status() == L.LSC_OK  # read clears
        c = conv.cpu().numpy()
        assert not c[1].any()
        ok = np.array([3, -1, 5], np.int32)
        _, conv_o, _ = oracle.gather(oracle_pool(w), pre, ok)
        np.testing.assert_array_equal(c[[0, 2]], conv_o[[0, 2]])
        assert L.lsc_scatter(P.pool, l, dev(idx), 3, conv, ssm, None) == L.LSC_OK
        assert P.status() == L.LSC_ERR_OUT_OF_RANGE
        np.testing.assert_array_equal(P.download(l), pre)  # gathered rows written back unchanged


# ---------------------------------------------------------------- decode

DECODE_CASES = [
    ("c0", {}), ("c0p", {}), ("s1", {}), ("s2", {}), ("s3", {}), ("s4", {}),
    ("s4", {"conv_width": 2}), ("c0", {"conv_width": 8}),
    # eight v heads share one q/k head: one work item holds all eight
    ("c0", {"num_v_heads": 8, "conv_dim": 2 * 16 + 8 * 16}),
    # Hk = Hv: one v head per work item
    ("s1", {"num_k_heads": 4, "conv_dim": 2 * 4 * 32 + 4 * 32}),
    # dk = 64 with fp32 state
    ("s3", {"head_k_dim": 64, "head_v_dim": 96, "conv_dim": 2 * 2 * 64 + 4 * 96}),
    # fp32 conv, width 4, 16-byte aligned segments, but a work item of 2*16 + 3*12 = 68
    # channels: not whole 8-channel groups, so the channel-by-channel conv path
    ("s4", {"conv_dtype": W.F32}),
]


def decode_case(w, seed, n=None, cold_frac=0.25, pad_row=True, has_init_null=False):
    rng = np.random.default_rng(seed)
    n = n or min(w.num_slots, 9)
    idx = rng.permutation(w.num_slots)[:n].astype(np.int32)
    if pad_row:
        idx[n // 2] = -1
    has = None if has_init_null else (rng.random(n) >= cold_frac).astype(np.uint8)
    x, cw, a, b = W.decode_inputs(w, n, seed=seed, layer=0)
    return idx, has, x, cw, a, b


def run_decode(P, l, w, idx, has, x, cw, a, b, stream=None, flags=0):
    n = len(idx)
    out = torch.full((n, w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
    dx, dw = conv_bytes_dev(x, w.conv_dtype), conv_bytes_dev(cw, w.conv_dtype)
    di = dev(idx)
    dh = dev(has) if has is not None else None
    da, db = dev(a), dev(b)
    args = L.decode_args(n, w.num_k_heads, di, dh, dx, dw, da, db, out, flags)
    rc = L.lsc_gdn_decode(P.pool, l, args, stream)
    torch.cuda.synchronize()
    return rc, out.cpu().numpy()


def check_decode(w, P, l, pre, idx, has, x, cw, a, b, out):
    reg_o = pre.copy()
    rc, out_o = oracle.gdn_decode(oracle_pool(w), reg_o, idx, has, W.to_dtype_bytes(x, w.conv_dtype),
                                  W.to_dtype_bytes(cw, w.conv_dtype), w.num_k_heads, a, b)
    assert rc == oracle.OK
    t = tol(w.ssm_dtype)
    np.testing.assert_allclose(out, out_o, **t)
    got = P.download(l)
    Lo = oracle_layout(w)
    pages_g = got.reshape(w.num_slots, w.page_bytes)
    pages_o = reg_o.reshape(w.num_slots, w.page_bytes)
    # conv state: the shift stores values unchanged, so bit-exact
    np.testing.assert_array_equal(pages_g[:, :Lo["conv_bytes"]], pages_o[:, :Lo["conv_bytes"]])
    ssm = slice(Lo["ssm_offset"], Lo["ssm_offset"] + Lo["ssm_bytes"])
    sg = W.from_dtype_bytes(np.ascontiguousarray(pages_g[:, ssm]), w.ssm_dtype)
    so = W.from_dtype_bytes(np.ascontiguousarray(pages_o[:, ssm]), w.ssm_dtype)
    np.testing.assert_allclose(sg, so, **t)
    mask = ~payload_mask(w, Lo)  # padding and inter-view gap: untouched
    np.testing.assert_array_equal(pages_g[:, mask], pre.reshape(w.num_slots, -1)[:, mask])
    untouched = [s for s in range(w.num_slots) if s not in set(idx.tolist())]
    np.testing.assert_array_equal(pages_g[untouched], pre.reshape(w.num_slots, -1)[untouched])


@pytest.mark.parametrize("name,kw", DECODE_CASES, ids=[f"{n}-{'-'.join(f'{k}{v}' for k, v in kw.items())}" for n, kw in DECODE_CASES])
def test_decode_matches_oracle(lsc, name, kw):
    w = workload(name, **kw)
    with DevPool(w, seed=7, random_padding=True) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, x, cw, a, b = decode_case(w, seed=3)
        rc, out = run_decode(P, l, w, idx, has, x, cw, a, b, torch.cuda.current_stream())
        assert rc == L.LSC_OK, L.lsc_error_string(rc)
        check_decode(w, P, l, pre, idx, has, x, cw, a, b, out)
        assert P.status() == L.LSC_OK


@pytest.mark.big
@pytest.mark.parametrize("flags", [0, L.LSC_DECODE_EARLY_STATE])
def test_decode_more_items_than_one_launch_holds(lsc, flags):
    """A CTA holds at most 512 work items per launch, so more than 512 x SMs /
    Hk rows are split over several launches; the result is the same."""
    w0 = W.small("s1")   # Hk = 2: the split happens below the 65535-row limit
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 512 * sms // w0.num_k_heads + 123
    assert n <= 65535
    w = workload("s1", num_slots=n + 7, layers=[W.GDN])
    with DevPool(w, seed=17) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, x, cw, a, b = decode_case(w, seed=19, n=n)
        rc, out = run_decode(P, l, w, idx, has, x, cw, a, b, flags=flags)
        assert rc == L.LSC_OK
        check_decode(w, P, l, pre, idx, has, x, cw, a, b, out)
        assert P.status() == L.LSC_OK


@pytest.mark.parametrize("flags", [0, L.LSC_DECODE_EARLY_STATE])
def test_decode_fp32_dk128_ring_wraps(lsc, flags):
    """The benchmarked decode instantiation (head_k_dim 128, fp32 state, bf16
    conv, width 4) with 512 rows of two q/k heads: 1024 work items, so each CTA
    holds six or seven items of four 32 KiB tiles and its ring of stages wraps
    several times; cold rows, a padding row and unselected slots included."""
    w = workload("s3", num_slots=600)
    with DevPool(w, seed=41, random_padding=True) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, x, cw, a, b = decode_case(w, seed=42, n=512, cold_frac=0.1)
        assert len(idx) * w.num_k_heads >= 6 * torch.cuda.get_device_properties(0).multi_processor_count
        rc, out = run_decode(P, l, w, idx, has, x, cw, a, b, torch.cuda.current_stream(), flags)
        assert rc == L.LSC_OK, L.lsc_error_string(rc)
        check_decode(w, P, l, pre, idx, has, x, cw, a, b, out)
        assert P.status() == L.LSC_OK


@pytest.mark.parametrize("name", ["c0p", "s1", "s3", "s4"])
def test_decode_early_state_chain_of_layers(lsc, name):
    """Every GDN layer of the pool decoded back to back on one stream with the
    early state flag and no host sync in between (each launch may read its
    rows and first state tiles while the previous layer's launch runs), then
    each layer against the oracle.  Covers the vector and the channel-by-channel
    conv paths, cold rows and a padding row."""
    w = workload(name, layers=[W.GDN, W.ATTN, W.GDN, W.GDN, W.ATTN, W.GDN])
    with DevPool(w, seed=23, random_padding=True) as P:
        s = torch.cuda.Stream()
        keep, cases = [], {}
        for l in P.gdn_layers:
            idx, has, x, cw, a, b = decode_case(w, seed=100 + l)
            n = len(idx)
            out = torch.full((n, w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
            t = [dev(idx), dev(has), conv_bytes_dev(x, w.conv_dtype), conv_bytes_dev(cw, w.conv_dtype), dev(a),
                 dev(b), out]
            keep.append(t)
            cases[l] = (idx, has, x, cw, a, b, out)
        torch.cuda.synchronize()
        for l, t in zip(P.gdn_layers, keep):
            args = L.decode_args(len(cases[l][0]), w.num_k_heads, *t, flags=L.LSC_DECODE_EARLY_STATE)
            assert L.lsc_gdn_decode(P.pool, l, args, s) == L.LSC_OK
        torch.cuda.synchronize()
        for l in P.gdn_layers:
            idx, has, x, cw, a, b, out = cases[l]
            check_decode(w, P, l, P.host[l].copy(), idx, has, x, cw, a, b, out.cpu().numpy())
        assert P.status() == L.LSC_OK


def test_decode_early_state_same_layer_disjoint_rows(lsc):
    """Two decodes of one layer back to back on one stream, on disjoint row
    sets, the second with the early state flag: the first writes none of the
    second's rows, which is what the flag asks of the kernel before it.  Both
    against the oracle applied in order."""
    w = workload("s3", num_slots=600)
    with DevPool(w, seed=31, random_padding=True) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        rng = np.random.default_rng(32)
        perm = rng.permutation(w.num_slots).astype(np.int32)
        calls = []
        for h, flags in ((0, 0), (1, L.LSC_DECODE_EARLY_STATE)):
            idx = perm[h * 300:(h + 1) * 300].copy()
            idx[7] = -1
            has = (rng.random(300) >= 0.2).astype(np.uint8)
            x, cw, a, b = W.decode_inputs(w, 300, seed=40 + h, layer=0)
            out = torch.full((300, w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
            t = [dev(idx), dev(has), conv_bytes_dev(x, w.conv_dtype), conv_bytes_dev(cw, w.conv_dtype), dev(a), dev(b),
                 out]
            calls.append((idx, has, x, cw, a, b, out, t, flags))
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        for idx, has, x, cw, a, b, out, t, flags in calls:
            args = L.decode_args(len(idx), w.num_k_heads, *t, flags=flags)
            assert L.lsc_gdn_decode(P.pool, l, args, s) == L.LSC_OK
        torch.cuda.synchronize()
        reg = pre.copy()
        for idx, has, x, cw, a, b, out, t, flags in calls:
            rc, o = oracle.gdn_decode(oracle_pool(w), reg, idx, has, W.to_dtype_bytes(x, w.conv_dtype),
                                      W.to_dtype_bytes(cw, w.conv_dtype), w.num_k_heads, a, b)
            assert rc == oracle.OK
            np.testing.assert_allclose(out.cpu().numpy(), o, **tol(w.ssm_dtype))
        got = P.download(l).reshape(w.num_slots, -1)
        Lo = oracle_layout(w)
        exp = reg.reshape(w.num_slots, -1)
        np.testing.assert_array_equal(got[:, :Lo["conv_bytes"]], exp[:, :Lo["conv_bytes"]])
        ssm = slice(Lo["ssm_offset"], Lo["ssm_offset"] + Lo["ssm_bytes"])
        np.testing.assert_allclose(W.from_dtype_bytes(np.ascontiguousarray(got[:, ssm]), w.ssm_dtype),
                                   W.from_dtype_bytes(np.ascontiguousarray(exp[:, ssm]), w.ssm_dtype),
                                   **tol(w.ssm_dtype))
        mask = ~payload_mask(w, Lo)
        np.testing.assert_array_equal(got[:, mask], pre.reshape(w.num_slots, -1)[:, mask])
        assert P.status() == L.LSC_OK


def test_decode_two_steps_all_warm(lsc):
    """Two consecutive tokens on the same slots (the second reads what the first
    wrote), has_init NULL."""
    w = workload("s2")
    with DevPool(w, seed=8) as P:
        l = P.gdn_layers[1]
        pre = P.host[l].copy()
        for step in range(2):
            idx, has, x, cw, a, b = decode_case(w, seed=11, pad_row=False, has_init_null=True)
            x = x + step  # a different token
            rc, out = run_decode(P, l, w, idx, has, x, cw, a, b)
            assert rc == L.LSC_OK
            check_decode(w, P, l, pre, idx, has, x, cw, a, b, out)
            pre = P.download(l)


def test_decode_out_of_range_row(lsc):
    w = workload("s4")
    with DevPool(w, seed=9) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, x, cw, a, b = decode_case(w, seed=4, pad_row=False)
        bad = idx.copy()
        bad[1] = w.num_slots + 2
        rc, out = run_decode(P, l, w, bad, has, x, cw, a, b)
        assert rc == L.LSC_OK
        assert P.status() == L.LSC_ERR_OUT_OF_RANGE
        assert not out[1].any()
        ok = idx.copy()
        ok[1] = -1
        check_decode(w, P, l, pre, ok, has, x, cw, a, b, out)


@pytest.mark.parametrize("name", ["c0p", "s4"])  # vector conv path / channel-by-channel path
def test_decode_bounded_wait_expiry_reports_and_stays_usable(lsc, name, monkeypatch):
    """LSC_FAULT=timeout0 makes every mbarrier wait of the decode give up at
    once: the kernel records LSC_ERR_DEV_TIMEOUT, drains its copies in flight
    and returns.  The rows' states are then unspecified, but nothing outside
    the rows' conv and ssm views is written, and the context stays usable."""
    w = workload(name)
    Lo = oracle_layout(w)
    with DevPool(w, seed=15) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, x, cw, a, b = decode_case(w, seed=5)
        monkeypatch.setenv("LSC_FAULT", "timeout0")
        rc, _ = run_decode(P, l, w, idx, has, x, cw, a, b)
        monkeypatch.delenv("LSC_FAULT")
        assert rc == L.LSC_OK
        assert P.status() == L.LSC_ERR_DEV_TIMEOUT
        got = P.download(l).reshape(w.num_slots, -1)
        touched = np.zeros((w.num_slots, w.page_bytes), bool)
        touched[idx[idx >= 0]] = payload_mask(w, Lo)
        np.testing.assert_array_equal(got[~touched], pre.reshape(w.num_slots, -1)[~touched])
        P.region(l).copy_(torch.from_numpy(pre))  # put the pre-image back
        rc, out = run_decode(P, l, w, idx, has, x, cw, a, b)
        assert rc == L.LSC_OK and P.status() == L.LSC_OK
        check_decode(w, P, l, pre, idx, has, x, cw, a, b, out)


def test_decode_rejects(lsc):
    w = workload("c0")
    with DevPool(w) as P:
        args = L.decode_args(2, 3, 1, 1, 1, 1, 1, 1, 1)  # Hv % Hk != 0
        assert L.lsc_gdn_decode(P.pool, 0, args) == L.LSC_ERR_INVALID_ARG
        args = L.decode_args(2, 1, 1, 1, 1, 1, 1, 1, 1)
        assert L.lsc_gdn_decode(P.pool, 1, args) == L.LSC_ERR_STATELESS_LAYER
        args = L.decode_args(0, 1, None, None, None, None, None, None, None)
        assert L.lsc_gdn_decode(P.pool, 0, args) == L.LSC_OK
        for bad in (2, 0x80000000, L.LSC_DECODE_EARLY_STATE | 4):  # flag bits the call does not define
            args = L.decode_args(2, 1, 256, 256, 256, 256, 256, 256, 256, bad)
            assert L.lsc_gdn_decode(P.pool, 0, args) == L.LSC_ERR_INVALID_ARG
    w = workload("c0", head_k_dim=24, conv_dim=2 * 24 + 2 * 16, ssm_dtype=W.F32)
    with DevPool(w) as P:
        # aligned stand-in addresses (never dereferenced: the shape is refused first)
        args = L.decode_args(2, 1, 256, 256, 256, 256, 256, 256, 256)
        assert L.lsc_gdn_decode(P.pool, 0, args) == L.LSC_ERR_UNSUPPORTED
        args = L.decode_args(2, 1, 1, 1, 1, 1, 1, 1, 1)
        assert L.lsc_gdn_decode(P.pool, 0, args) == L.LSC_ERR_MISALIGNED


# ---------------------------------------------------------------- recurrence

REC_CASES = [("c0", {}), ("s1", {}), ("s2", {}), ("s3", {}), ("s4", {}),
             ("s3", {"head_k_dim": 64, "head_v_dim": 96, "conv_dim": 2 * 2 * 64 + 4 * 96})]


def rec_case(w, lengths, seed, pad_seq=True):
    rng = np.random.default_rng(seed)
    idx = rng.permutation(w.num_slots)[:len(lengths)].astype(np.int32)
    if pad_seq:
        idx[-1] = -1
    has = (rng.random(len(lengths)) < 0.6).astype(np.uint8)
    cu, q, k, v, a, b = W.recurrent_inputs(w, lengths, seed=seed, layer=0)
    return idx, has, cu, q, k, v, a, b


def run_recurrent(P, l, w, idx, has, cu, q, k, v, a, b, algorithm=L.LSC_RECURRENT_AUTO):
    T = int(cu[-1])
    out = torch.full((max(T, 1), w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
    t = [dev(z) for z in (idx, has, cu, q, k, v, a, b)]
    args = L.recurrent_args(len(idx), w.num_k_heads, T, *t, out, algorithm=algorithm)
    rc = L.lsc_gdn_recurrent(P.pool, l, args, torch.cuda.current_stream())
    torch.cuda.synchronize()
    return rc, out.cpu().numpy()[:T]


def check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out):
    reg_o = pre.copy()
    rc, out_o = oracle.gdn_recurrent(oracle_pool(w), reg_o, idx, has, cu, w.num_k_heads, q, k, v, a, b)
    assert rc == oracle.OK
    t = tol(w.ssm_dtype)
    np.testing.assert_allclose(out, out_o, **t)
    got = P.download(l)
    Lo = oracle_layout(w)
    pg, po = got.reshape(w.num_slots, -1), reg_o.reshape(w.num_slots, -1)
    ssm = slice(Lo["ssm_offset"], Lo["ssm_offset"] + Lo["ssm_bytes"])
    np.testing.assert_allclose(W.from_dtype_bytes(np.ascontiguousarray(pg[:, ssm]), w.ssm_dtype),
                               W.from_dtype_bytes(np.ascontiguousarray(po[:, ssm]), w.ssm_dtype), **t)
    other = np.ones(w.page_bytes, bool)
    other[ssm] = False  # conv state, gap and padding: untouched
    np.testing.assert_array_equal(pg[:, other], pre.reshape(w.num_slots, -1)[:, other])


REC_ALGOS = {"token": L.LSC_RECURRENT_TOKEN, "chunked": L.LSC_RECURRENT_CHUNKED}

# head_k_dim 128 with head_v_dim below 128 for the chunked form: a multiple of 4
# (16-byte v rows) and an odd one (4-byte v copies, a ragged last row pair)
REC_CASES_128 = [("s3", {"head_v_dim": 100, "conv_dim": 2 * 2 * 128 + 4 * 100}),
                 ("s2", {"head_v_dim": 37, "conv_dim": 2 * 2 * 128 + 4 * 37}),
                 ("s3", {"head_v_dim": 1, "conv_dim": 2 * 2 * 128 + 4 * 1})]


def _case_id(n, kw):
    return f"{n}-{'-'.join(f'{k}{v}' for k, v in kw.items())}"


@pytest.mark.parametrize("algo", list(REC_ALGOS))
@pytest.mark.parametrize("name,kw", REC_CASES + REC_CASES_128, ids=[_case_id(n, kw) for n, kw in REC_CASES + REC_CASES_128])
def test_recurrent_matches_oracle(lsc, name, kw, algo):
    w = workload(name, **kw)
    lengths = [0, 1, 15, 16, 17, 40, 5][:min(7, w.num_slots)]
    with DevPool(w, seed=12, random_padding=True) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, q, k, v, a, b = rec_case(w, lengths, seed=5)
        rc, out = run_recurrent(P, l, w, idx, has, cu, q, k, v, a, b, REC_ALGOS[algo])
        if algo == "chunked" and w.head_k_dim != 128:
            assert rc == L.LSC_ERR_UNSUPPORTED
            np.testing.assert_array_equal(P.download(l), pre)
            return
        assert rc == L.LSC_OK, L.lsc_error_string(rc)
        check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out)
        assert P.status() == L.LSC_OK


@pytest.mark.parametrize("algo", list(REC_ALGOS))
def test_recurrent_long_sequence_fp32(lsc, algo):
    """A few hundred tokens: the recurrence stays within the fp32 bound."""
    w = workload("s3")
    with DevPool(w, seed=13) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, q, k, v, a, b = rec_case(w, [300, 129], seed=6, pad_seq=False)
        rc, out = run_recurrent(P, l, w, idx, has, cu, q, k, v, a, b, REC_ALGOS[algo])
        assert rc == L.LSC_OK
        check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out)


@pytest.mark.parametrize("algo", list(REC_ALGOS))
def test_recurrent_equals_decode_free_steps(lsc, algo):
    """alpha = 1, beta = 0 at every token: the state is unchanged bit for bit
    and o_t = S q_t (the closed form of the benchmark spec, on the GPU)."""
    w = workload("s2")
    with DevPool(w, seed=14) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, q, k, v, a, b = rec_case(w, [9, 20], seed=7, pad_seq=False)
        has[:] = 1
        a[:] = 1.0
        b[:] = 0.0
        rc, out = run_recurrent(P, l, w, idx, has, cu, q, k, v, a, b, REC_ALGOS[algo])
        assert rc == L.LSC_OK
        np.testing.assert_array_equal(P.download(l), pre)
        check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out)


@pytest.mark.parametrize("algo", list(REC_ALGOS))
def test_recurrent_gate_extremes(lsc, algo):
    """alpha = 0 (the state restarts from b v k^T), alpha ~ 1e-9 (the decay
    products underflow inside a chunk) and beta = 1, inside and across chunks."""
    w = workload("s3")
    with DevPool(w, seed=15) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, q, k, v, a, b = rec_case(w, [50, 33, 16], seed=8, pad_seq=False)
        has[:] = 1
        a[3] = 0.0
        a[20:27] = 1e-9
        a[cu[1] + 15] = 0.0
        b[cu[1]:cu[1] + 10] = 1.0
        rc, out = run_recurrent(P, l, w, idx, has, cu, q, k, v, a, b, REC_ALGOS[algo])
        assert rc == L.LSC_OK
        check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out)


@pytest.mark.parametrize("algo", list(REC_ALGOS))
def test_recurrent_many_sequences(lsc, algo):
    """More sequences than the CTAs rank by length (256): the plain order."""
    w = workload("s3", num_slots=320)
    rng = np.random.default_rng(21)
    lengths = rng.integers(0, 24, 300).tolist()
    with DevPool(w, seed=16) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, q, k, v, a, b = rec_case(w, lengths, seed=10)
        rc, out = run_recurrent(P, l, w, idx, has, cu, q, k, v, a, b, REC_ALGOS[algo])
        assert rc == L.LSC_OK
        check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out)
        assert P.status() == L.LSC_OK


@pytest.mark.parametrize("algo", list(REC_ALGOS))
def test_recurrent_bad_rows_are_skipped_and_reported(lsc, algo):
    """A slot id past the pool: that sequence's outputs are zero, no state is
    touched, OUT_OF_RANGE is recorded; the other sequences are unaffected."""
    w = workload("s3")
    with DevPool(w, seed=17) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, q, k, v, a, b = rec_case(w, [20, 33, 7], seed=11, pad_seq=False)
        bad = idx.copy()
        bad[1] = w.num_slots + 3
        rc, out = run_recurrent(P, l, w, bad, has, cu, q, k, v, a, b, REC_ALGOS[algo])
        assert rc == L.LSC_OK
        assert P.status() == L.LSC_ERR_OUT_OF_RANGE
        np.testing.assert_array_equal(out[cu[1]:cu[2]], 0.0)
        ref = idx.copy()
        ref[1] = -1  # the oracle's view: a padding sequence
        check_recurrent(w, P, l, pre, ref, has, cu, q, k, v, a, b, out)


@pytest.mark.parametrize("algo", list(REC_ALGOS))
def test_recurrent_null_has_init_means_all_warm(lsc, algo):
    """has_init = NULL: every sequence starts from its slot's state."""
    w = workload("s3")
    with DevPool(w, seed=18) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, q, k, v, a, b = rec_case(w, [17, 5, 40], seed=12, pad_seq=False)
        T = int(cu[-1])
        out = torch.full((T, w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
        t = [dev(z) for z in (idx, cu, q, k, v, a, b)]
        args = L.recurrent_args(len(idx), w.num_k_heads, T, t[0], None, *t[1:], out, algorithm=REC_ALGOS[algo])
        assert L.lsc_gdn_recurrent(P.pool, l, args, torch.cuda.current_stream()) == L.LSC_OK
        torch.cuda.synchronize()
        has[:] = 1
        check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out.cpu().numpy())


def test_recurrent_rejects(lsc):
    w = workload("s1")
    with DevPool(w) as P:
        idx, has, cu, q, k, v, a, b = rec_case(w, [3], seed=9, pad_seq=False)
        for algo, rc_want in ((3, L.LSC_ERR_INVALID_ARG), (-1, L.LSC_ERR_INVALID_ARG),
                              (L.LSC_RECURRENT_CHUNKED, L.LSC_ERR_UNSUPPORTED)):  # s1: head_k_dim 32
            rc, _ = run_recurrent(P, P.gdn_layers[0], w, idx, has, cu, q, k, v, a, b, algo)
            assert rc == rc_want
