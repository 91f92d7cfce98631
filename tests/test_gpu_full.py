"""Full-size parity at the serving workloads, in the launch configuration the
benchmark times.  The pools (10-79 GB) are filled on the device with torch's
seeded generator; the oracle checks sampled layers (whole layer regions, byte
for byte) and sampled sequences, which it computes one by one on the host."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_lsc_gb300 import lsc as L
from linear_attention_state_lsc_gb300 import workloads as W

from _gpu import DevPool, dev, tol
from _util import oracle_layout, oracle_pool
from test_gpu_parity import check_decode, run_decode, run_restore

pytestmark = [pytest.mark.gpu, pytest.mark.big]


def _one_layer_pool(w):
    return oracle_pool(w, layers=[W.GDN])


def _restore_full(name, sample_gdn):
    w = W.get(name)
    rows = W.restore_rows(name)
    with DevPool(w, seed=0, device_fill=True) as P:
        sample = [P.gdn_layers[g] for g in sample_gdn]
        pre = {l: P.download(l) for l in sample}
        rc, rep, hs = run_restore(P, rows, w.block_size)
        assert rc == L.LSC_OK and rep.launches == 1
        hs_o = rows.hs_prefill.copy()
        for l in sample:
            reg = pre[l].copy()
            h = rows.hs_prefill.copy()
            assert oracle.restore(_one_layer_pool(w), {0: reg}, rows.live, rows.src, rows.nkv, w.block_size,
                                  rows.initialized, h) == oracle.OK
            np.testing.assert_array_equal(P.download(l), reg)
            hs_o = h
        np.testing.assert_array_equal(hs, hs_o)
        assert P.status() == L.LSC_OK
        return rep


def test_c1_restore_serving_scale(lsc):
    rep = _restore_full("c1", [0, 17, 35])
    assert rep.n_hit == 64 and rep.bytes_copied == 64 * 36 * 2146304


def test_c3_restore_storm(lsc):
    rep = _restore_full("c3", [0, 35])
    assert (rep.n_hit, rep.n_miss, rep.n_noop) == (205, 154, 153)


@pytest.mark.parametrize("flags", [0, L.LSC_DECODE_EARLY_STATE])
def test_c2_decode_full_layer(lsc, flags):
    w = W.get("c2")
    with DevPool(w, seed=0, device_fill=True) as P:
        rng = np.random.default_rng(2)
        for g, n in ((1, 192), (0, 256)):  # 192 rows leave 64 slots unselected
            l = P.gdn_layers[g]
            pre = P.download(l)
            idx = rng.permutation(w.num_slots)[:n].astype(np.int32)
            has = np.ones(n, np.uint8)
            x, cw, a, b = W.decode_inputs(w, n, seed=0, layer=l)
            rc, out = run_decode(P, l, w, idx, has, x, cw, a, b, flags=flags)
            assert rc == L.LSC_OK
            check_decode(w, P, l, pre, idx, has, x, cw, a, b, out)
        assert P.status() == L.LSC_OK


@pytest.mark.parametrize("algorithm", [L.LSC_RECURRENT_TOKEN, L.LSC_RECURRENT_CHUNKED], ids=["token", "chunked"])
def test_c4_resume_prefill_sampled_sequences(lsc, algorithm):
    w = W.get("c4")
    lengths = W.seq_lengths(64, 64, 2048, seed=0)
    rng = np.random.default_rng(4)
    with DevPool(w, seed=0, device_fill=True) as P:
        l = P.gdn_layers[0]
        pre = P.download(l)
        idx = rng.permutation(w.num_slots)[:64].astype(np.int32)
        has = (rng.random(64) < 0.5).astype(np.uint8)
        cu, q, k, v, a, b = W.recurrent_inputs(w, lengths, seed=0, layer=l)
        T = int(cu[-1])
        out = torch.empty((T, w.num_v_heads, w.head_v_dim), device="cuda")
        t = [dev(z) for z in (idx, has, cu, q, k, v, a, b)]
        args = L.recurrent_args(64, w.num_k_heads, T, *t, out, algorithm=algorithm)
        assert L.lsc_gdn_recurrent(P.pool, l, args, torch.cuda.current_stream()) == L.LSC_OK
        torch.cuda.synchronize()
        got = P.download(l).reshape(w.num_slots, -1)
        out = out.cpu().numpy()
        Lo = oracle_layout(w)
        ssm = slice(Lo["ssm_offset"], Lo["ssm_offset"] + Lo["ssm_bytes"])
        picks = [int(np.argmax(lengths)), int(np.argmin(lengths)), 31]
        for i in picks:
            sl = slice(cu[i], cu[i + 1])
            reg = pre.copy()
            sub_cu = np.array([0, lengths[i]], np.int32)
            rc, o = oracle.gdn_recurrent(oracle_pool(w), reg, idx[i:i + 1], has[i:i + 1], sub_cu, w.num_k_heads,
                                         q[sl], k[sl], v[sl], a[sl], b[sl])
            assert rc == oracle.OK
            np.testing.assert_allclose(out[sl], o, **tol(w.ssm_dtype))
            s = idx[i]
            np.testing.assert_allclose(W.from_dtype_bytes(np.ascontiguousarray(got[s, ssm]), w.ssm_dtype),
                                       W.from_dtype_bytes(np.ascontiguousarray(reg.reshape(w.num_slots, -1)[s, ssm]),
                                                          w.ssm_dtype), **tol(w.ssm_dtype))
        # conv states and padding of every slot untouched, unselected slots unchanged
        other = np.ones(w.page_bytes, bool)
        other[ssm] = False
        np.testing.assert_array_equal(got[:, other], pre.reshape(w.num_slots, -1)[:, other])
        unsel = sorted(set(range(w.num_slots)) - set(idx.tolist()))
        np.testing.assert_array_equal(got[unsel], pre.reshape(w.num_slots, -1)[unsel])
        assert P.status() == L.LSC_OK


@pytest.mark.parametrize("flags", [0, L.LSC_DECODE_EARLY_STATE])
def test_c1_serving_step_back_to_back(lsc, flags):
    """The benchmarked step as the benchmark issues it: lsc_restore of the 64
    c1 rows on a prepare stream, an event, then 36 lsc_gdn_decode launches back
    to back on the forward stream with no host sync, then a second token (36
    more launches).  Hit rows, has_initial_state, both tokens' outputs and the
    final states of three sampled layers against the oracle.  With the early
    state flag each launch streams its layer's first state tiles while the
    previous layer's launch finishes (the first launch of each token follows
    the event or the other layer's decode, neither writing its rows)."""
    w = W.get("c1")
    rows = W.restore_rows("c1")
    n = len(rows.live)
    with DevPool(w, seed=0, device_fill=True) as P:
        sample = [P.gdn_layers[g] for g in (0, 17, 35)]
        pre = {l: P.download(l) for l in sample}
        inputs = {}  # (token, layer) -> x, conv weights, alpha, beta (float32, host)
        for tok in range(2):
            for l in P.gdn_layers:
                x, cw, a, b = W.decode_inputs(w, n, seed=tok, layer=l)
                inputs[tok, l] = (x, cw, a, b)
        bf = torch.bfloat16
        idx = dev(rows.live.astype(np.int32))
        hs = dev(rows.hs_prefill)
        dx = {k: torch.from_numpy(v[0]).to(bf).cuda() for k, v in inputs.items()}
        dw = {l: torch.from_numpy(inputs[0, l][1]).to(bf).cuda() for l in P.gdn_layers}
        da = {k: dev(v[2]) for k, v in inputs.items()}
        db = {k: dev(v[3]) for k, v in inputs.items()}
        out = {k: torch.full((n, w.num_v_heads, w.head_v_dim), float("nan"), device="cuda") for k in inputs}
        ops = L.ops_array(rows.live, rows.src, rows.restore_hash, rows.save_hash, rows.save_slot)
        prep, fwd = torch.cuda.Stream(), torch.cuda.current_stream()
        ev = torch.cuda.Event()
        ev.record(fwd)
        torch.cuda.synchronize()
        prep.wait_stream(fwd)
        rc, rep = L.lsc_restore(P.pool, ops, rows.nkv, rows.block_size, rows.initialized, hs, prep, ev)
        assert rc == L.LSC_OK and rep.n_hit == 64 and rep.launches == 1
        fwd.wait_event(ev)
        for tok in range(2):
            for l in P.gdn_layers:
                args = L.decode_args(n, w.num_k_heads, idx, hs, dx[tok, l], dw[l], da[tok, l], db[tok, l],
                                     out[tok, l], flags)
                assert L.lsc_gdn_decode(P.pool, l, args, fwd) == L.LSC_OK
        torch.cuda.synchronize()
        hs_o = rows.hs_prefill.copy()
        Lo = oracle_layout(w)
        t = tol(w.ssm_dtype)
        for l in sample:
            reg = pre[l].copy()
            h = rows.hs_prefill.copy()
            assert oracle.restore(_one_layer_pool(w), {0: reg}, rows.live, rows.src, rows.nkv, rows.block_size,
                                  rows.initialized, h) == oracle.OK
            hs_o = h
            for tok in range(2):
                x, cw, a, b = inputs[tok, l]
                rc, o = oracle.gdn_decode(oracle_pool(w), reg, rows.live, h, W.to_dtype_bytes(x, w.conv_dtype),
                                          W.to_dtype_bytes(inputs[0, l][1], w.conv_dtype), w.num_k_heads, a, b)
                assert rc == oracle.OK
                np.testing.assert_allclose(out[tok, l].cpu().numpy(), o, **t)
            got = P.download(l).reshape(w.num_slots, -1)
            exp = reg.reshape(w.num_slots, -1)
            np.testing.assert_array_equal(got[:, :Lo["conv_bytes"]], exp[:, :Lo["conv_bytes"]])
            ssm = slice(Lo["ssm_offset"], Lo["ssm_offset"] + Lo["ssm_bytes"])
            np.testing.assert_allclose(W.from_dtype_bytes(np.ascontiguousarray(got[:, ssm]), w.ssm_dtype),
                                       W.from_dtype_bytes(np.ascontiguousarray(exp[:, ssm]), w.ssm_dtype), **t)
            unsel = sorted(set(range(w.num_slots)) - set(rows.live.tolist()))
            np.testing.assert_array_equal(got[unsel], pre[l].reshape(w.num_slots, -1)[unsel])
        np.testing.assert_array_equal(hs.cpu().numpy(), hs_o)
        assert P.status() == L.LSC_OK
