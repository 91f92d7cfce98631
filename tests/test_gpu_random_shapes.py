"""Seeded random shapes against the oracle: q/k head counts, v heads per q/k
head (1, 2, 4, 8), head dims, conv widths 2..8, both dtypes of each state and
varying page padding, for the fused decode, both recurrence orders, the
prefill conv, and (bit-exact) the restore, gather and scatter -- beyond the
fixed cases of test_gpu_parity.py and test_gpu_prefill.py.  The shapes are drawn once from a fixed seed, so a failure
names a reproducible case.

Sources: vLLM-Ascend "非连续 KV Cache" §6 (causal_conv1d_update,
recurrent_gated_delta_rule); Kapitsa "Attention 与 Gated DeltaNet 保存的历史不同".
"""
import numpy as np
import pytest
import torch

from linear_attention_state_lsc_gb300 import lsc as L
from linear_attention_state_lsc_gb300 import workloads as W

from _gpu import DevPool
import oracle
from _util import oracle_layout, oracle_pool
from test_gpu_parity import (REC_ALGOS, check_decode, check_recurrent, decode_case, oracle_restore, rec_case,
                             run_decode, run_recurrent, run_restore, workload)

pytestmark = pytest.mark.gpu


def random_shapes(seed, n):
    rng = np.random.default_rng(seed)
    shapes = []
    for _ in range(n):
        hk = int(rng.choice([1, 2, 3]))
        group = int(rng.choice([1, 2, 4, 8]))
        dk = int(rng.choice([16, 32, 64, 128]))
        dv = int(rng.choice([8, 12, 24, 37, 64, 96, 128]))
        shapes.append(dict(num_k_heads=hk, num_v_heads=hk * group, head_k_dim=dk, head_v_dim=dv,
                           conv_width=int(rng.integers(2, 9)), conv_dim=2 * hk * dk + hk * group * dv,
                           conv_dtype=str(rng.choice([W.F32, W.BF16])), ssm_dtype=str(rng.choice([W.F32, W.BF16]))))
    return shapes


SHAPES = random_shapes(2026, 16)


def _id(kw):
    return "Hk{num_k_heads}-Hv{num_v_heads}-dk{head_k_dim}-dv{head_v_dim}-W{conv_width}-{conv_dtype}-{ssm_dtype}".format(**kw)


@pytest.mark.parametrize("kw", SHAPES, ids=[_id(k) for k in SHAPES])
def test_decode_random_shape(lsc, kw):
    w = workload("s1", **kw)
    with DevPool(w, seed=31, random_padding=True) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, x, cw, a, b = decode_case(w, seed=32)
        rc, out = run_decode(P, l, w, idx, has, x, cw, a, b, torch.cuda.current_stream())
        assert rc == L.LSC_OK, L.lsc_error_string(rc)
        check_decode(w, P, l, pre, idx, has, x, cw, a, b, out)
        assert P.status() == L.LSC_OK


@pytest.mark.parametrize("algo", list(REC_ALGOS))
@pytest.mark.parametrize("kw", SHAPES, ids=[_id(k) for k in SHAPES])
def test_recurrent_random_shape(lsc, kw, algo):
    w = workload("s1", **kw)
    lengths = [33, 0, 16, 7, 70]
    with DevPool(w, seed=33, random_padding=True) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, q, k, v, a, b = rec_case(w, lengths, seed=34)
        rc, out = run_recurrent(P, l, w, idx, has, cu, q, k, v, a, b, REC_ALGOS[algo])
        if algo == "chunked" and w.head_k_dim != 128:
            assert rc == L.LSC_ERR_UNSUPPORTED
            return
        assert rc == L.LSC_OK, L.lsc_error_string(rc)
        check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out)
        assert P.status() == L.LSC_OK


@pytest.mark.parametrize("x_offset", [0, 1], ids=["aligned", "x-off-16B"])
@pytest.mark.parametrize("kw", SHAPES, ids=[_id(k) for k in SHAPES])
def test_prefill_conv_random_shape(lsc, kw, x_offset):
    """The fused 8-channel path where the shape allows it (channel counts and
    head dims that are multiples of 8, dk/8 a power of two), the two-pass path
    otherwise or with x off a 16-byte boundary."""
    from test_gpu_prefill import check, inputs, run
    w = workload("s1", **kw)
    x_offset *= W.ESIZE[w.conv_dtype]
    lengths = [0, 1, w.conv_width - 1, w.conv_width, 70, 9]
    with DevPool(w, seed=35, random_padding=True) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, xr, cwr = inputs(w, lengths, seed=36)
        rc, q, k, v = run(P, l, w, idx, has, cu, xr, cwr, x_offset)
        assert rc == L.LSC_OK, L.lsc_error_string(rc)
        check(w, P, l, pre, idx, has, cu, xr, cwr, q, k, v)
        assert P.status() == L.LSC_OK


def _padded(kw, i):
    """The shape with 16 x (0..32) bytes of page padding, varying per case."""
    w = workload("s1", **kw)
    w.page_bytes += 16 * ((7 * i + 3) % 33)
    return w


@pytest.mark.parametrize("i", range(len(SHAPES)), ids=[_id(k) for k in SHAPES])
def test_restore_random_shape(lsc, i):
    """Bit-exact against the oracle over the 16-combination rows, random bytes
    in every page's padding (which must survive)."""
    w = _padded(SHAPES[i], i)
    rows = W.combo_rows(w.num_slots, w.block_size, seed=37 + i)
    with DevPool(w, seed=38, random_padding=True) as P:
        pre = {l: P.host[l].copy() for l in P.gdn_layers}
        rc, rep, hs = run_restore(P, rows, w.block_size)
        assert rc == L.LSC_OK
        rc_o, regions, hs_o = oracle_restore(w, P, pre, rows, w.block_size)
        assert rc_o == oracle.OK
        np.testing.assert_array_equal(hs, hs_o)
        for l in P.gdn_layers:
            np.testing.assert_array_equal(P.download(l), regions[l])
        assert P.status() == L.LSC_OK


@pytest.mark.parametrize("i", range(len(SHAPES)), ids=[_id(k) for k in SHAPES])
def test_gather_scatter_random_shape(lsc, i):
    w = _padded(SHAPES[i], i)
    Lo = oracle_layout(w)
    rng = np.random.default_rng(39 + i)
    n = 9
    idx = rng.permutation(w.num_slots)[:n].astype(np.int32)
    idx[4] = -1
    has = (rng.random(n) < 0.7).astype(np.uint8)
    with DevPool(w, seed=40, random_padding=True) as P:
        l = P.gdn_layers[-1]
        pre = P.host[l].copy()
        conv = torch.full((n, Lo["conv_bytes"]), 0x5A, dtype=torch.uint8, device="cuda")
        ssm = torch.full((n, Lo["ssm_bytes"]), 0x5A, dtype=torch.uint8, device="cuda")
        di, dh = dev_(idx), dev_(has)
        assert L.lsc_gather(P.pool, l, di, dh, n, conv, ssm, torch.cuda.current_stream()) == L.LSC_OK
        rc, conv_o, ssm_o = oracle.gather(oracle_pool(w), pre, idx, has)
        assert rc == oracle.OK
        np.testing.assert_array_equal(conv.cpu().numpy(), conv_o)
        np.testing.assert_array_equal(ssm.cpu().numpy(), ssm_o)
        new_conv = torch.from_numpy(rng.integers(0, 256, conv_o.shape, dtype=np.uint8)).cuda()
        new_ssm = torch.from_numpy(rng.integers(0, 256, ssm_o.shape, dtype=np.uint8)).cuda()
        assert L.lsc_scatter(P.pool, l, di, n, new_conv, new_ssm, torch.cuda.current_stream()) == L.LSC_OK
        reg_o = pre.copy()
        assert oracle.scatter(oracle_pool(w), reg_o, idx, new_conv.cpu().numpy(), new_ssm.cpu().numpy()) == oracle.OK
        np.testing.assert_array_equal(P.download(l), reg_o)
        assert P.status() == L.LSC_OK


def dev_(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()
