"""Seeded random shapes for the fused decode and the recurrence against the
oracle: q/k head counts, v heads per q/k head (1, 2, 4, 8), head dims, conv
widths 2..8 and both dtypes of each state, beyond the fixed cases of
test_gpu_parity.py.  The shapes are drawn once from a fixed seed, so a failure
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
from test_gpu_parity import (REC_ALGOS, check_decode, check_recurrent, decode_case, rec_case, run_decode,
                             run_recurrent, workload)

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
