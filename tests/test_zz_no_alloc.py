"""GPU: lsc_gdn_recurrent_noalloc -- the chunked resumed-prefill recurrence for
callers that may not allocate device memory at call time (its per-chunk
records go to a scratch array the library keeps on each device instead of a
caller buffer or a stream-ordered allocation).

Checked against lsc_gdn_recurrent (chunked order, library-allocated workspace)
on two pools with the same pre-image, over two calls in a row, so the second
call reuses the scratch array the first one left behind and starts from the
states the first one wrote.  This file is collected last so that a run that
stops at its first failure has run every other test before it."""
import numpy as np
import pytest
import torch

from linear_attention_state_lsc_gb300 import lsc as L
from linear_attention_state_lsc_gb300 import workloads as W

from _gpu import DevPool, dev, tol
from _util import oracle_layout
from test_gpu_parity import rec_case, workload

pytestmark = pytest.mark.gpu


def _call(fn, P, l, w, idx, has, cu, q, k, v, a, b):
    T = int(cu[-1])
    out = torch.full((T, w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
    t = [dev(z) for z in (idx, has, cu, q, k, v, a, b)]
    args = L.recurrent_args(len(idx), w.num_k_heads, T, *t, out, algorithm=L.LSC_RECURRENT_CHUNKED)
    rc = fn(P.pool, l, args, torch.cuda.current_stream())
    torch.cuda.synchronize()
    return rc, out.cpu().numpy()


@pytest.mark.parametrize("name", ["s3", "s2"])  # fp32 and bf16 state, head_k_dim 128
def test_noalloc_matches_the_allocating_call_twice_in_a_row(name):
    w = workload(name)
    lengths = [100, 64, 7, 0, 150][:w.num_slots]
    Lo = oracle_layout(w)
    ssm = slice(Lo["ssm_offset"], Lo["ssm_offset"] + Lo["ssm_bytes"])
    with DevPool(w, seed=41) as A, DevPool(w, seed=41) as B:
        l = A.gdn_layers[0]
        for call in range(2):
            idx, has, cu, q, k, v, a, b = rec_case(w, lengths, seed=42 + call)
            rc_a, out_a = _call(L.lsc_gdn_recurrent, A, l, w, idx, has, cu, q, k, v, a, b)
            rc_b, out_b = _call(L.lsc_gdn_recurrent_noalloc, B, l, w, idx, has, cu, q, k, v, a, b)
            assert rc_a == L.LSC_OK and rc_b == L.LSC_OK, (rc_a, rc_b)
            assert A.status() == L.LSC_OK and B.status() == L.LSC_OK
            t = tol(w.ssm_dtype)
            np.testing.assert_allclose(out_b, out_a, **t)
            ga = A.download(l).reshape(w.num_slots, -1)
            gb = B.download(l).reshape(w.num_slots, -1)
            np.testing.assert_allclose(W.from_dtype_bytes(np.ascontiguousarray(gb[:, ssm]), w.ssm_dtype),
                                       W.from_dtype_bytes(np.ascontiguousarray(ga[:, ssm]), w.ssm_dtype), **t)
            other = np.ones(w.page_bytes, bool)
            other[ssm] = False
            np.testing.assert_array_equal(gb[:, other], ga[:, other])


def test_noalloc_refuses_what_does_not_fit_or_asks_for_a_workspace():
    """A call whose records exceed the scratch array: NO_MEMORY; a caller
    workspace or the token order: INVALID_ARG; head_k_dim 32: UNSUPPORTED.
    Nothing is written in any case."""
    w = workload("s3", num_slots=40)
    with DevPool(w, seed=43) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        # 40 sequences x 1000 tokens: 665 chunk slots x 4 v heads x 33 344 B = 88.7 MB > 64 MiB
        lengths = [1000] * 40
        idx, has, cu, q, k, v, a, b = rec_case(w, lengths, seed=44, pad_seq=False)
        T = int(cu[-1])
        out = torch.full((T, w.num_v_heads, w.head_v_dim), 3.0, device="cuda")
        t = [dev(z) for z in (idx, has, cu, q, k, v, a, b)]
        big = L.recurrent_args(len(idx), w.num_k_heads, T, *t, out, algorithm=L.LSC_RECURRENT_CHUNKED)
        rc, need = L.lsc_gdn_recurrent_workspace_bytes(P.pool, big)
        assert rc == L.LSC_OK and need > 64 << 20
        assert L.lsc_gdn_recurrent_noalloc(P.pool, l, big, torch.cuda.current_stream()) == L.LSC_ERR_NO_MEMORY
        small_idx, small_has, cu2, q2, k2, v2, a2, b2 = rec_case(w, [10], seed=45, pad_seq=False)
        t2 = [dev(z) for z in (small_idx, small_has, cu2, q2, k2, v2, a2, b2)]
        ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
        with_ws = L.recurrent_args(1, w.num_k_heads, 10, *t2, out, algorithm=L.LSC_RECURRENT_CHUNKED,
                                   workspace=ws, workspace_bytes=ws.numel())
        assert L.lsc_gdn_recurrent_noalloc(P.pool, l, with_ws, torch.cuda.current_stream()) == L.LSC_ERR_INVALID_ARG
        token = L.recurrent_args(1, w.num_k_heads, 10, *t2, out, algorithm=L.LSC_RECURRENT_TOKEN)
        assert L.lsc_gdn_recurrent_noalloc(P.pool, l, token, torch.cuda.current_stream()) == L.LSC_ERR_INVALID_ARG
        torch.cuda.synchronize()
        np.testing.assert_array_equal(P.download(l), pre)
        assert (out.cpu().numpy() == 3.0).all()
    w32 = workload("s1")
    with DevPool(w32, seed=46) as P:
        l = P.gdn_layers[0]
        idx, has, cu, q, k, v, a, b = rec_case(w32, [5], seed=47, pad_seq=False)
        rc, _ = _call(L.lsc_gdn_recurrent_noalloc, P, l, w32, idx, has, cu, q, k, v, a, b)
        assert rc == L.LSC_ERR_UNSUPPORTED
