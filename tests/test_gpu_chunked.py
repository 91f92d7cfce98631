"""GPU: the chunked order of the resumed-prefill recurrence (64-token chunks on
the tensor cores) -- its workspace through the C ABI (size query, a caller's
buffer, the library's stream-ordered one, rejected buffers), AUTO selecting
it, and chunk-boundary and many-chunk cases against the CPU oracle."""
import numpy as np
import pytest
import torch

from linear_attention_state_lsc_gb300 import lsc as L

from _gpu import DevPool, dev
from test_gpu_parity import check_recurrent, rec_case, run_recurrent, workload

pytestmark = pytest.mark.gpu

REC_BYTES = 33344  # one record: T' and B (64 x 64 fp32 each), E, F, e_last


def _args(w, idx, has, cu, q, k, v, a, b, out, algorithm, workspace=None, workspace_bytes=0):
    T = int(cu[-1])
    t = [dev(z) for z in (idx, has, cu, q, k, v, a, b)]
    return L.recurrent_args(len(idx), w.num_k_heads, T, *t, out, algorithm=algorithm, workspace=workspace,
                            workspace_bytes=workspace_bytes), t


def test_workspace_query():
    """0 for the token order; one record per (chunk slot, v head) otherwise,
    with (T + 63) / 64 + n_seq chunk slots; AUTO follows head_k_dim."""
    for name, dk128 in (("s3", True), ("s1", False)):
        w = workload(name)
        with DevPool(w) as P:
            idx, has, cu, q, k, v, a, b = rec_case(w, [70, 1, 0, 64], seed=3)
            T = int(cu[-1])
            out = torch.empty((T, w.num_v_heads, w.head_v_dim), device="cuda")
            want = ((T + 63) // 64 + len(idx)) * w.num_v_heads * REC_BYTES
            for algo, expect in ((L.LSC_RECURRENT_TOKEN, 0), (L.LSC_RECURRENT_CHUNKED, want),
                                 (L.LSC_RECURRENT_AUTO, want if dk128 else 0)):
                args, _ = _args(w, idx, has, cu, q, k, v, a, b, out, algo)
                rc, n = L.lsc_gdn_recurrent_workspace_bytes(P.pool, args)
                assert rc == L.LSC_OK and n == expect, (name, algo, n, expect)


@pytest.mark.parametrize("name", ["s3", "s2"])  # fp32 and bf16 state
def test_caller_workspace_matches_library_workspace(name):
    """A caller's workspace (filled with NaN first) gives the same bytes as the
    library's stream-ordered one, and both match the oracle."""
    w = workload(name)
    lengths = [129, 64, 1, 0, 200, 63][:w.num_slots]
    results = []
    for caller in (False, True):
        with DevPool(w, seed=31) as P:
            l = P.gdn_layers[0]
            pre = P.host[l].copy()
            idx, has, cu, q, k, v, a, b = rec_case(w, lengths, seed=32)
            T = int(cu[-1])
            out = torch.full((T, w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
            args, _ = _args(w, idx, has, cu, q, k, v, a, b, out, L.LSC_RECURRENT_CHUNKED)
            ws = None
            if caller:
                rc, n = L.lsc_gdn_recurrent_workspace_bytes(P.pool, args)
                assert rc == L.LSC_OK
                ws = torch.full((n // 4,), float("nan"), device="cuda")
                args, _t = _args(w, idx, has, cu, q, k, v, a, b, out, L.LSC_RECURRENT_CHUNKED, ws, n)
            assert L.lsc_gdn_recurrent(P.pool, l, args, torch.cuda.current_stream()) == L.LSC_OK
            torch.cuda.synchronize()
            assert P.status() == L.LSC_OK
            got_out = out.cpu().numpy()
            check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, got_out)
            results.append((got_out.copy(), P.download(l).copy()))
    np.testing.assert_array_equal(results[0][0], results[1][0])
    np.testing.assert_array_equal(results[0][1], results[1][1])


def test_workspace_rejected_before_any_work():
    """Too small: INVALID_ARG; not 16-byte aligned: MISALIGNED; nothing written."""
    w = workload("s3")
    with DevPool(w, seed=33) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, q, k, v, a, b = rec_case(w, [80, 5], seed=34, pad_seq=False)
        T = int(cu[-1])
        out = torch.full((T, w.num_v_heads, w.head_v_dim), 7.0, device="cuda")
        args, _ = _args(w, idx, has, cu, q, k, v, a, b, out, L.LSC_RECURRENT_CHUNKED)
        rc, n = L.lsc_gdn_recurrent_workspace_bytes(P.pool, args)
        ws = torch.zeros(n // 4 + 16, device="cuda")
        for ptr, nbytes, want in ((ws.data_ptr(), n - 16, L.LSC_ERR_INVALID_ARG),
                                  (ws.data_ptr() + 4, n, L.LSC_ERR_MISALIGNED)):
            bad, _t = _args(w, idx, has, cu, q, k, v, a, b, out, L.LSC_RECURRENT_CHUNKED, ptr, nbytes)
            assert L.lsc_gdn_recurrent(P.pool, l, bad, torch.cuda.current_stream()) == want
        torch.cuda.synchronize()
        np.testing.assert_array_equal(P.download(l), pre)
        assert (out.cpu().numpy() == 7.0).all()


def test_auto_takes_the_chunked_order_at_head_k_dim_128():
    """AUTO at head_k_dim 128 runs the chunked order: bit-identical to an
    explicit CHUNKED call, and within tolerance of the oracle."""
    w = workload("s3")
    lengths = [64, 65, 127, 3]
    outs = []
    for algo in (L.LSC_RECURRENT_AUTO, L.LSC_RECURRENT_CHUNKED):
        with DevPool(w, seed=35) as P:
            l = P.gdn_layers[0]
            pre = P.host[l].copy()
            idx, has, cu, q, k, v, a, b = rec_case(w, lengths, seed=36)
            rc, out = run_recurrent(P, l, w, idx, has, cu, q, k, v, a, b, algo)
            assert rc == L.LSC_OK
            check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out)
            outs.append((out, P.download(l)))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_chunked_many_chunks_and_every_tail():
    """Sequences of 1..130 tokens and 1000 tokens (16 chunks), warm and cold,
    beside one another: every chunk-tail length, the longest chain."""
    w = workload("s3", num_slots=12)
    lengths = [1, 2, 31, 32, 33, 63, 64, 65, 127, 128, 130, 1000]
    with DevPool(w, seed=37) as P:
        l = P.gdn_layers[0]
        pre = P.host[l].copy()
        idx, has, cu, q, k, v, a, b = rec_case(w, lengths, seed=38, pad_seq=False)
        rc, out = run_recurrent(P, l, w, idx, has, cu, q, k, v, a, b, L.LSC_RECURRENT_CHUNKED)
        assert rc == L.LSC_OK
        check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out)
        assert P.status() == L.LSC_OK
