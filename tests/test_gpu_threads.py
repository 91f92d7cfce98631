"""Two pools driven from two host threads at once, each on its own stream.

The launchers keep a kernel's dynamic shared-memory limit, the opt-in limit
of a block and the copy kernels' occupancy per device, behind atomics; these
tests make two threads launch the decode, the recurrence and the restore
concurrently -- in this process, and in a fresh process where the threads'
calls are the first launches of each kernel -- and check both threads'
results against the oracle.  (One GPU here: the per-device keying itself is
exercised only for device 0.)
"""
import os
import subprocess
import sys
import threading

import numpy as np
import pytest
import torch

from linear_attention_state_lsc_gb300 import lsc as L

from _gpu import DevPool, conv_bytes_dev, dev
from test_gpu_parity import check_decode, check_recurrent, decode_case, oracle_restore, rec_case, workload

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _decode_job(w, seed):
    """A pool, inputs and a closure that enqueues one decode on `stream`."""
    P = DevPool(w, seed=seed, random_padding=True)
    l = P.gdn_layers[0]
    pre = P.host[l].copy()
    idx, has, x, cw, a, b = decode_case(w, seed=seed, n=min(w.num_slots, 12))
    n = len(idx)
    out = torch.full((n, w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
    t = [dev(idx), dev(has), conv_bytes_dev(x, w.conv_dtype), conv_bytes_dev(cw, w.conv_dtype), dev(a), dev(b)]
    args = L.decode_args(n, w.num_k_heads, t[0], t[1], t[2], t[3], t[4], t[5], out)

    def launch(stream):
        return L.lsc_gdn_decode(P.pool, l, args, stream)

    def check():
        check_decode(w, P, l, pre, idx, has, x, cw, a, b, out.cpu().numpy())
        assert P.status() == L.LSC_OK

    return P, launch, check, t


def _recurrent_job(w, seed, algorithm):
    P = DevPool(w, seed=seed)
    l = P.gdn_layers[0]
    pre = P.host[l].copy()
    idx, has, cu, q, k, v, a, b = rec_case(w, [33, 17, 5], seed=seed, pad_seq=False)
    T = int(cu[-1])
    out = torch.full((T, w.num_v_heads, w.head_v_dim), float("nan"), device="cuda")
    t = [dev(z) for z in (idx, has, cu, q, k, v, a, b)]
    args = L.recurrent_args(len(idx), w.num_k_heads, T, *t, out, algorithm=algorithm)

    def launch(stream):
        return L.lsc_gdn_recurrent(P.pool, l, args, stream)

    def check():
        check_recurrent(w, P, l, pre, idx, has, cu, q, k, v, a, b, out.cpu().numpy())
        assert P.status() == L.LSC_OK

    return P, launch, check, t


def _restore_job(w, seed):
    from linear_attention_state_lsc_gb300 import workloads as W
    P = DevPool(w, seed=seed)
    rows = W.combo_rows(w.num_slots, w.block_size, seed=seed)
    pre = {l: P.host[l].copy() for l in P.gdn_layers}
    hs = dev(rows.hs_prefill)
    ops = L.ops_array(rows.live, rows.src, rows.restore_hash, rows.save_hash, rows.save_slot)

    def launch(stream):
        rc, _ = L.lsc_restore(P.pool, ops, rows.nkv, w.block_size, rows.initialized, hs, stream, None)
        return rc

    def check():
        _, regions, hs_o = oracle_restore(w, P, pre, rows, w.block_size)
        np.testing.assert_array_equal(hs.cpu().numpy(), hs_o)
        for l in P.gdn_layers:
            np.testing.assert_array_equal(P.download(l), regions[l])

    return P, launch, check, hs


def run_concurrently(jobs, rounds=1):
    """Each job's launch runs on its own host thread and stream; the threads
    start together (a barrier) and each waits for its own stream."""
    streams = [torch.cuda.Stream() for _ in jobs]
    torch.cuda.synchronize()
    start = threading.Barrier(len(jobs))
    rcs = [None] * len(jobs)

    def worker(j):
        start.wait()
        codes = []
        for _ in range(rounds):
            codes.append(jobs[j][1](streams[j]))
        streams[j].synchronize()
        rcs[j] = codes

    th = [threading.Thread(target=worker, args=(j,)) for j in range(len(jobs))]
    for t in th:
        t.start()
    for t in th:
        t.join()
    torch.cuda.synchronize()
    return rcs


def _all_jobs():
    return [
        _decode_job(workload("s3"), seed=31),                     # fp32 state, dk 128
        _decode_job(workload("s2"), seed=32),                     # bf16 state, dk 128
        _recurrent_job(workload("s3"), 33, L.LSC_RECURRENT_TOKEN),
        _recurrent_job(workload("s3"), 34, L.LSC_RECURRENT_CHUNKED),
        _recurrent_job(workload("s1"), 35, L.LSC_RECURRENT_TOKEN),  # dk 32: the other token kernel
        _restore_job(workload("s4", num_slots=24), seed=36),
    ]


def test_two_threads_two_pools_decode_recurrence_restore(lsc):
    jobs = _all_jobs()
    try:
        rcs = run_concurrently(jobs)
        assert all(c == [L.LSC_OK] for c in rcs), rcs
        for j in jobs:
            j[2]()
    finally:
        for j in jobs:
            j[0].close()


def _fresh_process_main():
    """Body of the fresh-process test: the threads' calls are the first
    launches of every kernel in this process."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    L.load()
    jobs = _all_jobs()
    rcs = run_concurrently(jobs)
    assert all(c == [L.LSC_OK] for c in rcs), rcs
    for j in jobs:
        j[2]()
    for j in jobs:
        j[0].close()
    print("FRESH-OK")


def test_first_launches_from_two_threads_in_a_fresh_process(lsc):
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([ROOT, os.path.join(ROOT, "tests"), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, "-c", "import test_gpu_threads as t; t._fresh_process_main()"],
                       cwd=os.path.join(ROOT, "tests"), env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "FRESH-OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
