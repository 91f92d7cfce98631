"""The N > 1 host path of bench.py with two gloo ranks on the CPU.

The hot path does not shard: N GPUs run N independent replicas, each on its
own seeded pool and rows, and the job's clock is the slowest rank's.  These
tests run the pieces of that path that need no GPU (rank setup, the
max-over-ranks clock, the whole-job rate, the rank-0-only reference line) as
two processes joined by a gloo process group on 127.0.0.1.
"""
import json
import os
import socket
import sys
import types

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})


def _clock_worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    _env(rank, world, port)
    import torch.distributed as dist
    import bench
    from linear_attention_state_lsc_gb300 import workloads as W
    r, local, wsz = bench.dist_env()
    dist.init_process_group("gloo", init_method="env://")
    elapsed = 1.0 + 0.25 * rank          # rank 1 is the slower replica
    job = bench.max_over_ranks(elapsed, "cpu")
    rate = bench.whole_job_rate(wsz, 1000.0, job)
    rows = W.restore_rows("c1", seed=r)  # each rank's replica draws its own rows
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"env": [r, local, wsz], "job": job, "rate": rate, "live": rows.live.tolist()}, f)


def _reference_worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    _env(rank, world, port)
    out = open(os.path.join(out_dir, f"ref{rank}.txt"), "w")
    sys.stdout = out
    import bench
    # a stand-in sample so that the test exercises the rank logic, not the oracle
    bench.oracle_sample = lambda: ((lambda: None), 10 ** 6, 1, 1)
    import oracle.build
    oracle.build.build = lambda *a, **k: None
    bench.run_reference(types.SimpleNamespace(steps=2, warmup=1))
    out.flush()


def _spawn(fn, tmp_path, world=2):
    port = _free_port()
    mp.spawn(fn, args=(world, port, str(tmp_path)), nprocs=world, join=True)


def test_two_ranks_take_the_slowest_clock(tmp_path):
    _spawn(_clock_worker, tmp_path)
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["env"] == [0, 0, 2] and r1["env"] == [1, 1, 2]
    assert r0["job"] == r1["job"] == 1.25
    # whole job: both ranks' units over the slowest rank's time
    assert r0["rate"] == pytest.approx(2 * 1000.0 / 1.25)
    # the replicas are independent: different seeded rows
    assert r0["live"] != r1["live"]


def test_reference_line_from_rank_zero_only(tmp_path):
    _spawn(_reference_worker, tmp_path)
    lines0 = [l for l in open(tmp_path / "ref0.txt") if l.strip()]
    lines1 = [l for l in open(tmp_path / "ref1.txt") if l.strip()]
    assert lines1 == []
    assert len(lines0) == 1
    d = json.loads(lines0[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_single_rank_clock_is_local():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(1, 7.0, 2.0) == 3.5
    assert np.isclose(bench.whole_job_rate(4, 7.0, 2.0), 14.0)
