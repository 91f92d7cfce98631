#!/usr/bin/env python
"""Benchmark of the linear-state prefix cache hot path on GB300.

One step (workload "c1-serving-step": 36 GDN + 12 attention layers, 256 slots,
conv [8192, 3] bf16, ssm [32, 128, 128] fp32, 4 KiB-rounded pages):
  1. lsc_restore of 64 rows, all hits, on a prepare stream, signalling an event;
  2. the forward stream waits on the event, then runs lsc_gdn_decode for the 64
     restored rows on each of the 36 GDN layers (one decode token).
value = algorithmic HBM bytes of the step / step time (GB/s); rows/s beside it.
Also measured in the same run (rank 0, N = 1): the 256-row bf16 decode layer,
the 512-row restore storm and the token-by-token resume prefill.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lsc|reference] [--no-parts]
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "restore & gather→GDN-step→scatter HBM GB/s (fraction of GB300 peak); rows/s"
UNIT = "GB/s"
FALLBACK_HBM = 6800.0
DECODE_FLAGS = 1  # LSC_DECODE_EARLY_STATE


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["lsc", "reference"], default="lsc")
    ap.add_argument("--no-parts", action="store_true", help="headline step only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--ncu-case", choices=sorted(NCU_CASES), default=None,
                    help="run only one kernel on a reduced pool (2 GDN layers), for profiler captures")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM, "fallback"


def measured(key, default):
    """One figure of MEASURED_PEAKS.json, or `default` when the file is absent."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if key in d:
            return float(d[key])
    return default


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(x, device):
    """The largest of every rank's x (an elapsed time): the job's clock is its
    slowest replica.  With one rank, x itself."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, elapsed):
    """Units all ranks processed per second of the slowest rank's clock
    (replicas: every rank processes the same number of units)."""
    return world * units_per_rank / elapsed


# ---------------------------------------------------------------- clocks

class Clocks:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.window = None  # (start, end) host time.time() of the timed region

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self, t_start, t_end):
        self.window = (t_start, t_end)

    @staticmethod
    def _ts(text):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        samples = []  # (time, sm, max, reasons)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                sm, mx = float(f[2]), float(f[3])
            except ValueError:
                continue
            samples.append((self._ts(f[0]), sm, mx, {n for n, v in zip(names, f[6:10]) if v.lower() == "active"}))
        os.unlink(self.path)
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        timed = []
        if self.window:
            a, b = self.window
            timed = [x for x in samples if x[0] is not None and a <= x[0] <= b]
        top = max(x[1] for x in samples)
        loaded = [x for x in samples if x[1] >= 0.5 * top] or samples
        use = timed or loaded
        reasons = set().union(*(x[3] for x in use))
        return {"sm_mhz": statistics.median(x[1] for x in use), "sm_max_mhz": max(x[2] for x in samples),
                "reasons": sorted(reasons), "samples": len(samples), "samples_in_timed_region": len(timed),
                "sm_mhz_basis": "median of the samples inside the timed region" if timed else
                                "median of the samples under load (none fell inside the timed region)",
                "sample_period_ms": 50}


# ---------------------------------------------------------------- pools

def make_pool(L, W, w, seed):
    """Allocate and fill a pool on the current device; returns (buf, pool, views)."""
    import torch
    kinds = [L.LSC_LAYER_GDN if k == W.GDN else L.LSC_LAYER_ATTENTION for k in w.layers]
    dt = {W.F32: L.LSC_F32, W.BF16: L.LSC_BF16}
    desc = L.make_pool_desc(kinds, w.num_slots, w.conv_dim, w.conv_width, dt[w.conv_dtype], w.num_v_heads,
                            w.head_v_dim, w.head_k_dim, dt[w.ssm_dtype], w.page_bytes)
    nbytes = L.lsc_pool_required_bytes(desc)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    rc, pool = L.lsc_pool_create(desc, buf, nbytes)
    if rc != L.LSC_OK:
        raise RuntimeError(L.lsc_error_string(rc))
    views = {}
    for l in w.gdn_layers:
        rc, v = L.lsc_pool_layer_view(pool, l)
        assert rc == L.LSC_OK
        views[l] = v
        off = v.region - buf.data_ptr()
        fill = [(0, v.conv_bytes // W.ESIZE[w.conv_dtype], w.conv_dtype),
                (v.ssm_offset_bytes, v.ssm_bytes // W.ESIZE[w.ssm_dtype], w.ssm_dtype)]
        W.fill_region_device(buf[off:off + v.region_bytes], w.num_slots, w.page_bytes, fill, w.pad_byte,
                             seed * 1000 + l)
    torch.cuda.synchronize()
    return buf, pool, views


def restore_bytes(view, n_hit, n_gdn, n_rows):
    """Algorithmic bytes of a restore: read + write of both views per (hit, layer),
    plus one has_initial_state byte per written row."""
    return 2 * n_hit * n_gdn * (view.conv_bytes + view.ssm_bytes) + n_rows


def decode_bytes(view, w, n):
    """Algorithmic bytes of one decode launch over n rows: conv + ssm state read and
    written, x, alpha, beta, out, idx, has_init per row; the conv weights once."""
    es = 2 if w.conv_dtype == "bf16" else 4
    per_row = (2 * (view.conv_bytes + view.ssm_bytes) + w.conv_dim * es + 2 * w.num_v_heads * 4
               + w.num_v_heads * w.head_v_dim * 4 + 4 + 1)
    return n * per_row + w.conv_dim * w.conv_width * es


def kernel_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["source_sha"]:
        return None
    return d["bytes_per_launch"]


# ---------------------------------------------------------------- our arm

def serving_step_inputs(W, w, rows, seed=0):
    n = len(rows.live)
    xs, abs_ = [], []
    for l in w.gdn_layers:
        x, cw, a, b = W.decode_inputs(w, n, seed=seed, layer=l)
        xs.append((x, cw))
        abs_.append((a, b))
    return xs, abs_


def run_lsc(args):
    import torch
    import torch.distributed as dist
    from linear_attention_state_lsc_gb300 import lsc as L
    from linear_attention_state_lsc_gb300 import workloads as W

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    L.load()
    hbm_peak, peak_src = peaks()

    w = W.get("c1")
    rows = W.restore_rows("c1", seed=rank)  # each rank is an independent replica
    buf, pool, views = make_pool(L, W, w, seed=rank)
    v0 = views[w.gdn_layers[0]]
    n = len(rows.live)
    n_gdn = len(w.gdn_layers)
    ops = L.ops_array(rows.live, rows.src, rows.restore_hash, rows.save_hash, rows.save_slot)

    # device-resident inputs of the step
    bf = torch.bfloat16
    idx = torch.from_numpy(rows.live.astype(np.int32)).cuda()
    hs = torch.empty(n, dtype=torch.uint8, device="cuda")
    hs_prefill = torch.from_numpy(rows.hs_prefill.copy()).cuda()
    xs, abs_ = serving_step_inputs(W, w, rows, seed=rank)
    X = torch.stack([torch.from_numpy(x) for x, _ in xs]).to(bf).cuda()          # [36, n, C]
    CW = torch.stack([torch.from_numpy(cw) for _, cw in xs]).to(bf).cuda()       # [36, C, W]
    A = torch.stack([torch.from_numpy(a) for a, _ in abs_]).cuda()               # [36, n, Hv]
    B = torch.stack([torch.from_numpy(b) for _, b in abs_]).cuda()
    OUT = torch.empty((n_gdn, n, w.num_v_heads, w.head_v_dim), device="cuda")
    # each decode launch may stream its layer's first state tiles while the
    # previous layer's launch finishes: no launch of the chain writes another
    # layer's state, and the first one follows the restore's event
    dargs = [L.decode_args(n, w.num_k_heads, idx, hs, X[g], CW[g], A[g], B[g], OUT[g], DECODE_FLAGS)
             for g in range(n_gdn)]

    prep = torch.cuda.Stream()
    fwd = torch.cuda.current_stream()
    ev_done = torch.cuda.Event()
    ev_done.record(fwd)
    torch.cuda.synchronize()
    ev = {k: [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] for k in ("r0", "r1", "d0", "d1")}

    def step(i=None):
        hs.copy_(hs_prefill)
        prep.wait_stream(fwd)
        if i is not None:
            ev["r0"][i].record(prep)
        rc, _ = L.lsc_restore(pool, ops, rows.nkv, rows.block_size, rows.initialized, hs, prep, ev_done)
        assert rc == L.LSC_OK, L.lsc_error_string(rc)
        if i is not None:
            ev["r1"][i].record(prep)
        fwd.wait_event(ev_done)
        if i is not None:
            ev["d0"][i].record(fwd)
        for g, l in enumerate(w.gdn_layers):
            rc = L.lsc_gdn_decode(pool, l, dargs[g], fwd)
            assert rc == L.LSC_OK, L.lsc_error_string(rc)
        if i is not None:
            ev["d1"][i].record(fwd)

    # the clock sampler runs from before the warm-up to after the timed region
    # (all under load), so short timed regions still get samples
    clocks = Clocks(local)
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    wall0 = time.time()
    t0.record(fwd)
    for i in range(args.steps):
        step(i)
    t1.record(fwd)
    torch.cuda.synchronize()
    clocks.mark(wall0, time.time())
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    ck = clocks.stop()
    ck["window"] = "sampler ran over the warm-up, the timed region and trailing untimed steps"
    elapsed = max_over_ranks(t0.elapsed_time(t1) / 1e3, "cuda")
    if world > 1:
        dist.barrier()
    assert L.lsc_pool_status(pool, fwd) == L.LSC_OK

    rb = restore_bytes(v0, n, n_gdn, n)
    db = n_gdn * decode_bytes(v0, w, n)
    step_bytes = rb + db
    t_restore = statistics.mean(ev["r0"][i].elapsed_time(ev["r1"][i]) for i in range(args.steps)) / 1e3
    t_decode = statistics.mean(ev["d0"][i].elapsed_time(ev["d1"][i]) for i in range(args.steps)) / 1e3 / n_gdn
    restore_gbs = rb / t_restore / 1e9
    decode_gbs = decode_bytes(v0, w, n) / t_decode / 1e9
    value = whole_job_rate(world, step_bytes * args.steps, elapsed) / 1e9
    rows_per_s = whole_job_rate(world, n * args.steps, elapsed)

    roof_restore = {"bound": "hbm", "kernel": "restore_bulk_kernel", "achieved": round(restore_gbs, 1),
                    "peak": hbm_peak, "unit": "GB/s", "frac": round(restore_gbs / hbm_peak, 4),
                    "traffic": kernel_traffic("restore_bulk_kernel"), "bytes_per_launch": rb,
                    "launch_ms": round(t_restore * 1e3, 4), "peak_source": peak_src}
    roof_decode = {"bound": "hbm", "kernel": "decode_kernel<128,f32>", "achieved": round(decode_gbs, 1),
                   "peak": hbm_peak, "unit": "GB/s", "frac": round(decode_gbs / hbm_peak, 4),
                   "traffic": kernel_traffic("decode_kernel<128,f32,2>"), "bytes_per_launch": decode_bytes(v0, w, n),
                   "launch_ms": round(t_decode * 1e3, 4), "peak_source": peak_src}
    dominant = roof_restore if t_restore >= t_decode * n_gdn else roof_decode

    # end to end through the public API with host buffers: per step, H2D of the
    # step's inputs from pinned memory, the calls, D2H of the outputs
    e2e = e2e_serving(args, L, torch, pool, w, rows, ops, n, n_gdn, X, CW, A, B, step_bytes, world)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f32", "data": "synthetic",
        "config": {"workload": "c1-serving-step", "layers": "36 GDN + 12 attention", "num_slots": w.num_slots,
                   "rows": n, "restore": "64 rows all hits x 36 GDN layers",
                   "decode": "1 token x 64 restored rows x 36 GDN layers",
                   "decode_flags": "LSC_DECODE_EARLY_STATE" if DECODE_FLAGS else "0",
                   "conv": "[8192,3] bf16", "ssm": "[32,128,128] f32", "page_bytes": w.page_bytes,
                   "l2": "inputs larger than L2 (9.9 GB restore, 9.9 GB decode per step)",
                   "parallelism": f"replicas x{world}"},
        "rows_per_s": round(rows_per_s, 1),
        "step_bytes": step_bytes,
        "roofline": dominant,
        "roofline_other": roof_decode if dominant is roof_restore else roof_restore,
        "clocks": ck,
        "e2e": e2e,
        "gpu_launches": args.steps * (1 + n_gdn),
    }
    L.lsc_pool_destroy(pool)
    del buf, X, OUT
    torch.cuda.empty_cache()

    if rank == 0 and world == 1 and not args.no_parts:
        line["parts"] = measure_parts(L, W, torch, hbm_peak)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(budget_s=12.0)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def e2e_serving(args, L, torch, pool, w, rows, ops, n, n_gdn, X, CW, A, B, step_bytes, world):
    hx = X.cpu().pin_memory()
    ha = A.cpu().pin_memory()
    hb = B.cpu().pin_memory()
    hhs = torch.from_numpy(rows.hs_prefill.copy()).pin_memory()
    hidx = torch.from_numpy(rows.live.astype(np.int32)).pin_memory()
    hout = torch.empty((n_gdn, n, w.num_v_heads, w.head_v_dim), pin_memory=True)
    dx, da, db = torch.empty_like(X), torch.empty_like(A), torch.empty_like(B)
    dhs = torch.empty(n, dtype=torch.uint8, device="cuda")
    didx = torch.empty(n, dtype=torch.int32, device="cuda")
    dout = torch.empty((n_gdn, n, w.num_v_heads, w.head_v_dim), device="cuda")
    dargs = [L.decode_args(n, w.num_k_heads, didx, dhs, dx[g], CW[g], da[g], db[g], dout[g], DECODE_FLAGS)
             for g in range(n_gdn)]
    prep = torch.cuda.Stream()
    d2h_stream = torch.cuda.Stream()
    fwd = torch.cuda.current_stream()
    evd = torch.cuda.Event()
    evd.record(fwd)
    ev_layer = [torch.cuda.Event() for _ in range(n_gdn)]
    h2d = hx.numel() * hx.element_size() + ha.numel() * 4 + hb.numel() * 4 + n + 4 * n
    d2h = hout.numel() * 4

    # The step as a serving loop would issue it: the restore's small inputs go
    # up on the prepare stream ahead of the restore, the decode inputs go up on
    # the forward stream while the restore runs, and each layer's output comes
    # back on a copy stream while the next layers decode.
    def step():
        prep.wait_stream(fwd)         # the previous step's decodes are done with the slots
        fwd.wait_stream(d2h_stream)   # ... and its outputs have left dout
        with torch.cuda.stream(prep):
            dhs.copy_(hhs, non_blocking=True)
            didx.copy_(hidx, non_blocking=True)
        rc, _ = L.lsc_restore(pool, ops, rows.nkv, rows.block_size, rows.initialized, dhs, prep, evd)
        assert rc == L.LSC_OK
        dx.copy_(hx, non_blocking=True)
        da.copy_(ha, non_blocking=True)
        db.copy_(hb, non_blocking=True)
        fwd.wait_event(evd)
        for g, l in enumerate(w.gdn_layers):
            assert L.lsc_gdn_decode(pool, l, dargs[g], fwd) == L.LSC_OK
            ev_layer[g].record(fwd)
            d2h_stream.wait_event(ev_layer[g])
            with torch.cuda.stream(d2h_stream):
                hout[g].copy_(dout[g], non_blocking=True)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    el = max_over_ranks(time.perf_counter() - t, "cuda")
    return {"value": round(whole_job_rate(world, step_bytes * args.steps, el) / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(el / args.steps * 1e3, 4), "clock": "host wall clock",
            "overlap": "restore inputs on the prepare stream, decode inputs H2D during the restore, per-layer D2H on a copy stream"}


def measure_parts(L, W, torch, hbm_peak, reps=5):
    parts = {}
    fwd = torch.cuda.current_stream()

    def timed(fn, k):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize()
        e0.record(fwd)
        for _ in range(k):
            fn()
        e1.record(fwd)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / k

    # context, not a target: the pages' own restore mechanism on c1 ([XN] §4.3),
    # per hit row and GDN layer a torch copy_ of the conv slot and a
    # narrow().copy_() of the ssm slot, enqueued on a prepare stream; beside it
    # the persistent restore launch on the same pool and rows
    w = W.get("c1")
    buf, pool, views = make_pool(L, W, w, seed=0)
    rows = W.restore_rows("c1", seed=0)
    hits = [(int(d), int(s)) for d, s in zip(rows.live, rows.src) if s >= 0]
    tviews = []
    for l in w.gdn_layers:
        v = views[l]
        pages = buf[v.region - buf.data_ptr():][:v.region_bytes].view(w.num_slots, w.page_bytes)
        conv = pages[:, :v.conv_bytes].view(torch.bfloat16)
        ssm = pages[:, v.ssm_offset_bytes:v.ssm_offset_bytes + v.ssm_bytes].view(torch.float32)
        tviews.append((conv, ssm))
    prep = torch.cuda.Stream()

    def torch_loop():
        with torch.cuda.stream(prep):
            for conv, ssm in tviews:
                for d, s_ in hits:
                    conv[d].copy_(conv[s_])
                    ssm.narrow(0, d, 1).copy_(ssm.narrow(0, s_, 1))

    def timed_on(stream, fn, k):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / k

    t_loop = timed_on(prep, torch_loop, 3)
    ops = L.ops_array(rows.live, rows.src, rows.restore_hash, rows.save_hash, rows.save_slot)
    hs = torch.empty(len(rows.live), dtype=torch.uint8, device="cuda")

    def lsc_call():
        rc, _ = L.lsc_restore(pool, ops, rows.nkv, rows.block_size, rows.initialized, hs, prep, None)
        assert rc == L.LSC_OK

    t_lsc = timed_on(prep, lsc_call, 3)
    v0 = views[w.gdn_layers[0]]
    nb = 2 * len(hits) * len(w.gdn_layers) * (v0.conv_bytes + v0.ssm_bytes)
    parts["restore_torch_loop_c1"] = {
        "workload": f"c1: {len(hits)} hit rows x {len(w.gdn_layers)} GDN layers, the pages' loop of torch copies "
                    f"({2 * len(hits) * len(w.gdn_layers)} copy_ calls per restore)",
        "kind": "context (the pages' mechanism), not a target", "launch_ms": round(t_loop * 1e3, 3),
        "GB/s": round(nb / t_loop / 1e9, 1), "frac": round(nb / t_loop / 1e9 / hbm_peak, 4),
        "restore_kernel_ms": round(t_lsc * 1e3, 3), "speedup_of_restore_kernel": round(t_loop / t_lsc, 2)}
    # the restore's two copy forms on the same pool and rows: 1-D TMA bulk
    # copies through shared memory (the default here) and 16-byte vectors
    # through registers (LSC_RESTORE_COPY=vector)
    t_bulk = timed_on(prep, lsc_call, 10)
    os.environ["LSC_RESTORE_COPY"] = "vector"
    try:
        t_vec = timed_on(prep, lsc_call, 10)
    finally:
        del os.environ["LSC_RESTORE_COPY"]
    parts["restore_c1_copy_forms"] = {
        "workload": f"c1: {len(hits)} hit rows x {len(w.gdn_layers)} GDN layers (9.89 GB), the serving step's restore",
        "bulk": {"kernel": "restore_bulk_kernel (the default: cp.async.bulk global -> shared -> global, "
                           "3 x 32 KiB stages, 2 CTAs per SM)",
                 "launch_ms": round(t_bulk * 1e3, 4), "GB/s": round(nb / t_bulk / 1e9, 1),
                 "frac": round(nb / t_bulk / 1e9 / hbm_peak, 4)},
        "vector": {"kernel": "restore_kernel (16-byte vectors, LSC_RESTORE_COPY=vector)",
                   "launch_ms": round(t_vec * 1e3, 4), "GB/s": round(nb / t_vec / 1e9, 1),
                   "frac": round(nb / t_vec / 1e9 / hbm_peak, 4)}}
    L.lsc_pool_destroy(pool)
    del buf, tviews, hs
    torch.cuda.empty_cache()

    # the serving step's decode chain (64 restored rows x 36 GDN layers, fp32
    # state) with and without the early state start, on the same pool and rows
    w = W.get("c1")
    rows = W.restore_rows("c1", seed=0)
    buf, pool, views = make_pool(L, W, w, seed=0)
    n = len(rows.live)
    idx = torch.from_numpy(rows.live.astype(np.int32)).cuda()
    has = torch.ones(n, dtype=torch.uint8, device="cuda")
    xs, abs_ = serving_step_inputs(W, w, rows)
    bf = torch.bfloat16
    X = torch.stack([torch.from_numpy(x) for x, _ in xs]).to(bf).cuda()
    CW = torch.stack([torch.from_numpy(cw) for _, cw in xs]).to(bf).cuda()
    A = torch.stack([torch.from_numpy(a) for a, _ in abs_]).cuda()
    B = torch.stack([torch.from_numpy(b) for _, b in abs_]).cuda()
    OUT = torch.empty((len(w.gdn_layers), n, w.num_v_heads, w.head_v_dim), device="cuda")
    v = views[w.gdn_layers[0]]
    bytes_ = decode_bytes(v, w, n)
    chain = {}
    for flags, key in ((0, "plain"), (1, "early_state")):
        dargs = [L.decode_args(n, w.num_k_heads, idx, has, X[g], CW[g], A[g], B[g], OUT[g], flags)
                 for g in range(len(w.gdn_layers))]

        def dec_chain():
            for g, l in enumerate(w.gdn_layers):
                assert L.lsc_gdn_decode(pool, l, dargs[g], fwd) == L.LSC_OK

        t = timed(dec_chain, 20) / len(w.gdn_layers)
        chain[key] = {"launch_ms": round(t * 1e3, 4), "GB/s": round(bytes_ / t / 1e9, 1),
                      "frac": round(bytes_ / t / 1e9 / hbm_peak, 4)}
    L.lsc_pool_destroy(pool)
    del buf, X, CW, A, B, OUT
    torch.cuda.empty_cache()
    # yardstick: the peak's own method (a torch copy) at the decode's launch
    # size -- 36 back-to-back copies of half the launch's bytes each, distinct
    # buffers per layer (10 GB in all, larger than L2)
    half = bytes_ // 2 // 16 * 16
    srcs = [torch.empty(half, dtype=torch.uint8, device="cuda") for _ in w.gdn_layers]
    dsts = [torch.empty(half, dtype=torch.uint8, device="cuda") for _ in w.gdn_layers]
    for t_ in srcs:
        t_.fill_(1)

    def copy_chain():
        for a_, b_ in zip(dsts, srcs):
            a_.copy_(b_)

    t = timed(copy_chain, 20) / len(w.gdn_layers)
    del srcs, dsts
    torch.cuda.empty_cache()
    parts["decode_c1_chain"] = {"workload": "c1 pool: 64 rows x 36 GDN layers, ssm f32, one launch per layer, "
                                            "layers back to back (the serving step's decode without its restore)",
                                "kernel": "decode_kernel<128,f32>", "bytes_per_launch": bytes_,
                                "plain": chain["plain"],
                                "early_state": chain["early_state"] | {
                                    "flags": "LSC_DECODE_EARLY_STATE: rows and first state tiles read before the "
                                             "wait for the previous layer's launch"},
                                "copy_yardstick": {"what": "torch copy_ (the measured peak's method) of the same "
                                                           "bytes per launch, 36 back to back", "launch_ms":
                                                   round(t * 1e3, 4), "GB/s": round(2 * half / t / 1e9, 1),
                                                   "frac": round(2 * half / t / 1e9 / hbm_peak, 4)}}

    # decode step at 256 rows, bf16 state, one launch per layer over 36 layers
    w = W.get("c2")
    buf, pool, views = make_pool(L, W, w, seed=0)
    n = 256
    rng = np.random.default_rng(0)
    idx = torch.from_numpy(rng.permutation(w.num_slots).astype(np.int32)).cuda()
    has = torch.ones(n, dtype=torch.uint8, device="cuda")
    x, cw, a, b = W.decode_inputs(w, n, seed=0, layer=0)
    X = torch.from_numpy(x).to(torch.bfloat16).cuda()
    CW = torch.from_numpy(cw).to(torch.bfloat16).cuda()
    A, B = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    out = torch.empty((n, w.num_v_heads, w.head_v_dim), device="cuda")
    da = L.decode_args(n, w.num_k_heads, idx, has, X, CW, A, B, out, DECODE_FLAGS)

    def dec_all():
        for l in w.gdn_layers:
            assert L.lsc_gdn_decode(pool, l, da, fwd) == L.LSC_OK

    t = timed(dec_all, reps) / len(w.gdn_layers)
    v = views[w.gdn_layers[0]]
    bytes_ = decode_bytes(v, w, n)
    parts["decode_c2"] = {"workload": "c2: 256 rows, ssm bf16, page +512 B, one launch per layer x 36",
                          "kernel": "decode_kernel<128,bf16,1>", "launch_ms": round(t * 1e3, 4),
                          "bytes_per_launch": bytes_, "GB/s": round(bytes_ / t / 1e9, 1),
                          "frac": round(bytes_ / t / 1e9 / hbm_peak, 4), "rows_per_s": round(n / t, 1),
                          "traffic": kernel_traffic("decode_kernel<128,bf16,1>")}
    L.lsc_pool_destroy(pool)
    del buf
    torch.cuda.empty_cache()

    # standalone gather and scatter on c2's pool: 256 rows, bf16 ssm, dense
    # conv [256, 8192, 3] bf16 (12.6 MB) and ssm [256, 32, 128, 128] bf16 (268 MB)
    w = W.get("c2")
    buf, pool, views = make_pool(L, W, w, seed=0)
    v = views[w.gdn_layers[0]]
    n = 256
    idx = torch.from_numpy(np.random.default_rng(1).permutation(w.num_slots).astype(np.int32)).cuda()
    conv_d = torch.empty((n, v.conv_bytes), dtype=torch.uint8, device="cuda")
    ssm_d = torch.empty((n, v.ssm_bytes), dtype=torch.uint8, device="cuda")
    i_l = [0]

    def gather_one():
        i_l[0] += 1
        l = w.gdn_layers[i_l[0] % len(w.gdn_layers)]
        assert L.lsc_gather(pool, l, idx, None, n, conv_d, ssm_d, fwd) == L.LSC_OK

    def scatter_one():
        i_l[0] += 1
        l = w.gdn_layers[i_l[0] % len(w.gdn_layers)]
        assert L.lsc_scatter(pool, l, idx, n, conv_d, ssm_d, fwd) == L.LSC_OK

    gs_bytes = 2 * n * (v.conv_bytes + v.ssm_bytes)
    for name, fn, kern in (("gather_c2", gather_one, "gather_kernel"), ("scatter_c2", scatter_one, "scatter_kernel")):
        t = timed(fn, 36)
        parts[name] = {"workload": "c2 pool: 256 rows (a permutation of the 256 slots), conv [8192,3] bf16 + ssm "
                                   "[32,128,128] bf16 per row, one GDN layer per launch, layers in turn",
                       "kernel": kern, "launch_ms": round(t * 1e3, 4), "bytes_per_launch": gs_bytes,
                       "GB/s": round(gs_bytes / t / 1e9, 1), "frac": round(gs_bytes / t / 1e9 / hbm_peak, 4),
                       "rows_per_s": round(n / t, 1), "bytes_basis": "conv + ssm views read and written per row",
                       "traffic": kernel_traffic(kern)}
    L.lsc_pool_destroy(pool)
    del buf, conv_d, ssm_d
    torch.cuda.empty_cache()

    # restore storm
    w = W.get("c3")
    rows = W.restore_rows("c3")
    buf, pool, views = make_pool(L, W, w, seed=0)
    ops = L.ops_array(rows.live, rows.src, rows.restore_hash, rows.save_hash, rows.save_slot)
    hs = torch.from_numpy(rows.hs_prefill.copy()).cuda()
    rep = {}

    def storm():
        rc, r = L.lsc_restore(pool, ops, rows.nkv, rows.block_size, rows.initialized, hs, fwd, None)
        assert rc == L.LSC_OK
        rep["r"] = r

    t = timed(storm, reps)
    r = rep["r"]
    v = views[w.gdn_layers[0]]
    bytes_ = restore_bytes(v, r.n_hit, len(w.gdn_layers), r.n_hit + r.n_miss)
    parts["restore_c3"] = {"workload": "c3: 512 rows over 1024 slots, 205 hit / 154 miss / 153 no-op, hot source",
                           "kernel": "restore_bulk_kernel", "launch_ms": round(t * 1e3, 4), "bytes_per_launch": bytes_,
                           "GB/s": round(bytes_ / t / 1e9, 1), "frac": round(bytes_ / t / 1e9 / hbm_peak, 4),
                           "rows_per_s": round(512 / t, 1), "traffic": kernel_traffic("restore_bulk_kernel c3")}
    tr = parts["restore_c3"]["traffic"]
    parts["restore_c3"]["frac_basis"] = ("algorithmic: every hit's read counted, though the hot source's re-reads "
                                         "hit L2, so frac can exceed 1")
    parts["restore_c3"]["dram_frac"] = round(tr / t / 1e9 / hbm_peak, 4) if tr else None
    parts["restore_c3"]["dram_frac_basis"] = ("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch / launch "
                                              "time / peak; a lower bound, since lines still dirty in L2 when the "
                                              "kernel ends are not counted; null when the kernel changed since the "
                                              "counters were taken")
    L.lsc_pool_destroy(pool)
    del buf, hs
    torch.cuda.empty_cache()

    # resume prefill: 64 sequences, 36 layers (one input set per layer is reused
    # across layers to bound memory; every layer has its own state)
    w = W.get("c4")
    buf, pool, views = make_pool(L, W, w, seed=0)
    lengths = W.seq_lengths(64, 64, 2048, seed=0)
    cu, q, k, vv, a, b = W.recurrent_inputs(w, lengths, seed=0, layer=0)
    T = int(cu[-1])
    rng = np.random.default_rng(4)
    idx = torch.from_numpy(rng.permutation(w.num_slots)[:64].astype(np.int32)).cuda()
    has = torch.from_numpy((rng.random(64) < 0.5).astype(np.uint8)).cuda()
    dev = [torch.from_numpy(z).cuda() for z in (cu, q, k, vv, a, b)]
    out = torch.empty((T, w.num_v_heads, w.head_v_dim), device="cuda")
    def rec_all(ra):
        for l in w.gdn_layers:
            assert L.lsc_gdn_recurrent(pool, l, ra, fwd) == L.LSC_OK

    nl = len(w.gdn_layers)
    flops = 6.0 * T * w.num_v_heads * w.head_v_dim * w.head_k_dim * nl
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    fp32_peak = sms * 128 * 2 * 2070e6
    # the chunked order's caller workspace, allocated once outside the timing
    ra0 = L.recurrent_args(64, w.num_k_heads, T, idx, has, *dev, out, algorithm=L.LSC_RECURRENT_AUTO)
    _, ws_bytes = L.lsc_gdn_recurrent_workspace_bytes(pool, ra0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    rec = {}
    for algo in (L.LSC_RECURRENT_AUTO, L.LSC_RECURRENT_TOKEN):
        ra = L.recurrent_args(64, w.num_k_heads, T, idx, has, *dev, out, algorithm=algo,
                              workspace=ws if algo == L.LSC_RECURRENT_AUTO else None,
                              workspace_bytes=ws_bytes if algo == L.LSC_RECURRENT_AUTO else 0)
        rec[algo] = timed(lambda: rec_all(ra), 2)
    t, t_tok = rec[L.LSC_RECURRENT_AUTO], rec[L.LSC_RECURRENT_TOKEN]
    # tensor-core work of the chunked order, tf32 x 3 passes: per (chunk, v head)
    # [P'|R'] 2*128*128*128, D and O 2*128*64*64 each, the update 2*128*128*64;
    # per (chunk, qk head) the Gram product 2*128*64*128
    n_chunks = sum((int(n) + 63) // 64 for n in lengths)
    tc_flops = 3.0 * nl * (n_chunks * w.num_v_heads * (2.0 * 128 ** 3 + 2 * 2 * 128 * 64 * 64 + 2 * 128 * 128 * 64)
                           + n_chunks * w.num_k_heads * 2.0 * 128 * 64 * 128)
    tf32_peak = measured("bf16_tflops", 1900.0) * 1e12 * 1.1 / 2.25
    parts["recurrent_c4"] = {"workload": f"c4: 64 sequences, {T} tokens, 36 layers, state [32,128,128] f32",
                             "kernel": "chunk_prep_kernel + chunked_tc_kernel<f32> (64-token chunks on the tensor "
                                       "cores, tf32 x 3; the default at head_k_dim 128)",
                             "ms_per_36_layers": round(t * 1e3, 3),
                             "token_layers_per_s": round(T * nl / t, 1),
                             "TFLOP/s": round(flops / t / 1e12, 2),
                             "roofline": {"bound": "alu", "peak_TFLOP/s": round(fp32_peak / 1e12, 1),
                                          "frac": round(flops / t / fp32_peak, 4),
                                          "peak_basis": f"{sms} SMs x 128 FP32 lanes x 2 flop x 2070 MHz: the token "
                                                        "recurrence's own bound, kept for comparison"},
                             "flops_basis": "algorithmic: 6 dk dv per (token, v head) -- S k, the rank-1 update, "
                                            "S q -- whichever order computes it",
                             "tensor": {"TFLOP/s_issued": round(tc_flops / t / 1e12, 1),
                                        "tf32_peak_TFLOP/s": round(tf32_peak / 1e12, 1),
                                        "frac": round(tc_flops / t / tf32_peak, 4),
                                        "peak_basis": "measured bf16 burst x 1.1/2.25 (tf32 vs bf16 nominal)",
                                        "work_basis": "tf32 x 3 products of both kernels"},
                             "workspace_bytes_per_layer": int(ws_bytes),
                             "token": {"kernel": "recurrent128_kernel<f32> (token order, two tokens per pass)",
                                       "ms_per_36_layers": round(t_tok * 1e3, 3),
                                       "frac": round(flops / t_tok / fp32_peak, 4)},
                             "speedup_vs_token": round(t_tok / t, 3)}
    del ws
    L.lsc_pool_destroy(pool)
    del buf, out, dev
    torch.cuda.empty_cache()

    # prefill conv of the same token mix (x bf16 [T, 8192] -> q, k, v fp32, conv
    # states updated), on two GDN layers of c4's shapes, alternating
    w = W.get("c4")
    w.layers = [W.GDN, W.ATTN, W.GDN]
    buf, pool, views = make_pool(L, W, w, seed=0)
    cu, x, cw = W.prefill_inputs(w, lengths, seed=0, layer=0)
    T = int(cu[-1])
    idx = torch.from_numpy(rng.permutation(w.num_slots)[:64].astype(np.int32)).cuda()
    xd = torch.from_numpy(x).to(torch.bfloat16).cuda()
    cwd = torch.from_numpy(cw).to(torch.bfloat16).cuda()
    q = torch.empty((T, w.num_k_heads, w.head_k_dim), device="cuda")
    k = torch.empty_like(q)
    v = torch.empty((T, w.num_v_heads, w.head_v_dim), device="cuda")
    pa = L.prefill_conv_args(64, w.num_k_heads, T, idx, has, torch.from_numpy(cu).cuda(), xd, cwd, q, k, v)
    i_l = [0]

    def conv_one():
        i_l[0] += 1
        assert L.lsc_gdn_prefill_conv(pool, w.gdn_layers[i_l[0] % 2], pa, fwd) == L.LSC_OK

    t = timed(conv_one, 10)
    C, Wd = w.conv_dim, w.conv_width
    pbytes = T * C * (2 + 4) + C * Wd * 2 + 64 * C * (Wd - 1) * 2 * 2
    parts["prefill_conv_c4"] = {"workload": f"c4: 64 sequences, {T} tokens, conv [8192, 3] bf16 from the slots, "
                                            "q/k/v fp32 out, one layer per launch",
                                "kernel": "prefill_conv_vec_kernel<bf16,4> + prefill_state_kernel",
                                "launch_ms": round(t * 1e3, 4), "bytes_per_launch": pbytes,
                                "GB/s": round(pbytes / t / 1e9, 1), "frac": round(pbytes / t / 1e9 / hbm_peak, 4),
                                "bytes_basis": "x read (bf16) + q, k, v written (fp32) + weights + conv state read and "
                                               "written per sequence"}
    L.lsc_pool_destroy(pool)
    del buf, xd, q, k, v
    torch.cuda.empty_cache()
    # copy_prefix: 12 attention layers, 2048 blocks of 64 tokens x 2 kv heads x 256
    # dims bf16 (64 KiB) in 64.5 KiB pages; 16 prefixes of 2016 tokens (31 full
    # blocks + a half block) copied into other blocks
    d = L.lsc_kv_pool_desc(12, 2048, 64, 2, 256, L.LSC_BF16, 65536 + 512)
    kvn = L.lsc_kv_pool_required_bytes(d)
    kbuf = torch.empty(kvn, dtype=torch.uint8, device="cuda")
    kbuf.view(torch.int32).random_(generator=torch.Generator(device="cuda").manual_seed(0))
    rc, kpool = L.lsc_kv_pool_create(d, kbuf, kvn)
    assert rc == L.LSC_OK
    perm = np.random.default_rng(7).permutation(2048)
    ksrc, kdst, knt = [], [], []
    for i in range(16):
        ksrc += list(perm[64 * i:64 * i + 32])
        kdst += list(perm[1024 + 64 * i:1024 + 64 * i + 32])
        knt += [64] * 31 + [32]
    kops = L.kv_ops(ksrc, kdst, knt)
    nb = [0]

    def copy_one():
        rc, nb[0] = L.lsc_copy_prefix(kpool, kops, fwd)
        assert rc == L.LSC_OK

    t = timed(copy_one, 20)
    kbytes = 2 * nb[0]  # read + write
    parts["copy_prefix_kv"] = {"workload": "12 attention layers, 2048 blocks x 64 tokens x 2 kv heads x 256 dims bf16 "
                                           "in 64.5 KiB pages; 16 prefixes of 2016 tokens (512 block ops)",
                               "kernel": "kv_copy_kernel", "launch_ms": round(t * 1e3, 4),
                               "bytes_per_launch": kbytes, "GB/s": round(kbytes / t / 1e9, 1),
                               "frac": round(kbytes / t / 1e9 / hbm_peak, 4),
                               "bytes_basis": "token rows copied: read + write"}
    L.lsc_kv_pool_destroy(kpool)
    del kbuf
    torch.cuda.empty_cache()
    parts["prefix_cache_host"] = measure_prefix_cache(L)
    parts["snapshot_store_c1"] = measure_store(L, W, torch)
    return parts


def measure_store(L, W, torch, n_slots=8):
    """Save and load a c1 slot's linear state (36 GDN layers: conv + ssm views,
    77.3 MB) through the snapshot store in a scratch directory of the host:
    device -> pinned host -> CRC-32C -> temporary file -> rename, and back."""
    import shutil
    import tempfile
    w = W.get("c1")
    w.num_slots = n_slots
    buf, pool, views = make_pool(L, W, w, seed=0)
    d = tempfile.mkdtemp(prefix="lsc_store_")
    try:
        rc, st = L.lsc_store_open(d, 0xC1, 1 << 40)
        assert rc == L.LSC_OK
        v0 = views[w.gdn_layers[0]]
        per = len(w.gdn_layers) * (v0.conv_bytes + v0.ssm_bytes)
        fwd = torch.cuda.current_stream()
        t0 = time.perf_counter()
        for i in range(n_slots):
            assert L.lsc_store_save_state(st, 100 + i, pool, i, fwd) == L.LSC_OK
        t_save = (time.perf_counter() - t0) / n_slots
        t0 = time.perf_counter()
        for i in range(n_slots):
            assert L.lsc_store_load_state(st, 100 + i, pool, n_slots - 1 - i, fwd) == L.LSC_OK
        t_load = (time.perf_counter() - t0) / n_slots
        L.lsc_store_close(st)
    finally:
        shutil.rmtree(d, ignore_errors=True)
        L.lsc_pool_destroy(pool)
        del buf
        torch.cuda.empty_cache()
    return {"workload": f"c1 slot snapshot: 36 GDN layers, {per} bytes of conv + ssm views per slot, "
                        f"{n_slots} slots saved then loaded, host scratch directory",
            "bytes_per_slot": per, "save_ms": round(t_save * 1e3, 2), "load_ms": round(t_load * 1e3, 2),
            "save_GB/s": round(per / t_save / 1e9, 2), "load_GB/s": round(per / t_load / 1e9, 2),
            "clock": "host wall clock; includes D2H / H2D, CRC-32C, file write + fsync + rename / read",
            "bound": "host I/O and CRC (no HBM roofline)"}


def prefix_cache_schedule(steps, num_slots=1024, block=64, batch=256, churn=4, seed=0):
    """A deterministic scheduler workload: `batch` running sequences advance 16
    tokens per step; a sequence saves its prefix at every block boundary and a
    new one asks to restore its family's 4-block prefix; `churn` sequences
    finish and are replaced every step.  Returns per-step (rows, released,
    joined) -- rows as lsc_pc_row tuples."""
    rng = np.random.default_rng(seed)
    fam = {}
    tokens = {}
    nxt = 0
    for _ in range(batch):
        fam[nxt], tokens[nxt] = int(rng.integers(1, 65)), 0
        nxt += 1
    sched = []
    for _ in range(steps):
        rows = []
        for s in sorted(tokens):
            new = tokens[s] == 0
            after = 4 * block if new else tokens[s] + 16
            rh = (fam[s] << 32) | 4 if new else 0
            sh = (fam[s] << 32) | (after // block) if after % block == 0 else 0
            rows.append((s, rh, sh, after))
            tokens[s] = after
        gone = [int(x) for x in rng.choice(sorted(tokens), churn, replace=False)]
        joined = []
        for g in gone:
            del tokens[g], fam[g]
            fam[nxt], tokens[nxt] = int(rng.integers(1, 65)), 0
            joined.append(nxt)
            nxt += 1
        sched.append((rows, gone, joined))
    return sched, num_slots, block, batch


def measure_prefix_cache(L, steps=3000, oracle_steps=60):
    """Host-side cost of the scheduler's prefix cache per step (resolve + commit
    + sequence churn), through the C ABI; the plain oracle on a prefix of the
    same schedule beside it."""
    sched, num_slots, block, batch = prefix_cache_schedule(steps)
    arrays = [L.pc_rows(*zip(*rows)) for rows, _, _ in sched]
    rc, pc = L.lsc_pc_create(num_slots, block)
    assert rc == L.LSC_OK
    for s in range(batch):
        assert L.lsc_pc_allocate_live_slot(pc, s)[0] == L.LSC_OK
    saves = hits = 0
    t = time.perf_counter()
    for arr, (_, gone, joined) in zip(arrays, sched):
        rc, ops, init, rep = L.lsc_pc_resolve(pc, arr)
        assert rc == L.LSC_OK
        saves += rep.save
        hits += rep.restore_hit
        assert L.lsc_pc_commit(pc) == L.LSC_OK
        for g in gone:
            assert L.lsc_pc_release_sequence(pc, g) == L.LSC_OK
        for j in joined:
            assert L.lsc_pc_allocate_live_slot(pc, j)[0] == L.LSC_OK
    el = time.perf_counter() - t
    counts = L.lsc_pc_counts(pc)[1]
    L.lsc_pc_destroy(pc)
    from oracle.prefix_cache import PrefixCache  # the plain model, timed as it stands
    orc = PrefixCache(num_slots, block)
    for s in range(batch):
        orc.allocate_live_slot(s)
    t = time.perf_counter()
    for rows, gone, joined in sched[:oracle_steps]:
        orc.resolve(rows)
        orc.commit()
        for g in gone:
            orc.release_sequence(g)
        for j in joined:
            orc.allocate_live_slot(j)
    el_o = time.perf_counter() - t
    return {"workload": f"{num_slots} slots, {batch}-row batches, 4 sequences replaced per step, "
                        f"saves at {block}-token boundaries, restores of 4-block family prefixes",
            "us_per_step": round(el / steps * 1e6, 2), "rows_per_s": round(batch * steps / el, 1),
            "steps": steps, "promotions": saves, "restore_hits": hits,
            "final_free_live_checkpoint_reserved": list(counts),
            "oracle_us_per_step": round(el_o / oracle_steps * 1e6, 1), "oracle_steps": oracle_steps,
            "clock": "host wall clock, one thread, includes the ctypes calls"}


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(n_rows=None, seed=0):
    """A bounded sample of the serving step on the host: the same pages, shapes
    and layers as the c1 step, with n_rows restore+decode rows (2 n_rows slots);
    by default one row per host thread (the oracle parallelises over rows)."""
    import oracle
    from linear_attention_state_lsc_gb300 import workloads as W
    if n_rows is None:
        n_rows = max(1, min(16, oracle.num_threads()))
    w = W.get("c1")
    w.num_slots = 2 * n_rows
    kinds = [oracle.GDN if k == W.GDN else oracle.ATTENTION for k in w.layers]
    pool = oracle.Pool(kinds, w.num_slots, w.conv_dim, w.conv_width, oracle.BF16, w.num_v_heads,
                       w.head_v_dim, w.head_k_dim, oracle.F32, w.page_bytes)
    _, Lo = oracle.layout(pool)
    regions = {}
    rng = np.random.default_rng(seed)
    for l in w.gdn_layers:
        regions[l] = rng.integers(0, 256, w.num_slots * w.page_bytes, dtype=np.uint8)
        pages = regions[l].reshape(w.num_slots, w.page_bytes)
        vals = rng.standard_normal((w.num_slots, Lo["ssm_elems"]), dtype=np.float32)
        pages[:, Lo["ssm_offset"]:Lo["ssm_offset"] + Lo["ssm_bytes"]] = vals.view(np.uint8).reshape(w.num_slots, -1)
        conv = W.to_dtype_bytes(rng.standard_normal((w.num_slots, Lo["conv_elems"]), dtype=np.float32), W.BF16)
        pages[:, :Lo["conv_bytes"]] = conv
    live = np.arange(n_rows, dtype=np.int32)
    src = np.arange(n_rows, 2 * n_rows, dtype=np.int32)
    nkv = np.full(n_rows, 64, np.int32)
    init = np.zeros(n_rows, np.uint8)
    inputs = [W.decode_inputs(w, n_rows, seed=seed, layer=l) for l in w.gdn_layers]
    inputs = [(W.to_dtype_bytes(x, W.BF16), W.to_dtype_bytes(cw, W.BF16), a, b) for x, cw, a, b in inputs]
    per_row = 2 * len(w.gdn_layers) * (Lo["conv_bytes"] + Lo["ssm_bytes"]) + 1
    dec_row = 2 * (Lo["conv_bytes"] + Lo["ssm_bytes"]) + w.conv_dim * 2 + 2 * w.num_v_heads * 4 + \
        w.num_v_heads * w.head_v_dim * 4 + 5
    step_bytes = n_rows * per_row + len(w.gdn_layers) * (n_rows * dec_row + w.conv_dim * w.conv_width * 2)

    def run():
        hs = (nkv > 0).astype(np.uint8)
        rc = oracle.restore(pool, regions, live, src, nkv, 64, init, hs)
        assert rc == oracle.OK
        for g, l in enumerate(w.gdn_layers):
            x, cw, a, b = inputs[g]
            rc, _ = oracle.gdn_decode(pool, regions[l], live, hs, x, cw, w.num_k_heads, a, b)
            assert rc == oracle.OK

    return run, step_bytes, n_rows, min(n_rows, oracle.num_threads())


def oracle_recurrent_sample(n_seq=None, tokens=128, seed=0):
    """A bounded sample of the c4 resume prefill on the host: n_seq sequences
    (one per host thread by default) of `tokens` tokens on one GDN layer of c4's
    shapes, all warm; returns (run, token_layers per run, flops per run)."""
    import oracle
    from linear_attention_state_lsc_gb300 import workloads as W
    if n_seq is None:
        n_seq = max(1, min(16, oracle.num_threads()))
    w = W.get("c4")
    w.num_slots = n_seq
    pool = oracle.Pool([oracle.GDN], n_seq, w.conv_dim, w.conv_width, oracle.BF16, w.num_v_heads, w.head_v_dim,
                       w.head_k_dim, oracle.F32, w.page_bytes)
    _, Lo = oracle.layout(pool)
    rng = np.random.default_rng(seed)
    region = np.zeros(n_seq * w.page_bytes, np.uint8)
    pages = region.reshape(n_seq, w.page_bytes)
    vals = rng.standard_normal((n_seq, Lo["ssm_elems"]), dtype=np.float32)
    pages[:, Lo["ssm_offset"]:Lo["ssm_offset"] + Lo["ssm_bytes"]] = vals.view(np.uint8).reshape(n_seq, -1)
    lengths = np.full(n_seq, tokens, np.int32)
    cu, q, k, v, a, b = W.recurrent_inputs(w, lengths, seed=seed, layer=0)
    idx = np.arange(n_seq, dtype=np.int32)
    has = np.ones(n_seq, np.uint8)
    T = int(cu[-1])

    def run():
        rc, _ = oracle.gdn_recurrent(pool, region, idx, has, cu, w.num_k_heads, q, k, v, a, b)
        assert rc == oracle.OK

    return run, T, T * w.num_v_heads * 6 * w.head_k_dim * w.head_v_dim, n_seq


def cpu_baseline(budget_s=12.0, recurrent_budget_s=3.0):
    import oracle.build as ob
    ob.build()
    run, step_bytes, n_rows, threads = oracle_sample()
    run()
    t = time.perf_counter()
    k = 0
    while time.perf_counter() - t < budget_s:
        run()
        k += 1
    el = time.perf_counter() - t
    line = {"value": round(step_bytes * k / el / 1e9, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
            "rows_per_s": round(n_rows * k / el, 3),
            "sample": f"c1 serving step on {n_rows} rows (restore x 36 GDN layers + 36 decode layers), "
                      f"{k} repetitions in {el:.1f} s, OpenMP over rows"}
    # the resume-prefill recurrence (c4 shapes) on the same host cores
    run, tl, flops, n_seq = oracle_recurrent_sample()
    run()
    t = time.perf_counter()
    k = 0
    while time.perf_counter() - t < recurrent_budget_s:
        run()
        k += 1
    el = time.perf_counter() - t
    line["recurrent_c4"] = {"token_layers_per_s": round(tl * k / el, 1), "GFLOP/s": round(flops * k / el / 1e9, 2),
                            "flops_basis": "6 dk dv per (token, v head), as the GPU line",
                            "sample": f"{n_seq} warm sequences x {tl // n_seq} tokens on one c4 layer "
                                      f"(state [32,128,128] f32), {k} repetitions in {el:.1f} s, "
                                      f"double precision, OpenMP over (sequence, head)"}
    return line


def run_reference(args):
    rank, local, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo", init_method="env://")
        if rank != 0:
            dist.barrier()
            dist.destroy_process_group()
            return
    import oracle.build as ob
    ob.build()
    run, step_bytes, n_rows, threads = oracle_sample()
    for _ in range(args.warmup):
        run()
    t = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t
    value = step_bytes * args.steps / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic",
            "config": {"workload": "c1-serving-step", "sample_rows": n_rows, "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"c1 serving step restricted to {n_rows} rows per step"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------------- profiler cases

NCU_CASES = {
    # name: (workload, rows, kernel)
    "decode_f32": ("c1", 64, "decode"),      # serving-step decode: fp32 state, 64 rows, 277 MB per launch
    "decode_bf16": ("c2", 256, "decode"),    # bf16 state, 256 rows, 571 MB per launch
    "restore": ("c1", 64, "restore"),        # 64 hits x 2 layers, 549 MB per launch
    "restore_c3": ("c3", 512, "restore"),    # the c3 storm on 2 of its 36 layers (4.4 GB pool, 1.76 GB algorithmic)
    "recurrent": ("c4", 16, "recurrent"),    # 16 sequences of 64..512 tokens, one layer (token order)
    "recurrent_chunked": ("c4", 16, "recurrent_chunked"),  # the same, 64-token chunks (preparation + state kernels)
    "prefill": ("c4", 32, "prefill"),        # prefill conv: 32 sequences of 64..2048 tokens, one layer
    "copy_prefix": ("c1", 4, "copy_prefix"), # K/V copy: 12 layers x 512 blocks of 64 KiB, 4 prefixes of 32 blocks
    "restore_vector": ("c1", 64, "restore_vector"),  # the restore case as 16-byte vectors (LSC_RESTORE_COPY=vector)
    "gather": ("c2", 256, "gather"),         # c2 pool, 256 rows -> dense conv + ssm (281 MB per launch)
    "scatter": ("c2", 256, "scatter"),       # the same, dense -> slots
}


def run_ncu_case(args):
    """A reduced copy of one kernel's workload: the same shapes, page and rows,
    2 GDN layers instead of 36, so that a profiler capture stays small."""
    import torch
    from linear_attention_state_lsc_gb300 import lsc as L
    from linear_attention_state_lsc_gb300 import workloads as W
    torch.cuda.set_device(0)
    L.load()
    name, n, kind = NCU_CASES[args.ncu_case]
    w = W.get(name)
    w.layers = [W.GDN, W.ATTN, W.GDN]
    buf, pool, views = make_pool(L, W, w, seed=0)
    fwd = torch.cuda.current_stream()
    rng = np.random.default_rng(0)
    if kind == "copy_prefix":
        d = L.lsc_kv_pool_desc(12, 512, 64, 2, 256, L.LSC_BF16, 65536 + 512)
        kvn = L.lsc_kv_pool_required_bytes(d)
        kbuf = torch.zeros(kvn, dtype=torch.uint8, device="cuda")
        rc, kpool = L.lsc_kv_pool_create(d, kbuf, kvn)
        assert rc == L.LSC_OK
        perm = rng.permutation(512)
        kops = L.kv_ops(perm[:32 * n], perm[256:256 + 32 * n], [64] * (32 * n))

        def launch(i):
            assert L.lsc_copy_prefix(kpool, kops, fwd)[0] == L.LSC_OK
    elif kind in ("restore", "restore_vector"):
        if kind == "restore_vector":
            os.environ["LSC_RESTORE_COPY"] = "vector"
        rows = W.restore_rows(name)
        ops = L.ops_array(rows.live, rows.src, rows.restore_hash, rows.save_hash, rows.save_slot)
        hs = torch.from_numpy(rows.hs_prefill.copy()).cuda()

        def launch(i):
            rc, _ = L.lsc_restore(pool, ops, rows.nkv, rows.block_size, rows.initialized, hs, fwd, None)
            assert rc == L.LSC_OK
    elif kind in ("gather", "scatter"):
        idx = torch.from_numpy(rng.permutation(w.num_slots)[:n].astype(np.int32)).cuda()
        v = views[w.gdn_layers[0]]
        conv_d = torch.zeros((n, v.conv_bytes), dtype=torch.uint8, device="cuda")
        ssm_d = torch.zeros((n, v.ssm_bytes), dtype=torch.uint8, device="cuda")

        def launch(i):
            l = w.gdn_layers[i % 2]
            if kind == "gather":
                assert L.lsc_gather(pool, l, idx, None, n, conv_d, ssm_d, fwd) == L.LSC_OK
            else:
                assert L.lsc_scatter(pool, l, idx, n, conv_d, ssm_d, fwd) == L.LSC_OK
    elif kind == "decode":
        idx = torch.from_numpy(rng.permutation(w.num_slots)[:n].astype(np.int32)).cuda()
        has = torch.ones(n, dtype=torch.uint8, device="cuda")
        x, cw, a, b = W.decode_inputs(w, n, seed=0, layer=0)
        t = [torch.from_numpy(x).to(torch.bfloat16).cuda(), torch.from_numpy(cw).to(torch.bfloat16).cuda(),
             torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()]
        out = torch.empty((n, w.num_v_heads, w.head_v_dim), device="cuda")
        da = L.decode_args(n, w.num_k_heads, idx, has, *t, out, DECODE_FLAGS)

        def launch(i):
            assert L.lsc_gdn_decode(pool, w.gdn_layers[i % 2], da, fwd) == L.LSC_OK
    elif kind == "prefill":
        lengths = W.seq_lengths(n, 64, 2048, seed=0)
        cu, x, cw = W.prefill_inputs(w, lengths, seed=0, layer=0)
        T = int(cu[-1])
        idx = torch.from_numpy(rng.permutation(w.num_slots)[:n].astype(np.int32)).cuda()
        has = torch.ones(n, dtype=torch.uint8, device="cuda")
        q = torch.empty((T, w.num_k_heads, w.head_k_dim), device="cuda")
        k = torch.empty_like(q)
        v = torch.empty((T, w.num_v_heads, w.head_v_dim), device="cuda")
        pa = L.prefill_conv_args(n, w.num_k_heads, T, idx, has, torch.from_numpy(cu).cuda(),
                                 torch.from_numpy(x).to(torch.bfloat16).cuda(),
                                 torch.from_numpy(cw).to(torch.bfloat16).cuda(), q, k, v)

        def launch(i):
            assert L.lsc_gdn_prefill_conv(pool, w.gdn_layers[i % 2], pa, fwd) == L.LSC_OK
    else:
        lengths = W.seq_lengths(n, 64, 512, seed=0)
        cu, q, k, vv, a, b = W.recurrent_inputs(w, lengths, seed=0, layer=0)
        T = int(cu[-1])
        idx = torch.from_numpy(rng.permutation(w.num_slots)[:n].astype(np.int32)).cuda()
        has = torch.ones(n, dtype=torch.uint8, device="cuda")
        dev = [torch.from_numpy(z).cuda() for z in (cu, q, k, vv, a, b)]
        out = torch.empty((T, w.num_v_heads, w.head_v_dim), device="cuda")
        algo = L.LSC_RECURRENT_CHUNKED if kind == "recurrent_chunked" else L.LSC_RECURRENT_TOKEN
        ra = L.recurrent_args(n, w.num_k_heads, T, idx, has, *dev, out, algorithm=algo)

        def launch(i):
            assert L.lsc_gdn_recurrent(pool, w.gdn_layers[i % 2], ra, fwd) == L.LSC_OK

    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(fwd)
    for i in range(args.steps):
        launch(i)
    e1.record(fwd)
    torch.cuda.synchronize()
    assert L.lsc_pool_status(pool, fwd) == L.LSC_OK
    print(json.dumps({"ncu_case": args.ncu_case, "launches": args.steps,
                      "ms_per_launch": round(e0.elapsed_time(e1) / args.steps, 4)}))
    L.lsc_pool_destroy(pool)


if __name__ == "__main__":
    a = parse()
    if a.ncu_case:
        run_ncu_case(a)
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_lsc(a)
