#!/usr/bin/env python3
"""Benchmark of the DCP top-K merge on one GB300 (or N independent replicas).

One step = one dcp_topk_merge launch over the prefill-scale workload
(T=8192 query rows, dcp=4 shards, K=2048 candidates per shard: 512 MiB of
rank-major candidates in, 128 MiB of sorted winners out), inputs resident in
HBM.  The timed region is bracketed by a barrier and a device synchronize;
the launches run back to back between two CUDA events on the launching
stream (the per-launch time is their span over the step count).  Inputs
(640 MiB) exceed the 129 MB L2, so no flush is needed between launches.

Prints one JSON line (rank 0).  Besides the headline, the line carries the
decode-size latencies (16 rows: the random and the tie-heavy workload), the
selector shapes of the first page's benchmark table (16 rows with 4096, 8192
and 16384 candidates; 64 and 256 rows with 8192), the local-top-K + merge
sweep, the HBM roofline of the merge kernel, the oracle timed on the host
cores, and an end-to-end number through the Python API with host buffers.

``--impl reference`` times the CPU oracle instead (the only reference this
method has): a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "merge rows/s at K=2048, DCP=4 (prefill-scale merge, T=8192)"
UNIT = "rows/s"
WORKLOAD = ("prefill merge: T=8192 rows, dcp=4, K=2048 (8192 candidates/row), rank-major fp32 "
            "scores bf16-rounded N(mu_t,1) with mu_t=(t mod 64)/8-4, distinct int32 ids per "
            "shard range, row_starts=262144*(t//256), seed 4")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "merge_prefill_T8192_ncu.txt")


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def kernel_source_hash():
    csrc = os.path.join(ROOT, "sparse_attention_indexer_stable_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        kv = {}
        for line in open(PROFILE_SUMMARY):
            if ":" in line and not line.startswith("#"):
                k, _, v = line.partition(":")
                kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout=3.0):
        """Block until the sampler has produced a line (nvidia-smi takes a
        moment to start), so that a short timed region is covered."""
        end = time.perf_counter() + timeout
        while self.proc is not None and not self.lines and time.perf_counter() < end:
            time.sleep(0.01)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def time_launches(torch, fn, steps, stream):
    """The K steps back to back between two CUDA events recorded on `stream`
    (an event between launches would keep each launch from overlapping its
    start with the previous one's end, as the library's launches do in a
    stream of work).  Returns the (start, end) events."""
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
    return a, b


def median_of_reps(torch, fn, stream, reps=7, launches=200, graph=False):
    """Median over `reps` repetitions of the mean per-launch time of
    `launches` back-to-back launches (µs)."""
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(launches):
                fn()
        run = g.replay
    else:
        def run():
            for _ in range(launches):
                fn()
    out = []
    for _ in range(reps + 1):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            run()
            b.record(stream)
        b.synchronize()
        out.append(a.elapsed_time(b) * 1000.0 / launches)
    return statistics.median(out[1:])


def cold_launch_us(torch, fn, stream, reps=21):
    """Median device time (µs) of single launches with the L2 flushed before
    each (a 256 MiB write, twice the 129 MB L2), so that the inputs come from
    HBM.  The flush, the start event, the launch and the end event are queued
    together: the flush keeps the stream busy while the host queues the rest,
    so the interval holds the launch alone, not the host's launch latency."""
    flush = torch.empty(64 << 20, dtype=torch.float32, device=stream.device)
    out = []
    for _ in range(reps + 1):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
            a.record(stream)
            fn()
            b.record(stream)
        b.synchronize()
        out.append(a.elapsed_time(b) * 1000.0)
    del flush
    return statistics.median(out[1:])


def cold_inputs_launch_us(torch, fns, stream):
    """Median device time (µs) of single launches whose inputs are not in L2:
    fns[i] runs on its own copy of the inputs, the copies together larger
    than L2 and used in turn, so each launch reads its inputs from HBM while
    the kernel's code stays cached.  The launches are queued together, each
    between two events (which also keeps it from overlapping its neighbours),
    so no interval holds the host's launch latency."""
    evs = []
    with torch.cuda.stream(stream):
        for fn in fns:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
    stream.synchronize()
    return statistics.median(a.elapsed_time(b) * 1000.0 for a, b in evs[len(evs) // 2:])


def replica_throughput(torch, local_ms, rows_per_step, steps, dist=None, device=None):
    """Whole-job rows/s over the ranks of a replicas-only run: every rank
    processed rows_per_step * steps rows; the job took the slowest rank's
    time.  Returns (rows/s, max ms over ranks, world size)."""
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    world = 1
    if dist is not None and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        world = dist.get_world_size()
    max_ms = float(t.item())
    return rows_per_step * steps * world / (max_ms / 1000.0), max_ms, world


def cpu_oracle_sample(m, budget_s=10.0):
    """The oracle as it stands, single-threaded, on rows of the workload until
    about budget_s seconds have passed.  Returns (rows/s, rows, seconds)."""
    import oracle

    oracle.build()
    rows_done, t0 = 0, time.perf_counter()
    batch = 64
    order = np.random.default_rng(0).permutation(m.T)
    while True:
        rows = order[rows_done % m.T: rows_done % m.T + batch]
        oracle.merge(m.scores, m.ids, m.row_starts, rows=rows)
        rows_done += len(rows)
        el = time.perf_counter() - t0
        if el >= budget_s or rows_done >= 4 * m.T:
            return rows_done / el, rows_done, el


def cpu_oracle_sample_threads(m, threads, budget_s=5.0):
    """The same oracle, unchanged, on `threads` host threads at once, each on
    its own rows (rows are independent; the C call releases the GIL): the
    whole host's throughput.  Returns (rows/s, rows, seconds)."""
    import concurrent.futures

    import oracle

    oracle.build()
    order = np.random.default_rng(2).permutation(m.T)
    batch = 16
    counts = [0] * threads
    stop = time.perf_counter() + budget_s

    def work(k):
        i = k * batch
        while time.perf_counter() < stop:
            start = i % m.T
            rows = order[start:start + batch]
            oracle.merge(m.scores, m.ids, m.row_starts, rows=rows)
            counts[k] += len(rows)
            i += threads * batch

    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(threads) as pool:
        list(pool.map(work, range(threads)))
    el = time.perf_counter() - t0
    return sum(counts) / el, sum(counts), el


def run_reference(args):
    rank = env_int("RANK", 0)
    if rank != 0:
        return 0
    m = workloads.prefill()
    per_step = []
    import oracle

    oracle.build()
    rng = np.random.default_rng(1)
    # size each step's sample so the whole run stays within about two minutes
    t0 = time.perf_counter()
    oracle.merge(m.scores, m.ids, m.row_starts, rows=np.arange(16))
    per_row = (time.perf_counter() - t0) / 16
    sample_rows = int(max(1, min(256, 120.0 / (args.steps + args.warmup) / per_row)))
    for k in range(args.warmup + args.steps):
        rows = rng.choice(m.T, sample_rows, replace=False)
        t0 = time.perf_counter()
        oracle.merge(m.scores, m.ids, m.row_starts, rows=rows)
        el = time.perf_counter() - t0
        if k >= args.warmup:
            per_step.append(el)
    tot = sum(per_step)
    value = sample_rows * len(per_step) / tot
    sample = (f"{sample_rows} random rows of the prefill workload per step, single-threaded "
              f"C oracle (qsort of 64-bit keys)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * tot / len(per_step), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "host": host_cpu()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def host_cpu() -> dict:
    """The host the CPU oracle runs on: architecture, logical cores, model."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"machine": platform.machine(), "nproc": os.cpu_count(), "model": model}


def run_ours(args):
    import torch

    import sparse_attention_indexer_stable_gb300 as dk

    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local_rank = env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist = dist_mod
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    stream = torch.cuda.Stream(device=dev)
    if args.workload.startswith("sweep"):
        # the fused top-K over one sweep size's logits (dcp=4, L=4096, K=2048)
        T_sw = int(args.workload[len("sweep"):])
        lg = torch.from_numpy(workloads.sweep_logits(T_sw)).to(dev)
        m = workloads.FusedShape(T_sw, lg.shape[0], lg.shape[2], 2048)
        out_ids = torch.empty((m.T, m.K), dtype=torch.int32, device=dev)
        out_scores = torch.empty((m.T, m.K), dtype=torch.float32, device=dev)

        def step():
            dk.fused_topk(lg, m.K, out_scores=out_scores, out_ids=out_ids, stream=stream)
    else:
        m = workloads.NAMED[args.workload]()
        scores = torch.from_numpy(m.scores).to(dev)
        ids = torch.from_numpy(m.ids).to(dev)
        rs = None if m.row_starts is None else torch.from_numpy(m.row_starts).to(dev)
        out_ids = torch.empty((m.T, m.K), dtype=torch.int32, device=dev)
        out_scores = torch.empty((m.T, m.K), dtype=torch.float32, device=dev)

        def step():
            dk.merge(scores, ids, rs, out_ids=out_ids, out_scores=out_scores, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        clk.wait_first()
        t0 = time.perf_counter()
        evs = time_launches(torch, step, args.steps, stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        barrier()
        torch.cuda.synchronize(dev)
        # the same step as 7 repetitions of 200 back-to-back launches (the
        # first page's protocol; about 0.3 s at prefill size), so the clock
        # record also covers a long stretch of the kernel
        us_7x200 = median_of_reps(torch, step, stream, reps=7, launches=200)
        torch.cuda.synchronize(dev)
    total_ms = evs[0].elapsed_time(evs[1])
    value, max_ms, _ = replica_throughput(torch, total_ms, m.T, args.steps, dist, dev)

    # roofline of the merge kernel (the only kernel of the step)
    alg_bytes = m.algorithmic_bytes()
    avg_launch_ms = total_ms / args.steps
    achieved = alg_bytes / (avg_launch_ms / 1000.0) / 1e9
    peak, peak_kind = hbm_peak()

    # decode-size latencies and the local top-K + merge sweep (rank 0 only)
    extras = {}
    if rank == 0 and not args.skip_extras:
        extras = decode_and_sweep(torch, dk, dev, stream)

    # end to end through the Python API with host buffers
    e2e = None
    if not args.skip_extras and not args.workload.startswith("sweep"):
        e2e = end_to_end(torch, dk, m, dev, stream, steps=max(3, min(20, args.steps)))
    cpu = cpu_all = None
    if rank == 0 and world == 1 and not args.skip_extras and not args.workload.startswith("sweep"):
        v, rows, secs = cpu_oracle_sample(m, budget_s=args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{rows} rows of the prefill workload ({secs:.1f} s), single-threaded "
                         f"C oracle", "host": host_cpu()}
        threads = os.cpu_count() or 1
        vt, rows_t, secs_t = cpu_oracle_sample_threads(m, threads)
        cpu_all = {"value": vt, "unit": UNIT, "cores": threads, "kind": "oracle",
                   "sample": f"{rows_t} rows of the prefill workload ({secs_t:.1f} s), the same "
                             f"C oracle on {threads} threads, rows split between them"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD if args.workload == "prefill" else args.workload,
                       "T": m.T, "dcp": m.dcp, "K": m.K,
                       "chunk_rows": 1024, "l2": "inputs 640 MiB > 129 MB L2, no flush",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "us_per_launch": 1000.0 * avg_launch_ms,
            "us_per_launch_median_7x200": us_7x200,
            "achieved_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": profiled_traffic() if args.workload == "prefill" else None,
                         "algorithmic_bytes": alg_bytes},
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "wall_s_timed_region": wall,
        }
        line.update(extras)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def decode_and_sweep(torch, dk, dev, stream):
    out = {}
    for name in ("decode", "tieheavy"):
        m = workloads.NAMED[name]()
        s = torch.from_numpy(m.scores).to(dev)
        i = torch.from_numpy(m.ids).to(dev)
        oi = torch.empty((m.T, m.K), dtype=torch.int32, device=dev)
        os_ = torch.empty((m.T, m.K), dtype=torch.float32, device=dev)

        def fn():
            dk.merge(s, i, out_ids=oi, out_scores=os_, stream=stream)

        # the C ABI called with prepared arguments: the launch cost without
        # the Python wrapper's checks
        lib = dk.library()
        args = (s.data_ptr(), i.data_ptr(), m.T, m.dcp, m.K, None, oi.data_ptr(),
                os_.data_ptr(), None, 0, stream.cuda_stream)

        def raw():
            lib.dcp_topk_merge(*args)

        out[f"{name}_T{m.T}_us_per_launch"] = median_of_reps(torch, raw, stream)
        out[f"{name}_T{m.T}_us_per_graph_replay"] = median_of_reps(torch, raw, stream, graph=True)
        out[f"{name}_T{m.T}_us_per_python_call"] = median_of_reps(torch, fn, stream)
        # single launches on inputs from HBM (200 copies of the 1 MiB of
        # candidates, cycled twice), and with the whole L2 flushed, code too
        copies = [(s.clone(), i.clone()) for _ in range(200)]
        fns = [(lambda a=(sc.data_ptr(), ic.data_ptr(), m.T, m.dcp, m.K, None, oi.data_ptr(),
                           os_.data_ptr(), None, 0, stream.cuda_stream): lib.dcp_topk_merge(*a))
               for sc, ic in copies * 2]
        out[f"{name}_T{m.T}_us_cold_inputs"] = cold_inputs_launch_us(torch, fns, stream)
        del copies, fns
        out[f"{name}_T{m.T}_us_cold_l2_flushed"] = cold_launch_us(torch, raw, stream)
    # the selector shapes of the first page's table (K=2048; candidates dcp*K;
    # random fp32 scores), timed like the decode merge
    shapes = {}
    for T, dcp in ((16, 2), (16, 4), (16, 8), (64, 4), (256, 4)):
        m = workloads.decode(seed=50 + T + dcp, T=T, dcp=dcp)
        s = torch.from_numpy(m.scores).to(dev)
        i = torch.from_numpy(m.ids).to(dev)
        oi = torch.empty((m.T, m.K), dtype=torch.int32, device=dev)
        os_ = torch.empty((m.T, m.K), dtype=torch.float32, device=dev)
        lib = dk.library()
        args = (s.data_ptr(), i.data_ptr(), m.T, m.dcp, m.K, None, oi.data_ptr(),
                os_.data_ptr(), None, 0, stream.cuda_stream)

        def raw():
            lib.dcp_topk_merge(*args)

        shapes[f"rows{T}_candidates{dcp * m.K}"] = {
            "us_per_launch": median_of_reps(torch, raw, stream),
            "us_per_graph_replay": median_of_reps(torch, raw, stream, graph=True)}
    out["selector_shapes_K2048"] = shapes
    # K=4096 (16 rows, dcp=4: 16384 candidates per row)
    m = workloads.decode(seed=77, T=16, dcp=4, K=4096)
    s4 = torch.from_numpy(m.scores).to(dev)
    i4 = torch.from_numpy(m.ids).to(dev)
    oi4 = torch.empty((m.T, m.K), dtype=torch.int32, device=dev)
    os4 = torch.empty((m.T, m.K), dtype=torch.float32, device=dev)
    args4 = (s4.data_ptr(), i4.data_ptr(), m.T, m.dcp, m.K, None, oi4.data_ptr(), os4.data_ptr(),
             None, 0, stream.cuda_stream)

    def raw4():
        dk.library().dcp_topk_merge(*args4)

    out["merge_T16_dcp4_K4096_us_per_launch"] = median_of_reps(torch, raw4, stream)
    # rows whose K-th key is -inf: merges of short shards (80% of the slots
    # padding) and of the local top-Ks of causally masked rows
    short = {}
    for T in (16, 1024):
        m = workloads.random_merge(60 + T, T, 4, 2048, mode="bf16", pad_frac=0.8)
        s_ = torch.from_numpy(m.scores).to(dev)
        i_ = torch.from_numpy(m.ids).to(dev)
        oi_ = torch.empty((m.T, m.K), dtype=torch.int32, device=dev)
        os2 = torch.empty((m.T, m.K), dtype=torch.float32, device=dev)
        a_ = (s_.data_ptr(), i_.data_ptr(), m.T, m.dcp, m.K, None, oi_.data_ptr(), os2.data_ptr(),
              None, 0, stream.cuda_stream)
        short[f"padding80_T{T}_us_per_launch"] = median_of_reps(
            torch, lambda: dk.library().dcp_topk_merge(*a_), stream, launches=50)
    for T in (16, 1024):
        lg = torch.from_numpy(workloads.masked_logits(T)).to(dev)
        cs = torch.empty((4, T, 2048), dtype=torch.float32, device=dev)
        ci = torch.empty((4, T, 2048), dtype=torch.int32, device=dev)
        for r in range(4):
            dk.local_topk(lg[r], 2048, r, 4, out_scores=cs[r], out_ids=ci[r], stream=stream)
        oi_ = torch.empty((T, 2048), dtype=torch.int32, device=dev)
        os2 = torch.empty((T, 2048), dtype=torch.float32, device=dev)
        a_ = (cs.data_ptr(), ci.data_ptr(), T, 4, 2048, None, oi_.data_ptr(), os2.data_ptr(),
              None, 0, stream.cuda_stream)
        short[f"masked_merge_T{T}_us_per_launch"] = median_of_reps(
            torch, lambda: dk.library().dcp_topk_merge(*a_), stream, launches=50)
    out["neginf_threshold_merges"] = short
    sweep = {}
    K = 2048
    for T in workloads.SWEEP_T:
        logits = torch.from_numpy(workloads.sweep_logits(T)).to(dev)
        dcp = logits.shape[0]
        cs = torch.empty((dcp, T, K), dtype=torch.float32, device=dev)
        ci = torch.empty((dcp, T, K), dtype=torch.int32, device=dev)
        oi = torch.empty((T, K), dtype=torch.int32, device=dev)
        os_ = torch.empty((T, K), dtype=torch.float32, device=dev)

        def fn():
            for r in range(dcp):
                dk.local_topk(logits[r], K, r, dcp, out_scores=cs[r], out_ids=ci[r], stream=stream)
            dk.merge(cs, ci, out_ids=oi, out_scores=os_, stream=stream)

        fo_s = torch.empty((T, K), dtype=torch.float32, device=dev)
        fo_i = torch.empty((T, K), dtype=torch.int32, device=dev)

        def fused():
            dk.fused_topk(logits, K, out_scores=fo_s, out_ids=fo_i, stream=stream)

        def fused_inter():
            dk.fused_topk(logits, K, out_scores=fo_s, out_ids=fo_i, stream=stream,
                          layout="interleaved")

        sweep[str(T)] = {"us_per_step_launch": median_of_reps(torch, fn, stream, launches=50),
                         "us_per_step_graph": median_of_reps(torch, fn, stream, launches=50,
                                                             graph=True),
                         "fused_us_per_launch": median_of_reps(torch, fused, stream, launches=50),
                         "fused_us_per_graph_replay": median_of_reps(torch, fused, stream,
                                                                     launches=50, graph=True),
                         "fused_interleaved_us_per_graph_replay": median_of_reps(
                             torch, fused_inter, stream, launches=50, graph=True)}
    out["sweep_local4_plus_merge_and_fused"] = sweep
    return out


def end_to_end(torch, dk, m, dev, stream, steps, chunk=4096):
    """Same metric through the public API: every step copies the inputs from
    pinned host memory, merges, and reads the result back to pinned host
    memory, all inside the timed region.

    The rows are independent, so a step is pipelined over chunks of `chunk`
    rows on three streams (on the GB300 host, 4096-row chunks measured
    fastest: 2.79 ms per prefill step against 2.94 with 1024 and 3.4 with
    512 or 2048): chunk c's inputs are copied in (one copy per shard
    and array: each shard's rows are contiguous in the rank-major layout)
    while chunk c-1 is merged and chunk c-2's results are copied out.  Two
    chunk buffers alternate.  The host result is checked against one direct
    merge of the whole workload afterwards."""
    dcp, T, K = m.dcp, m.T, m.K
    tc = min(chunk, T)
    n_chunks = (T + tc - 1) // tc
    h_s = torch.from_numpy(m.scores).pin_memory()
    h_i = torch.from_numpy(m.ids).pin_memory()
    h_r = torch.from_numpy(m.row_starts).pin_memory()
    h_oi = torch.empty((T, K), dtype=torch.int32).pin_memory()
    h_os = torch.empty((T, K), dtype=torch.float32).pin_memory()
    b_s = [torch.empty((dcp, tc, K), dtype=torch.float32, device=dev) for _ in range(2)]
    b_i = [torch.empty((dcp, tc, K), dtype=torch.int32, device=dev) for _ in range(2)]
    b_r = [torch.empty((tc,), dtype=torch.int32, device=dev) for _ in range(2)]
    d_oi = torch.empty((T, K), dtype=torch.int32, device=dev)
    d_os = torch.empty((T, K), dtype=torch.float32, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    merged = [None, None]  # per buffer: the event after its last merge
    copied = [None] * n_chunks  # per chunk: the event after its rows' last copy out

    def step():
        for c in range(n_chunks):
            t0 = c * tc
            n = min(tc, T - t0)
            k = c % 2
            loaded = torch.cuda.Event()
            with torch.cuda.stream(s_in):
                if merged[k] is not None:
                    s_in.wait_event(merged[k])  # the buffer's previous chunk is merged
                for r in range(dcp):
                    b_s[k][r, :n].copy_(h_s[r, t0:t0 + n], non_blocking=True)
                    b_i[k][r, :n].copy_(h_i[r, t0:t0 + n], non_blocking=True)
                b_r[k][:n].copy_(h_r[t0:t0 + n], non_blocking=True)
                loaded.record(s_in)
            stream.wait_event(loaded)
            if copied[c] is not None:
                stream.wait_event(copied[c])  # the last step's rows are out
            src_s = b_s[k] if n == tc else b_s[k][:, :n].contiguous()
            src_i = b_i[k] if n == tc else b_i[k][:, :n].contiguous()
            dk.merge(src_s, src_i, b_r[k][:n], out_ids=d_oi[t0:t0 + n],
                     out_scores=d_os[t0:t0 + n], stream=stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            merged[k] = ev
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev)
                h_oi[t0:t0 + n].copy_(d_oi[t0:t0 + n], non_blocking=True)
                h_os[t0:t0 + n].copy_(d_os[t0:t0 + n], non_blocking=True)
                done = torch.cuda.Event()
                done.record(s_out)
                copied[c] = done

    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    stream.wait_event(a)
    s_out.wait_event(a)
    for _ in range(steps):
        step()
    # the last step's last copy out follows every copy in and merge
    b.record(s_out)
    b.synchronize()
    ms = a.elapsed_time(b)
    torch.cuda.synchronize(dev)
    want_i, want_s = dk.merge(torch.from_numpy(m.scores).to(dev), torch.from_numpy(m.ids).to(dev),
                              torch.from_numpy(m.row_starts).to(dev), stream=stream)
    stream.synchronize()
    if not (torch.equal(h_oi, want_i.cpu()) and
            torch.equal(h_os.view(torch.int32), want_s.cpu().view(torch.int32))):
        raise RuntimeError("pipelined end-to-end result differs from the direct merge")
    h2d = h_s.numel() * 4 + h_i.numel() * 4 + h_r.numel() * 4
    d2h = h_oi.numel() * 4 + h_os.numel() * 4
    return {"value": T * steps / (ms / 1000.0), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / steps,
            "pipeline": f"{n_chunks} chunks of {tc} rows: copies in, merge and copies out "
                        f"overlapped on three streams"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--skip-extras", action="store_true",
                    help="time only the headline step (used for profiling runs)")
    ap.add_argument("--workload", default="prefill",
                    choices=sorted(workloads.NAMED) + [f"sweep{T}" for T in workloads.SWEEP_T],
                    help="the workload of the headline step (default: prefill); sweepT times "
                         "the fused top-K over the T-row sweep logits instead of a merge")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
