"""Benchmark of the rank-sum reduce hot path on one GB300 (or N replicas).

Headline workload: W=8 rank buffers, M=512 rows, N=8192 columns, bf16
(8 MB per rank message).  One step runs what that workload asks for: the plain
one-shot rank sum (ar) and the fused rank sum + residual + RMSNorm
(residual_out, norm_out), both through the C ABI.  value = algorithmic HBM
bytes of the step / device time, in GB/s.  Inputs rotate over enough sets that
each step reads data that is not in L2.

The same JSON line carries the other workloads under "rows" (M=1 latency per
call from CUDA-graph replay, fp32 fused, LL128 W=16 decode-reduce with stale
lines, LL and LL128 encode), the roofline of the dominant kernel, clocks seen
during the timed region, an end-to-end number with host buffers, and the CPU
oracle's time on a bounded sample.

  python bench.py [--steps K] [--warmup W] [--impl car|reference]
  torchrun --nproc-per-node N bench.py --gpus N ...   (weak scaling: one replica per GPU)
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

# most steps in one timed CUDA graph, and launches per per-kernel graph (see headline)
MAX_GRAPH_STEPS = 1024
GRAPH_LAUNCHES = 128
# input sets the headline step and its per-kernel graphs rotate over (see headline)
HEADLINE_SETS = 8
# device time (ns) of the hold kernel queued ahead of a start event (see hold_device)
HOLD_NS = 30000
# steps of the end-to-end measurement run on this many streams in turn, so
# one step's host copies overlap the next step's
E2E_STREAMS = 3
HEADLINE = "m512_w8"
METRIC = "HBM GB/s (fraction of GB300 peak) for W-way reduce+RMSNorm; µs/call at M=1"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
DOMINANT = "reduce_residual_rmsnorm_tma_kernel"   # the automatic fused kernel at M=512 (M >= SM count)


# ---------------------------------------------------------------------------
# algorithmic bytes (reads of every input once + writes of every output once)
# ---------------------------------------------------------------------------
def bytes_reduce(wl):
    D = wl.data_bytes
    return wl.W * D + D


def bytes_fused(wl, outputs):
    D = wl.data_bytes
    s = workloads.ELEM_SIZE[wl.dtype]
    return wl.W * D + D + wl.N * s + outputs * D


def ll128_wire_bytes(D):
    return 128 * ((D + 119) // 120)


def ll_wire_bytes(D):
    return 16 * ((D + 7) // 8)


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_digest(texts):
    """Hash of C++ sources with comments and blank lines removed."""
    h = hashlib.sha256()
    for text in texts:
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = (re.sub(r"//.*", "", line).rstrip() for line in text.splitlines())
        h.update("\n".join(line for line in lines if line).encode())
    return h.hexdigest()[:16]


def kernel_source_hash():
    """Digest of the dominant kernel's code: fused_tma.cu (the pipelined fused
    kernel, its launch shape and launcher) and car_device.cuh (the device
    helpers it is built with).  The key under which
    profiles/dram_traffic.json holds the ncu counters taken on that code."""
    texts = []
    for f in ("fused_tma.cu", "car_device.cuh"):
        with open(os.path.join(ROOT, "rank_sum_reduce_gb300", "csrc", f)) as fh:
            texts.append(fh.read())
    return code_digest(texts)


def ncu_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when the kernel changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None, "no ncu capture committed"
    if d.get("source_sha256") != kernel_source_hash():
        return None, "kernel changed since the ncu capture"
    return float(d["dram_bytes_per_launch"]), d.get("note", "")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (read-only queries)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        inside = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed region"
        if len(inside) < 3:   # short timed region: widen to the loaded window around it
            inside = [s for t, s in self.samples if t0 - 1.0 <= t <= t1 + 0.5]
            window = "timed region +-1 s (region shorter than the sampling interval)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        mx = [num(s[2]) for s in inside if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4) if s[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max((num(s[3]) or 0.0) for s in inside)}


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------
class Arm:
    def __init__(self, dev):
        import torch

        import rank_sum_reduce_gb300 as car

        self.torch = torch
        self.car = car
        self.dev = dev
        self.lib = car.lib()
        self.launches = 0

    def stream(self):
        return self.torch.cuda.current_stream().cuda_stream

    @staticmethod
    def table(ptrs):
        return (ctypes.c_void_p * len(ptrs))(*ptrs)


def make_sets(torch, wl, dev, n_sets, outputs=("ar", "ro", "no")):
    """n_sets independent input/output sets of the workload on the device,
    drawn as one [n_sets * M, N] tensor per role (views stay 16-byte aligned)."""
    import dataclasses

    big = dataclasses.replace(wl, M=wl.M * n_sets)
    xs, res, _ = workloads.make_inputs(big, dev)
    w = workloads.make_weight(wl, dev)
    outs = {k: torch.empty_like(res) for k in outputs}
    sets = []
    for i in range(n_sets):
        rows = slice(i * wl.M, (i + 1) * wl.M)
        sets.append({"xs": [x[rows] for x in xs], "res": res[rows], "w": w, **{k: o[rows] for k, o in outs.items()}})
    return sets


def n_sets_for(set_bytes, minimum=3):
    return max(minimum, -(-2 * L2_BYTES // set_bytes) + 1)


def hold_device():
    """Queue a short device-side wait (torch's spin kernel) on the current
    stream before a start event: the event and the work after it are then
    submitted while the GPU is still busy, so the event marks the end of the
    wait and host submission latency stays out of the timed region (the
    blocking-kernel technique of GPU benchmark suites)."""
    import torch

    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:   # without it the region also holds the host's submission latency
        sleep(int(HOLD_NS * 2.1))   # clock cycles at about 2.1 GHz


def capture(torch, launches):
    """A CUDA graph of `launches` (callables taking a stream handle), captured
    on a side stream after one untimed run of the same launches."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        for fn in launches:
            fn(side.cuda_stream)
        side.synchronize()
        with torch.cuda.graph(g, stream=side):
            for fn in launches:
                fn(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return g


def headline(arm, wl, steps, warmup, rank, world):
    """Timed steps: plain reduce + fused reduce/residual/RMSNorm on rotating sets
    (the two calls of a step on different sets: see step_fns).

    The timed region replays one CUDA graph that holds exactly `steps` steps
    (for more than MAX_GRAPH_STEPS steps, a graph of a whole number of set
    rotations replayed several times, then one graph of the rest), between one
    start and one end event.  Warm-up runs its own graph of `warmup` steps,
    and the timed steps continue the set rotation where it stopped.  Each
    kernel's average launch duration comes from graphs of at least
    GRAPH_LAUNCHES launches of that kernel alone, timed the same way.  Graphs
    keep host launch overhead out of the device timeline."""
    torch, car, lib = arm.torch, arm.car, arm.lib
    set_bytes = (wl.W + 1) * wl.data_bytes + 3 * wl.data_bytes
    # At least HEADLINE_SETS sets: with 4 sets of 96 MiB a graph of plain
    # reduces alone found part of its inputs still in L2 (11.46 us per launch
    # against 12.39-12.55 us with 5, 6 or 8 sets), although the step itself
    # measured the same with 4, 5 and 8 sets (25.52, 25.52, 25.62 us).
    R = max(n_sets_for(set_bytes), HEADLINE_SETS)
    sets = make_sets(torch, wl, arm.dev, R)
    st, h = car.car_create(wl.W, wl.M, wl.N, car.DTYPE_CODE[wl.dtype])
    car.check(st, "car_create")
    eps = ctypes.c_float(wl.eps)

    def reduce_fn(S):
        tbl = Arm.table([x.data_ptr() for x in S["xs"]])
        ar = S["ar"].data_ptr()

        def run(stream):
            if lib.car_reduce(h, tbl, ar, stream):
                raise RuntimeError(car.car_last_error())
        return run

    def fused_fn(S):
        tbl = Arm.table([x.data_ptr() for x in S["xs"]])
        res, w, ro, no = S["res"].data_ptr(), S["w"].data_ptr(), S["ro"].data_ptr(), S["no"].data_ptr()

        def run(stream):
            if lib.car_reduce_residual_rmsnorm(h, tbl, res, w, eps, ro, no, None, stream):
                raise RuntimeError(car.car_last_error())
        return run

    # Step i runs the reduce on set i and the fused op on set i + R/2, so no
    # input line of the fused call is still in L2 from the reduce call just
    # before it (both read the W ranks; with the same set in both calls the
    # step runs about 0.6 us faster at m512_w8 from that reuse).  Over R steps
    # every set gets both calls.
    def step_fns(i):
        return [reduce_fn(sets[i % R]), fused_fn(sets[(i + R // 2) % R])]

    def steps_graph(first, count):
        return capture(torch, [fn for i in range(first, first + count) for fn in step_fns(i)])

    # A graph boundary leaves a gap on the device and breaks the PDL chain
    # (the next graph's first kernel cannot overlap the last one's tail), so
    # the timed steps sit in as few graphs as possible: one for up to
    # MAX_GRAPH_STEPS steps.
    chunk = steps if steps <= MAX_GRAPH_STEPS else (MAX_GRAPH_STEPS // R) * R
    n_chunks, rest = divmod(steps, chunk)
    warm = steps_graph(0, warmup)
    body = steps_graph(warmup, chunk)
    tail = steps_graph(warmup + n_chunks * chunk, rest) if rest else None
    rep_launch = max(1, -(-GRAPH_LAUNCHES // R))
    reduce_all = capture(torch, [reduce_fn(S) for _ in range(rep_launch) for S in sets])
    fused_all = capture(torch, [fused_fn(S) for _ in range(rep_launch) for S in sets])
    cs = torch.cuda.current_stream()

    warm.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    hold_device()
    e0.record(cs)
    for _ in range(n_chunks):
        body.replay()
    if tail is not None:
        tail.replay()
    e1.record(cs)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    region_ms = e0.elapsed_time(e1)

    def per_launch(graph):
        graph.replay()
        launches = R * rep_launch
        reps = max(1, steps // launches)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        hold_device()
        a.record(cs)
        for _ in range(reps):
            graph.replay()
        b.record(cs)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps * launches)

    reduce_ms = per_launch(reduce_all)
    fused_ms = per_launch(fused_all)
    status = car.car_sync(h, cs.cuda_stream)
    if status != car.CAR_OK:
        raise RuntimeError(f"car_sync: {car.car_status_string(status)}")
    del warm, body, tail, reduce_all, fused_all
    car.check(car.car_destroy(h), "car_destroy")
    return {"region_ms": region_ms, "reduce_ms": reduce_ms, "fused_ms": fused_ms, "sets": R, "set_bytes": set_bytes,
            "t0": t0, "t1": t1, "launches": 2 * steps, "graphs": n_chunks + (1 if rest else 0),
            "steps_per_graph": chunk}


def e2e(arm, wl, steps, warmup, streams=1):
    """Same step through the public API with pinned host buffers: H2D of the
    step's inputs, the two calls, D2H of its three outputs, all timed.  The
    inputs (W ranks, residual, weight) sit in one pinned host buffer and one
    device buffer, and the outputs in one of each, so a step makes one copy
    each way (the copy engines charge a gap per copy).  With streams > 1,
    step i runs on stream i % streams with that stream's own device and host
    buffers, so one step's copies overlap the neighbouring steps' copies and
    kernels; every step still copies all of its inputs in and outputs out."""
    torch, car = arm.torch, arm.car
    dev = arm.dev
    xs, res, w = workloads.make_inputs(wl, dev)
    parts = xs + [res, w]
    sizes = [t.numel() * t.element_size() for t in parts]   # each a multiple of 16 bytes
    offs = [sum(sizes[:i]) for i in range(len(sizes))]
    total = sum(sizes)
    hin = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o, n in zip(parts, offs, sizes):
        hin[o:o + n].copy_(t.reshape(-1).view(torch.uint8).cpu())
    D = wl.data_bytes

    def views(buf, like):
        return [buf[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(like, offs, sizes)]

    c = car.Car(wl.W, wl.M, wl.N, wl.dtype)
    lanes = []
    for _ in range(streams):
        din = torch.empty(total, dtype=torch.uint8, device=dev)
        dout = torch.empty(3 * D, dtype=torch.uint8, device=dev)
        v = views(din, parts)
        outs = [dout[k * D:(k + 1) * D].view(res.dtype).view(res.shape) for k in range(3)]
        lanes.append({"stream": torch.cuda.Stream() if streams > 1 else torch.cuda.current_stream(),
                      "din": din, "dout": dout, "dx": v[:wl.W], "dres": v[wl.W], "dw": v[wl.W + 1], "outs": outs,
                      "hout": torch.empty(3 * D, dtype=torch.uint8).pin_memory()})

    def step(i):
        L = lanes[i % streams]
        with torch.cuda.stream(L["stream"]):
            L["din"].copy_(hin, non_blocking=True)
            c.reduce(L["dx"], L["outs"][0])
            c.reduce_residual_rmsnorm(L["dx"], L["dres"], L["dw"], wl.eps, L["outs"][1], L["outs"][2])
            L["hout"].copy_(L["dout"], non_blocking=True)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for L in lanes:
        if L["stream"] is not main:
            L["stream"].wait_event(e0)
    for i in range(steps):
        step(i)
    for L in lanes:
        if L["stream"] is not main:
            main.wait_stream(L["stream"])
    e1.record(main)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    c.close()
    return ms, total, 3 * D


def latency_row(arm, wl, outputs, calls=12000):
    """µs per call of the fused op at M=1 from CUDA-graph replay of `calls`
    back-to-back calls, each on its own buffer set (the sets together exceed
    2x L2 when that fits in `calls`, so most reads come from HBM)."""
    torch, car = arm.torch, arm.car
    set_bytes = bytes_fused(wl, outputs)
    n = min(calls, max(64, 2 * L2_BYTES // set_bytes + 1))
    sets = make_sets(torch, wl, arm.dev, n, outputs=("ar", "ro", "no"))
    c = car.Car(wl.W, wl.M, wl.N, wl.dtype)
    lib, h = arm.lib, c.h
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    eps = ctypes.c_float(wl.eps)
    tables = [Arm.table([x.data_ptr() for x in S["xs"]]) for S in sets]
    with torch.cuda.stream(stream):
        for S, tbl in zip(sets, tables):   # warm the launch path once outside capture
            lib.car_reduce_residual_rmsnorm(h, tbl, S["res"].data_ptr(), S["w"].data_ptr(), eps, S["ro"].data_ptr(),
                                            S["no"].data_ptr(), S["ar"].data_ptr() if outputs == 3 else None,
                                            stream.cuda_stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for S, tbl in zip(sets, tables):
                st = lib.car_reduce_residual_rmsnorm(h, tbl, S["res"].data_ptr(), S["w"].data_ptr(), eps,
                                                     S["ro"].data_ptr(), S["no"].data_ptr(),
                                                     S["ar"].data_ptr() if outputs == 3 else None,
                                                     torch.cuda.current_stream().cuda_stream)
                if st:
                    raise RuntimeError(car.car_last_error())
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / (reps * n)
    del g
    # the same calls launched one by one on a stream through the C ABI (no
    # graph): device time per call, and host wall time spent in each call
    cs = torch.cuda.current_stream()
    plain = min(n, 2000)

    def issue():
        for S, tbl in zip(sets[:plain], tables[:plain]):
            st = lib.car_reduce_residual_rmsnorm(h, tbl, S["res"].data_ptr(), S["w"].data_ptr(), eps,
                                                 S["ro"].data_ptr(), S["no"].data_ptr(),
                                                 S["ar"].data_ptr() if outputs == 3 else None, cs.cuda_stream)
            if st:
                raise RuntimeError(car.car_last_error())
    issue()
    torch.cuda.synchronize()
    e0.record(cs)
    t0 = time.perf_counter()
    issue()
    t1 = time.perf_counter()
    e1.record(cs)
    torch.cuda.synchronize()
    stream_us = e0.elapsed_time(e1) * 1000.0 / plain
    host_us = (t1 - t0) * 1e6 / plain
    c.close()
    return {"us_per_call": round(us, 3), "calls_per_graph": n, "bytes_per_call": set_bytes,
            "GBps": round(set_bytes / (us * 1e-6) / 1e9, 1),
            "stream_launch_us_per_call": round(stream_us, 3), "host_us_per_call": round(host_us, 3),
            "l2": "cold (sets exceed 2x L2)" if n * set_bytes > 2 * L2_BYTES else "partly warm"}


def isolated_latency(arm, wl, outputs, calls=200, n_sets=4):
    """Device time of single, isolated fused calls: `calls` times, L2 is
    flushed (a read of twice its size), a hold kernel is queued, then the
    start event, one CUDA-graph replay holding one call (buffer sets
    rotating), and the end event.  Returns the median and the 95th percentile
    in us, the samples' minimum and maximum, the same two figures for the
    C-ABI call launched straight onto the stream instead of through a graph
    (`direct_*`; the hold kernel covers the host's time in the call), and the
    median of the same sequence with nothing between the two events (what
    the event pair itself costs on the device)."""
    torch, car = arm.torch, arm.car
    sets = make_sets(torch, wl, arm.dev, n_sets, outputs=("ar", "ro", "no"))
    c = car.Car(wl.W, wl.M, wl.N, wl.dtype)
    lib, h = arm.lib, c.h
    eps = ctypes.c_float(wl.eps)

    def call_fn(S):
        tbl = Arm.table([x.data_ptr() for x in S["xs"]])
        args = (S["res"].data_ptr(), S["w"].data_ptr(), eps, S["ro"].data_ptr(), S["no"].data_ptr(),
                S["ar"].data_ptr() if outputs == 3 else None)

        def run(stream):
            if lib.car_reduce_residual_rmsnorm(h, tbl, *args, stream):
                raise RuntimeError(car.car_last_error())
        return run

    fns = [call_fn(S) for S in sets]
    graphs = [capture(torch, [f]) for f in fns]
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=arm.dev)
    cs = torch.cuda.current_stream()

    def sample(kind):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(evs):
            flush.sum()
            hold_device()
            a.record(cs)
            if kind == "graph":
                graphs[i % n_sets].replay()
            elif kind == "direct":
                fns[i % n_sets](cs.cuda_stream)
            b.record(cs)
        torch.cuda.synchronize()
        return sorted(a.elapsed_time(b) * 1000.0 for a, b in evs)

    def p95(v):
        return v[min(len(v) - 1, int(0.95 * len(v)))]

    us = sample("graph")
    direct = sample("direct")
    empty = sample("none")   # the same sequence with nothing between the events
    c.sync()   # raises if a bounded wait ran out
    del graphs, flush
    c.close()
    med = statistics.median(us)
    return {"median_us": round(med, 3), "p95_us": round(p95(us), 3),
            "min_us": round(us[0], 3), "max_us": round(us[-1], 3), "calls": calls,
            "direct_median_us": round(statistics.median(direct), 3), "direct_p95_us": round(p95(direct), 3),
            "empty_event_pair_median_us": round(statistics.median(empty), 3),
            "net_median_us": round(med - statistics.median(empty), 3)}


def timed(torch, fn, iters):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fn(0)
    torch.cuda.synchronize()
    e0.record()
    for i in range(iters):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def two_shot_row(arm, iters=200):
    """Two-shot bit pattern (owner-rotated sum) at the headline shape, graph replay."""
    torch, car, lib = arm.torch, arm.car, arm.lib
    wl = workloads.WORKLOADS[HEADLINE]
    set_bytes = (wl.W + 1) * wl.data_bytes
    R = n_sets_for(set_bytes)
    sets = make_sets(torch, wl, arm.dev, R, outputs=("ar",))
    st, h = car.car_create(wl.W, wl.M, wl.N, car.DTYPE_CODE[wl.dtype])
    car.check(st, "car_create")

    def fn(S):
        tbl = Arm.table([x.data_ptr() for x in S["xs"]])
        ar = S["ar"].data_ptr()

        def run(stream):
            if lib.car_reduce_two_shot(h, tbl, ar, stream):
                raise RuntimeError(car.car_last_error())
        return run

    per = R * max(1, -(-GRAPH_LAUNCHES // R))   # launches per graph (see headline)
    g = capture(torch, [fn(sets[i % R]) for i in range(per)])
    reps = max(1, iters // per)
    ms = timed(torch, lambda i: g.replay(), reps) / per
    del g
    car.check(car.car_destroy(h), "car_destroy")
    return {"workload": "two_shot_" + wl.name, "ms": round(ms, 4), "bytes": set_bytes,
            "GBps": round(set_bytes / (ms * 1e-3) / 1e9, 1), "sets": R}


def lamport_row(arm, wl, rounds=30, reps=20):
    """Lamport one-shot push at M=1, from graph replay, small enough to stay in
    L2: µs per round (W pushes + the receive: fused residual + RMSNorm,
    sentinel checks, refill of the previous region) on one receive buffer, and
    µs per receive alone.  For the latter, round j reads its own buffer, filled
    beforehand by that round's pushes: a receive refills another region of
    it, so every replay reads complete data (a receive-only sequence on one
    buffer would read regions its predecessors had just refilled)."""
    torch, car = arm.torch, arm.car
    c = car.Car(wl.W, wl.M, wl.N, wl.dtype)
    xs, res, w = workloads.make_inputs(wl, arm.dev)
    ro, no = torch.empty_like(res), torch.empty_like(res)

    def round_fn(j, push, comm):
        def run(stream):
            if push:
                for r, x in enumerate(xs):
                    c.lamport_push(x, r, j, comm, stream=stream)
            c.lamport_reduce_residual_rmsnorm(comm, j, res, w, wl.eps, ro, no, stream=stream)
        return run

    comm = torch.empty(c.lamport_buffer_bytes, dtype=torch.uint8, device=arm.dev)
    c.lamport_init(comm)
    full = capture(torch, [round_fn(j, True, comm) for j in range(rounds)])
    full.replay()
    n_stale, _ = c.lamport_report()
    per_round = timed(torch, lambda i: full.replay(), reps) * 1000.0 / rounds
    del full
    bufs = [torch.empty(c.lamport_buffer_bytes, dtype=torch.uint8, device=arm.dev) for _ in range(rounds)]
    for j, b in enumerate(bufs):
        c.lamport_init(b)
        for r, x in enumerate(xs):
            c.lamport_push(x, r, j, b)
    recv = capture(torch, [round_fn(j, False, bufs[j]) for j in range(rounds)])
    recv.replay()
    n_stale_recv, _ = c.lamport_report()
    per_recv = timed(torch, lambda i: recv.replay(), reps) * 1000.0 / rounds
    del recv, bufs
    c.close()
    return {"workload": "lamport_" + wl.name, "us_per_receive": round(per_recv, 3),
            "us_per_round_with_pushes": round(per_round, 3), "kernels_per_round": wl.W + 1,
            "stale_after_full_round": n_stale, "stale_after_receives": n_stale_recv,
            "l2": "warm (buffers fit in L2)"}


def fused_fp32_row(arm, iters=50):
    torch, car = arm.torch, arm.car
    wl = workloads.WORKLOADS["m2048_w4_fp32"]
    set_bytes = bytes_fused(wl, 2)
    R = n_sets_for(set_bytes, 2)
    sets = make_sets(torch, wl, arm.dev, R, outputs=("ro", "no"))
    c = car.Car(wl.W, wl.M, wl.N, wl.dtype)
    ms = timed(torch, lambda i: c.reduce_residual_rmsnorm(sets[i % R]["xs"], sets[i % R]["res"], sets[i % R]["w"],
                                                          wl.eps, sets[i % R]["ro"], sets[i % R]["no"]), iters)
    c.close()
    return {"workload": wl.name, "ms": round(ms, 4), "bytes": set_bytes,
            "GBps": round(set_bytes / (ms * 1e-3) / 1e9, 1), "sets": R}


def ll128_row(arm, iters=10):
    """W=16, M=N=8192 bf16 rank buffers in LL128 wire format (flag 7,
    floor(L/4096) stale lines per rank): encode (per rank) and
    validate + decode + reduce."""
    torch, car = arm.torch, arm.car
    wl = workloads.WORKLOADS["ll128_w16"]
    D = wl.data_bytes
    L = (D + 119) // 120
    xs = [workloads.make_x(wl, r, arm.dev) for r in range(wl.W)]
    c = car.Car(wl.W, wl.M, wl.N, wl.dtype)
    wires = [torch.empty(c.ll128_wire_bytes, dtype=torch.uint8, device=arm.dev) for _ in range(wl.W)]
    g = capture(torch, [(lambda x, wv: (lambda s: c.ll128_encode(x, wl.ll128_flag, wv, stream=s)))(x, wv)
                        for x, wv in zip(xs, wires)])
    enc_ms = timed(torch, lambda i: g.replay(), 3) / wl.W
    del g
    stale = workloads.stale_lines(L, wl.W, wl.seed, wl.ll128_stale_every)
    old = torch.tensor(list(wl.ll128_stale_flag.to_bytes(8, "little")), dtype=torch.uint8, device=arm.dev)
    for wv, idx in zip(wires, stale):
        wv.view(L, 16, 8)[idx.to(arm.dev), 15] = old
    out = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device=arm.dev)
    dec_ms = timed(torch, lambda i: c.ll128_decode_reduce(wires, wl.ll128_flag, out), iters)
    n_stale, pairs = c.ll128_report()
    planted = {(r, int(k)) for r, idx in enumerate(stale) for k in idx.tolist()}
    ok = n_stale == len(planted) and set(pairs) == planted
    c.close()
    dec_bytes = wl.W * ll128_wire_bytes(D) + D
    enc_bytes = D + ll128_wire_bytes(D)
    del wires, xs
    return {"workload": wl.name, "decode_reduce_ms": round(dec_ms, 4), "decode_reduce_bytes": dec_bytes,
            "decode_reduce_GBps": round(dec_bytes / (dec_ms * 1e-3) / 1e9, 1),
            "encode_ms_per_rank": round(enc_ms, 4), "encode_GBps": round(enc_bytes / (enc_ms * 1e-3) / 1e9, 1),
            "stale_reported": n_stale, "stale_planted": len(planted), "stale_set_matches": bool(ok)}


# the (M, N) shapes of the fused op's latency table in "用 Triton + Symmetric
# Memory 写一个 AllReduce + RMSNorm 融合算子" (measured there on four GPUs
# over NVLink, so context only)
PAGE_SHAPES = [(1, 2048), (8, 2048), (128, 2048), (1, 4096), (128, 4096), (1, 8192), (128, 8192)]


def page_shapes_row(arm):
    """µs per call of the fused op (W=4 bf16, residual_out + norm_out) at the
    page table's shapes, from CUDA-graph replay over cold buffer sets."""
    out = {}
    for M, N in PAGE_SHAPES:
        wl = workloads.custom(4, M, N, "bf16", seed=100 + M + N)
        r = latency_row(arm, wl, 2, calls=4000)
        out[f"m{M}_n{N}"] = {"us_per_call": r["us_per_call"], "GBps": r["GBps"]}
    return {"W": 4, "dtype": "bf16", "outputs": 2, "shapes": out}


def ll128_misaligned_row(arm, M, launches, reps=5):
    """LL128 encode and decode-reduce at W=8, N=8192 bf16 (M rows per rank)
    with the rank data and the output 16-byte aligned, then both at 4, 8 and
    12 bytes past a 16-byte boundary (the offsets of "LL128 对齐实验设计"):
    what the misaligned path costs.  µs per call from graph replay of
    `launches` calls."""
    torch, car = arm.torch, arm.car
    W, N = 8, 8192
    wl = workloads.custom(W, M, N, "bf16", seed=77)
    D = wl.data_bytes
    c = car.Car(W, M, N, "bf16")
    xs = [workloads.make_x(wl, r, arm.dev) for r in range(W)]
    wires = [torch.empty(c.ll128_wire_bytes, dtype=torch.uint8, device=arm.dev) for _ in range(W)]
    keep = []

    def at_offset(src, off):
        b = torch.empty(D + 32, dtype=torch.uint8, device=arm.dev)
        keep.append(b)
        v = b[off:off + D]
        if src is not None:
            v.copy_(src.reshape(-1).view(torch.uint8))
        return v

    def per_call_us(fns):
        g = capture(torch, fns)
        us = timed(torch, lambda i: g.replay(), reps) * 1000.0 / len(fns)
        del g
        return us

    row = {"workload": f"ll128_w8_m{M}_n8192_bf16", "bytes_per_rank": D}
    outs = {}
    offsets = (("aligned", 0), ("offset4", 4), ("offset8", 8), ("offset12", 12))
    for name, off in offsets:
        data = [at_offset(x, off) for x in xs]
        out = at_offset(None, off)
        enc = [(lambda d, wv: (lambda s: c.ll128_encode(d, 7, wv, stream=s)))(data[i % W], wires[i % W])
               for i in range(launches)]
        dec = [lambda s: c.ll128_decode_reduce(wires, 7, out, stream=s)] * launches
        e_us = per_call_us(enc)
        d_us = per_call_us(dec)
        torch.cuda.synchronize()
        outs[name] = out.clone()
        row[name] = {"encode_us": round(e_us, 3), "encode_GBps": round((D + ll128_wire_bytes(D)) / e_us / 1e3, 1),
                     "decode_reduce_us": round(d_us, 3),
                     "decode_reduce_GBps": round((W * ll128_wire_bytes(D) + D) / d_us / 1e3, 1)}
    row["misaligned_over_aligned"] = {
        name: {k: round(row[name][k] / row["aligned"][k], 3) for k in ("encode_us", "decode_reduce_us")}
        for name, _ in offsets[1:]}
    row["outputs_equal"] = all(bool(torch.equal(outs["aligned"], outs[name])) for name, _ in offsets[1:])
    row["stale_reported"] = c.ll128_report()[0]
    row["l2"] = "warm (wires fit in L2)" if W * ll128_wire_bytes(D) < L2_BYTES else "cold (wires exceed L2)"
    c.close()
    del wires, xs, keep
    return row


def ll_row(arm, reps=5):
    """LL encode + validate/decode/reduce at the headline shape (W=8, 8 MB per
    rank), µs per call from graph replay.  Both rotate over sets of rank data
    and wires whose total exceeds 2x L2, so every call reads from HBM: the
    decode over 3 sets of 8 wires (128 MiB each), the encode over the 24
    (data, wire) pairs of those sets."""
    torch, car = arm.torch, arm.car
    wl = workloads.WORKLOADS[HEADLINE]
    D = wl.data_bytes
    c = car.Car(wl.W, wl.M, wl.N, wl.dtype)
    n_sets = max(3, -(-2 * L2_BYTES // (wl.W * c.ll_wire_bytes)) + 1)
    xs = [workloads.make_x(workloads.custom(wl.W, wl.M, wl.N, wl.dtype, seed=wl.seed + k), r, arm.dev)
          for k in range(n_sets) for r in range(wl.W)]
    wires = [torch.empty(c.ll_wire_bytes, dtype=torch.uint8, device=arm.dev) for _ in xs]
    outs = [torch.empty_like(xs[0]) for _ in range(n_sets)]
    pairs = len(xs)
    enc = capture(torch, [(lambda x, wv: (lambda s: c.ll_encode(x, 7, wv, stream=s)))(xs[i % pairs], wires[i % pairs])
                          for i in range(-(-64 // pairs) * pairs)])
    n_enc = -(-64 // pairs) * pairs
    enc_ms = timed(torch, lambda i: enc.replay(), reps) / n_enc
    del enc
    n_dec = -(-32 // n_sets) * n_sets
    dec = capture(torch, [(lambda k: (lambda s: c.ll_decode_reduce(wires[k * wl.W:(k + 1) * wl.W], 7, outs[k],
                                                                   stream=s)))(i % n_sets) for i in range(n_dec)])
    dec_ms = timed(torch, lambda i: dec.replay(), reps) / n_dec
    del dec
    n_stale, _ = c.ll_report()
    c.close()
    dec_bytes = wl.W * ll_wire_bytes(D) + D
    enc_bytes = D + ll_wire_bytes(D)
    return {"workload": "ll_" + wl.name, "decode_reduce_ms": round(dec_ms, 4),
            "decode_reduce_GBps": round(dec_bytes / (dec_ms * 1e-3) / 1e9, 1),
            "encode_ms_per_rank": round(enc_ms, 4), "encode_GBps": round(enc_bytes / (enc_ms * 1e-3) / 1e9, 1),
            "stale_reported": n_stale,
            "l2": f"cold: decode rotates over {n_sets} sets of {wl.W} wires ({n_sets * wl.W * ll_wire_bytes(D) >> 20} MiB), "
                  f"encode over {pairs} (data, wire) pairs"}


def noalloc_row(arm, reps=5):
    """The allocation-free LL128 decode-reduce against the handle's, µs per
    call from graph replay of 64 calls on the same wires: a small message
    (W=4, 74 KB per rank, in L2) and the headline shape (W=8, 8 MiB per rank,
    wires rotating over sets above 2x L2).  The allocation-free call adds a
    memset before and a copy after its kernel."""
    torch, car = arm.torch, arm.car
    out = {}
    for name, (W, M, N, n_sets) in {"small_w4_74KB": (4, 37, 1000, 1), "m512_w8": (8, 512, 8192, 3)}.items():
        wl = workloads.custom(W, M, N, "bf16", seed=31)
        c = car.Car(W, M, N, "bf16")
        x = workloads.make_x(wl, 0, arm.dev)
        wires = [torch.empty(c.ll128_wire_bytes, dtype=torch.uint8, device=arm.dev) for _ in range(W * n_sets)]
        for wv in wires:
            c.ll128_encode(x, 7, wv)
        o = torch.empty_like(x)
        cap = 64
        rep = torch.zeros(16 + 8 * cap, dtype=torch.uint8, device=arm.dev)

        def handle_fn(k):
            return lambda s: c.ll128_decode_reduce(wires[k * W:(k + 1) * W], 7, o, stream=s)

        def noalloc_fn(k):
            ptrs = [wv.data_ptr() for wv in wires[k * W:(k + 1) * W]]

            def run(s):
                st = car.car_ll128_decode_reduce_noalloc(W, M, N, car.CAR_BF16, ptrs, 7, 1, o.data_ptr(),
                                                         rep.data_ptr(), cap, s)
                if st:
                    raise RuntimeError(car.car_last_error())
            return run

        row = {}
        for kind, fn in (("handle_us", handle_fn), ("noalloc_us", noalloc_fn)):
            fn(0)(torch.cuda.current_stream().cuda_stream)   # first call on the device: set-up outside capture
            g = capture(torch, [fn(i % n_sets) for i in range(64)])
            row[kind] = round(timed(torch, lambda i: g.replay(), reps) * 1000.0 / 64, 3)
            del g
        row["extra_us"] = round(row["noalloc_us"] - row["handle_us"], 3)
        out[name] = row
        c.close()
    return out


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value, world):
    """The largest of every rank's value (timing only; not on the data path)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(region_ms_local, steps, step_bytes, world):
    """Weak scaling: every rank runs `steps` steps of its own replica.  The
    job's time is the slowest rank's; value counts the bytes of all ranks."""
    region_ms = max_over_ranks(region_ms_local, world)
    ms_per_step = region_ms / steps
    return ms_per_step, world * step_bytes / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# CPU oracle (baseline) -- only this leg and --impl reference run oracle/
# ---------------------------------------------------------------------------
def oracle_step_time(wl, budget_s, xs=None, res=None, w=None):
    """Time the oracle on the headline step (plain sum + fused op) over whole
    batches until `budget_s` has passed; returns (GB/s, steps, seconds)."""
    import torch

    import oracle

    if xs is None:
        xs, res, w = workloads.make_inputs(wl, "cpu")
    ar, ro, no = torch.empty_like(res), torch.empty_like(res), torch.empty_like(res)
    bytes_step = bytes_reduce(wl) + bytes_fused(wl, 2)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.reduce(xs, wl.dtype, ar)
        oracle.reduce_residual_rmsnorm(xs, res, w, wl.eps, wl.M, wl.N, wl.dtype, ro, no)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return bytes_step * n / el / 1e9, n, el


REFERENCE_ROWS = 64   # rows of the headline batch per reference step (a bounded sample)


def run_reference(args):
    """The oracle as it stands, on this host's cores: each step is a bounded
    sample (REFERENCE_ROWS rows of the headline workload) through the plain
    sum and the fused op; value = algorithmic bytes of the sample / time."""
    rank, _, world = dist_env()
    if world > 1 and rank != 0:
        return
    import dataclasses

    full = workloads.WORKLOADS[HEADLINE]
    wl = dataclasses.replace(full, M=REFERENCE_ROWS)
    xs, res, w = workloads.make_inputs(wl, "cpu")
    for _ in range(args.warmup):
        oracle_step_time(wl, 0.0, xs, res, w)
    total_s, steps = 0.0, 0
    for _ in range(args.steps):
        _, k, el = oracle_step_time(wl, 0.0, xs, res, w)
        total_s += el
        steps += k
    bytes_step = bytes_reduce(wl) + bytes_fused(wl, 2)
    gbps = bytes_step * steps / total_s / 1e9
    ms = total_s * 1000.0 / steps
    sample = (f"{REFERENCE_ROWS} of {full.M} rows of {full.name} per step (plain reduce + fused), "
              "single-threaded C oracle")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbps, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{full.name}: W={full.W} rank buffers, M={full.M}, N={full.N}, bf16; step = "
                                   "plain reduce (ar) + fused reduce+residual+RMSNorm (residual_out, norm_out)",
                       "storage": full.dtype, "accumulate": "f32", "sample_rows": REFERENCE_ROWS},
            "cpu_baseline": {"value": round(gbps, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(gbps, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
PROFILE_CASES = {
    # name: (W, M, N, dtype); each case's working set exceeds L2 and stays a few hundred MB
    "ll128_decode": (16, 1024, 8192, "bf16"),
    "ll_decode": (8, 512, 8192, "bf16"),
    "fused_fp32": (4, 2048, 4096, "fp32"),
    # the headline kernels on the headline workload, rotating over 4 input sets (384 MiB)
    "fused_m512_w8": (8, 512, 8192, "bf16"),
    "reduce_m512_w8": (8, 512, 8192, "bf16"),
    # the fused row kernel at one of the page's latency-table shapes, rotating over 24 sets (353 MB)
    "fused_rows_m128_w4": (4, 128, 8192, "bf16"),
    # LL128 encode of one rank of the W=16 workload (134 MB of data, 143 MB of wire per launch)
    "ll128_encode_w16": (16, 8192, 8192, "bf16"),
}


def profile_case(name, launches=4):
    """Run one workload's kernel `launches` times and exit: a small, fixed
    command for ncu captures (the headline kernels one at a time, each launch
    on the next of 4 input sets, and kernels outside the headline step)."""
    import torch

    import rank_sum_reduce_gb300 as car

    W, M, N, dt = PROFILE_CASES[name]
    dev = torch.device("cuda", 0)
    if name in ("fused_m512_w8", "reduce_m512_w8"):
        wl = workloads.WORKLOADS[HEADLINE]
        sets = make_sets(torch, wl, dev, 4)
        with car.Car(wl.W, wl.M, wl.N, wl.dtype) as c:
            for i in range(launches):
                S = sets[i % 4]
                if name == "fused_m512_w8":
                    c.reduce_residual_rmsnorm(S["xs"], S["res"], S["w"], wl.eps, S["ro"], S["no"])
                else:
                    c.reduce(S["xs"], S["ar"])
            torch.cuda.synchronize()
            c.sync()
        print(f"profile case {name}: {wl.name}, {launches} launches over 4 input sets")
        return
    if name == "fused_rows_m128_w4":
        wl = workloads.custom(W, M, N, dt, seed=90)
        sets = make_sets(torch, wl, dev, 24, outputs=("ro", "no"))
        with car.Car(W, M, N, dt) as c:
            for i in range(launches):
                S = sets[i % 24]
                c.reduce_residual_rmsnorm(S["xs"], S["res"], S["w"], wl.eps, S["ro"], S["no"])
            torch.cuda.synchronize()
            c.sync()
        print(f"profile case {name}: W={W} M={M} N={N} {dt}, {launches} launches over 24 input sets")
        return
    if name == "ll128_encode_w16":
        wl = workloads.WORKLOADS["ll128_w16"]
        xs = [workloads.make_x(wl, r, dev) for r in range(2)]
        with car.Car(wl.W, wl.M, wl.N, wl.dtype) as c:
            wires = [torch.empty(c.ll128_wire_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
            for i in range(launches):
                c.ll128_encode(xs[i % 2], wl.ll128_flag, wires[i % 2])
            torch.cuda.synchronize()
        print(f"profile case {name}: {wl.name} rank data, {launches} encodes over 2 ranks")
        return
    wl = workloads.custom(W, M, N, dt, seed=90)
    xs = [workloads.make_x(wl, r, dev) for r in range(W)]
    out = torch.empty_like(xs[0])
    with car.Car(W, M, N, dt) as c:
        if name == "fused_fp32":
            res, w = workloads.make_residual(wl, dev), workloads.make_weight(wl, dev)
            ro = torch.empty_like(res)
            for _ in range(launches):
                c.reduce_residual_rmsnorm(xs, res, w, wl.eps, ro, out)
        else:
            ll128 = name == "ll128_decode"
            wb = c.ll128_wire_bytes if ll128 else c.ll_wire_bytes
            wires = [torch.empty(wb, dtype=torch.uint8, device=dev) for _ in range(W)]
            for x, wv in zip(xs, wires):
                (c.ll128_encode if ll128 else c.ll_encode)(x, 7, wv)
            for _ in range(launches):
                (c.ll128_decode_reduce if ll128 else c.ll_decode_reduce)(wires, 7, out)
        torch.cuda.synchronize()
        c.sync()
    print(f"profile case {name}: W={W} M={M} N={N} {dt}, {launches} launches")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1, help="GPUs (one process each under torchrun; replicas)")
    ap.add_argument("--steps", type=int, default=20000, help="timed steps (one plain reduce and one fused call each)")
    ap.add_argument("--warmup", type=int, default=50, help="untimed steps before the timed region")
    ap.add_argument("--impl", choices=["car", "reference"], default="car",
                    help="car: the CUDA path; reference: the CPU oracle on the host cores")
    ap.add_argument("--no-rows", action="store_true", help="skip the other workloads")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES),
                    help="run one workload's kernel a few times and exit (for ncu captures)")
    ap.add_argument("--profile-launches", type=int, default=4, help="launches of the --profile-case kernel")
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args.profile_case, args.profile_launches)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return

    rank, local_rank, world = dist_env()
    import torch

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    import __graft_entry__

    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    arm = Arm(dev)
    wl = workloads.WORKLOADS[HEADLINE]

    rows = {}
    m1 = {}
    if not args.no_rows and rank == 0:
        for key, name, outputs in (("m1_w2_fused_3out", "m1_w2", 3), ("m1_w8_fused", "m1_w8", 2)):
            wl_m1 = workloads.WORKLOADS[name]
            rows[key] = latency_row(arm, wl_m1, outputs)
            rows[key]["isolated"] = isolated_latency(arm, wl_m1, outputs)
            iso = rows[key]["isolated"]
            m1[name] = {"median_us": iso["median_us"], "p95_us": iso["p95_us"],
                        "direct_median_us": iso["direct_median_us"], "direct_p95_us": iso["direct_p95_us"],
                        "empty_events_us": iso["empty_event_pair_median_us"], "b2b_us_per_call": rows[key]["us_per_call"]}
        rows["lamport_m1_w2"] = lamport_row(arm, workloads.WORKLOADS["m1_w2"])
        rows["lamport_m1_w8"] = lamport_row(arm, workloads.WORKLOADS["m1_w8"])
        rows["m2048_w4_fp32_fused"] = fused_fp32_row(arm)
        rows["two_shot_m512_w8"] = two_shot_row(arm)
        rows["ll128_w16_decode_reduce"] = ll128_row(arm)
        rows["ll_m512_w8"] = ll_row(arm)
        rows["fused_w4_page_shapes"] = page_shapes_row(arm)
        rows["ll128_misaligned_1MiB"] = ll128_misaligned_row(arm, 64, 256)
        rows["ll128_misaligned_64MiB"] = ll128_misaligned_row(arm, 4096, 16)
        rows["ll128_noalloc_vs_handle"] = noalloc_row(arm)
        torch.cuda.empty_cache()

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    H = headline(arm, wl, args.steps, args.warmup, rank, world)
    if sampler:
        time.sleep(0.3)
        sampler.stop()
    step_bytes = bytes_reduce(wl) + bytes_fused(wl, 2)
    ms_per_step, value = aggregate(H["region_ms"], args.steps, step_bytes, world)

    e2e_steps = max(3, min(args.steps, 50))
    e2e_ms, h2d, d2h = e2e(arm, wl, e2e_steps, 3, streams=E2E_STREAMS)
    e2e_ms = max_over_ranks(e2e_ms, world)
    e2e_gbps = world * step_bytes / (e2e_ms * 1e-3) / 1e9
    e2e_serial_ms, _, _ = e2e(arm, wl, e2e_steps, 3, streams=1)
    e2e_serial_ms = max_over_ranks(e2e_serial_ms, world)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak()
    fused_bytes = bytes_fused(wl, 2)
    achieved = fused_bytes / (H["fused_ms"] * 1e-3) / 1e9
    traffic, traffic_note = ncu_traffic()
    reduce_achieved = bytes_reduce(wl) / (H["reduce_ms"] * 1e-3) / 1e9

    cpu = None
    if world == 1 and args.cpu_budget > 0:
        wl_cpu = wl
        gbps, n, el = oracle_step_time(wl_cpu, args.cpu_budget)
        cpu = {"value": round(gbps, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} full batch(es) of {wl.name} (plain reduce + fused) in {el:.1f} s, single thread",
               "online_cores": os.cpu_count()}

    clocks = sampler.summary(H["t0"], H["t1"]) if sampler else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{wl.name}: W={wl.W} rank buffers, M={wl.M}, N={wl.N}, bf16; step = plain "
                               "reduce (ar) + fused reduce+residual+RMSNorm (residual_out, norm_out)",
                   "timing": f"the K steps replayed from {H['graphs']} CUDA graph(s) of {H['steps_per_graph']} steps "
                             "cycling over the input sets, after a graph of the W warm-up steps; one start and one "
                             "end event around them, a hold kernel queued before the start event",
                   "storage": wl.dtype, "accumulate": "f32", "eps": wl.eps,
                   "l2": f"inputs rotate over {H['sets']} sets of {H['set_bytes'] >> 20} MiB (> 2x L2); "
                         f"a step's fused call reads the set {H['sets'] // 2} steps ahead of its reduce call's",
                   "bytes_per_step": step_bytes, "parallelism": f"{world} independent replica(s), no collective"},
        "gpu_launches": H["launches"],
        "kernels": {"rank_sum_reduce_kernel": {"ms_per_launch": round(H["reduce_ms"], 5),
                                               "bytes": bytes_reduce(wl), "GBps": round(reduce_achieved, 1),
                                               "frac": round(reduce_achieved / peak, 4)},
                    DOMINANT: {"ms_per_launch": round(H["fused_ms"], 5), "bytes": fused_bytes,
                               "GBps": round(achieved, 1), "frac": round(achieved / peak, 4)},
                    "method": "graphs of >= 128 launches cycling over the input sets, replayed; CUDA events around the replays"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": DOMINANT,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "traffic_note": traffic_note},
        "e2e": {"value": round(e2e_gbps, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps, "streams": E2E_STREAMS,
                "serial_value": round(world * step_bytes / (e2e_serial_ms * 1e-3) / 1e9, 2),
                "serial_ms_per_step": round(e2e_serial_ms, 4)},
        "clocks": clocks,
        "cpu_baseline": cpu,
        "rows": rows,
        # last, so that a truncated copy of the line keeps it: M=1 latency of
        # the fused call per isolated call (median, P95) and back to back
        "m1_latency": m1 or None,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
